// kvq_write_int4: random-sign Hadamard rotation + asymmetric INT4 quantization + page scatter.
//
// Follows int4_per_token_head.py, reshape_and_cache_int4 (single_rht of K and V, cast back to
// bf16) and _reshape_cache_int4_kernel (per (token, head) min/max, scale, zero-point hidden in the
// scale word's low mantissa bits, nibble packing, slot_mapping scatter). The rotation is fused:
// the rotated vector never goes to memory.
//
// Mapping: 8 lanes per vector, E = D/8 consecutive elements per lane; a warp handles K and V of two
// (token, kv head) pairs. The butterfly keeps the pages' stage order h = 1, 2, ..., D/2: stages
// h < E run in registers; for h = E, 2E, 4E the warp transposes its vectors through shared memory
// (a lane then holds the 8 rows of its columns), runs them in registers, and transposes back.
// Quantization avoids float<->int conversions: for u = x * inv + zp (two roundings, as the pages),
// clamp(rha(u), 0, 15) == trunc(clamp(u + 0.5, 0, 15.5)) (u + 0.5 rounded as the pages' rha does;
// for u < 0 both give 0), and trunc of a value in [0, 15.5] is the low bits of (value + 2^23)
// added with round-toward-zero.

#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {

__device__ unsigned g_flags_write = 0;

struct WriteParams {
  const __nv_bfloat16 *key, *value;
  int64_t k_stride_t, k_stride_h, v_stride_t, v_stride_h;
  uint8_t *k_cache, *v_cache;
  uint32_t *k_scale, *v_scale;
  const int64_t *slot_mapping;
  const float *signs;
  int32_t T, Hk, block_size;
  int64_t num_blocks;
};

// clamp(round_half_away(x), 0, 15) for the x = fp32 value the pages round (see above)
__device__ __forceinline__ uint32_t nibble_of(float x) {
  const float w = fminf(fmaxf(__fadd_rn(x, 0.5f), 0.f), 15.5f);
  return __float_as_uint(__fadd_rz(w, 8388608.0f)) & 0xFu;
}

template <int D>
struct WriteGeom {
  static constexpr int E = D / 8;          // elements per lane (one row of the 8 x E vector view)
  static constexpr int CPL = E / 8;        // columns per lane in the transposed view
  static constexpr int ROW = E + 4;        // padded row (words): conflict-free row and column access
  static constexpr int VEC = 8 * ROW + 16; // padded vector: the 4 vectors of a warp in two bank halves
};

template <int D>
__global__ void __launch_bounds__(256) write_int4_kernel(const WriteParams p) {
  using Wg = WriteGeom<D>;
  constexpr int E = Wg::E, CPL = Wg::CPL;
  __shared__ __align__(16) float s_buf[8][4 * Wg::VEC];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v = lane >> 3, l8 = lane & 7;  // vector of the warp (K/V of pair 0, K/V of pair 1), row
  const bool is_v = v & 1;
  const long long pair = static_cast<long long>(blockIdx.x) * 16 + warp * 2 + (v >> 1);
  const bool in_range = pair < static_cast<long long>(p.T) * p.Hk;
  bool valid = in_range;
  const int t = valid ? static_cast<int>(pair / p.Hk) : 0;
  const int h = valid ? static_cast<int>(pair % p.Hk) : 0;
  const long long slot = valid ? __ldg(p.slot_mapping + t) : -1;
  if (valid && slot >= p.num_blocks * p.block_size) {
    if (l8 == 0 && !is_v) atomicOr(&g_flags_write, ERR_SLOT);
    valid = false;
  }
  valid = valid && slot >= 0;  // padding tokens store nothing

  float x[E];
  {
    const __nv_bfloat16 *src = (is_v ? p.value + t * p.v_stride_t + h * p.v_stride_h
                                     : p.key + t * p.k_stride_t + h * p.k_stride_h) + l8 * E;
#pragma unroll
    for (int i = 0; i < E / 8; ++i) {
      // loaded whatever the slot says (a skipped token's row is read but not stored), so the
      // load does not wait for slot_mapping
      const uint4 raw = in_range ? __ldg(reinterpret_cast<const uint4 *>(src) + i) : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
        x[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
      }
    }
  }

  float *buf = &s_buf[warp][v * Wg::VEC];
  if (p.signs != nullptr) {
    // H (x * d1): exact sign flip, then stages h = 1 .. E/2 inside the lane's row
    const float4 *sg = reinterpret_cast<const float4 *>(p.signs + l8 * E);
#pragma unroll
    for (int i = 0; i < E / 4; ++i) {
      const float4 s = __ldg(sg + i);
      x[4 * i] *= s.x;
      x[4 * i + 1] *= s.y;
      x[4 * i + 2] *= s.z;
      x[4 * i + 3] *= s.w;
    }
    butterfly_local<E>(x);
    // stages h = E, 2E, 4E pair rows r and r ^ 1, 2, 4: transpose, butterfly over rows, back
#pragma unroll
    for (int i = 0; i < E / 4; ++i)
      *reinterpret_cast<float4 *>(buf + l8 * Wg::ROW + 4 * i) = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
    __syncwarp();
    float c[CPL][8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if constexpr (CPL == 2) {
        const float2 f = *reinterpret_cast<const float2 *>(buf + r * Wg::ROW + 2 * l8);
        c[0][r] = f.x;
        c[1][r] = f.y;
      } else {
        c[0][r] = buf[r * Wg::ROW + l8];
      }
    }
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc) butterfly_local<8>(c[cc]);
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if constexpr (CPL == 2)
        *reinterpret_cast<float2 *>(buf + r * Wg::ROW + 2 * l8) = make_float2(c[0][r], c[1][r]);
      else
        buf[r * Wg::ROW + l8] = c[0][r];
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < E / 4; ++i) {
      const float4 f = *reinterpret_cast<const float4 *>(buf + l8 * Wg::ROW + 4 * i);
      x[4 * i] = bf16_round(f.x);
      x[4 * i + 1] = bf16_round(f.y);
      x[4 * i + 2] = bf16_round(f.z);
      x[4 * i + 3] = bf16_round(f.w);
    }
  }

  float mn = x[0], mx = x[0];
#pragma unroll
  for (int j = 1; j < E; ++j) {
    mn = fminf(mn, x[j]);
    mx = fmaxf(mx, x[j]);
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(FULL, mn, m));
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, m));
  }
  const float scale = fmaxf(__fdiv_rn(__fsub_rn(mx, mn), 15.0f), 1e-6f);
  const uint32_t zpi = nibble_of(__fdiv_rn(-mn, scale));
  const float zp = static_cast<float>(zpi);
  const float inv = __fdiv_rn(1.0f, scale);

  uint32_t packed[E / 8];
#pragma unroll
  for (int i = 0; i < E / 8; ++i) {
    uint32_t wd = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) wd |= nibble_of(__fadd_rn(__fmul_rn(x[8 * i + k], inv), zp)) << (4 * k);
    packed[i] = wd;
  }
  if (!valid) return;
  const long long row = ((slot / p.block_size) * p.block_size + slot % p.block_size) * p.Hk + h;
  uint8_t *dst = (is_v ? p.v_cache : p.k_cache) + row * (D / 2) + l8 * (E / 2);
  if constexpr (E == 16)
    *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
  else
    *reinterpret_cast<uint32_t *>(dst) = packed[0];
  if (l8 == 0) (is_v ? p.v_scale : p.k_scale)[row] = (__float_as_uint(scale) & 0xFFFFFFF0u) | zpi;
}

bool take_flags_write(cudaStream_t stream, unsigned *host_word) {
  static const unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(host_word, g_flags_write, sizeof(unsigned), 0,
                                cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return false;
  return cudaMemcpyToSymbolAsync(g_flags_write, &zero, sizeof(unsigned), 0,
                                 cudaMemcpyHostToDevice, stream) == cudaSuccess;
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_write_int4(const void *key, const void *value, int64_t k_stride_t,
                                     int64_t k_stride_h, int64_t v_stride_t, int64_t v_stride_h,
                                     uint8_t *k_cache, uint8_t *v_cache, float *k_scale,
                                     float *v_scale, const int64_t *slot_mapping,
                                     const float *rht_signs, int32_t T, int32_t Hk, int32_t D,
                                     int32_t block_size, int64_t num_blocks,
                                     kvq_stream_t stream) {
  if (T < 0 || Hk < 1 || block_size < 1 || num_blocks < 1) return KVQ_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (T == 0) return KVQ_OK;
  if (!key || !value || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping)
    return KVQ_ERR_INVALID_ARG;
  const int vec = 8;  // elements per 16-byte vector load
  if (!aligned(key, vec * 2) || !aligned(value, vec * 2) || k_stride_t % vec || k_stride_h % vec ||
      v_stride_t % vec || v_stride_h % vec || k_stride_t < 0 || k_stride_h < 0 ||
      v_stride_t < 0 || v_stride_h < 0)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_scale, 4) ||
      !aligned(v_scale, 4) || !aligned(slot_mapping, 8) || (rht_signs && !aligned(rht_signs, 16)))
    return KVQ_ERR_INVALID_ARG;

  WriteParams p;
  p.key = static_cast<const __nv_bfloat16 *>(key);
  p.value = static_cast<const __nv_bfloat16 *>(value);
  p.k_stride_t = k_stride_t;
  p.k_stride_h = k_stride_h;
  p.v_stride_t = v_stride_t;
  p.v_stride_h = v_stride_h;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = reinterpret_cast<uint32_t *>(k_scale);
  p.v_scale = reinterpret_cast<uint32_t *>(v_scale);
  p.slot_mapping = slot_mapping;
  p.signs = rht_signs;
  p.T = T;
  p.Hk = Hk;
  p.block_size = block_size;
  p.num_blocks = num_blocks;

  const long long pairs = static_cast<long long>(T) * Hk;
  const unsigned grid = static_cast<unsigned>((pairs + 15) / 16);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 128)
    write_int4_kernel<128><<<grid, 256, 0, s>>>(p);
  else
    write_int4_kernel<64><<<grid, 256, 0, s>>>(p);
  return launch_status();
}
