// kvq_write_int4: random-sign Hadamard rotation + asymmetric INT4 quantization + page scatter.
//
// Follows int4_per_token_head.py, reshape_and_cache_int4 (single_rht of K and V, cast back to
// bf16) and _reshape_cache_int4_kernel (per (token, head) min/max, scale, zero-point hidden in the
// scale word's low mantissa bits, nibble packing, slot_mapping scatter). The rotation is fused:
// the rotated vector never goes to memory.
//
// Mapping: one warp per (token, kv head); lanes 0-15 handle K, lanes 16-31 handle V, each lane
// D/16 consecutive elements (one 16-byte load at D = 128). The butterfly runs in registers and
// over xor-shuffles inside each half-warp.

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

template <int D>
__global__ void __launch_bounds__(256) write_int4_kernel(const WriteParams p) {
  constexpr int EPL = D / 16;  // elements per lane
  const int lane = threadIdx.x & 31;
  const int l16 = lane & 15;
  const bool is_v = lane >= 16;
  const long long pair = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (pair >= static_cast<long long>(p.T) * p.Hk) return;  // warp-uniform
  const int t = static_cast<int>(pair / p.Hk);
  const int h = static_cast<int>(pair % p.Hk);
  const long long slot = __ldg(p.slot_mapping + t);
  if (slot < 0) return;  // padding token: nothing stored (warp-uniform)
  if (slot >= p.num_blocks * p.block_size) {
    if (lane == 0) atomicOr(&g_flags_write, ERR_SLOT);
    return;
  }

  const __nv_bfloat16 *src = is_v ? p.value + t * p.v_stride_t + h * p.v_stride_h
                                  : p.key + t * p.k_stride_t + h * p.k_stride_h;
  src += l16 * EPL;
  float x[EPL];
  if constexpr (EPL == 8) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(src));
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(src));
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }

  if (p.signs != nullptr) {
    // H (x * d1): sign flip (exact), butterfly stages h = 1 .. D/2 in increasing order.
    const float4 *sg = reinterpret_cast<const float4 *>(p.signs + l16 * EPL);
#pragma unroll
    for (int i = 0; i < EPL / 4; ++i) {
      const float4 s = __ldg(sg + i);
      x[4 * i] *= s.x;
      x[4 * i + 1] *= s.y;
      x[4 * i + 2] *= s.z;
      x[4 * i + 3] *= s.w;
    }
    butterfly_local<EPL>(x);
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) {
#pragma unroll
      for (int j = 0; j < EPL; ++j) x[j] = butterfly_xor(x[j], l16, m);
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j) x[j] = bf16_round(x[j]);
  }

  float mn = x[0], mx = x[0];
#pragma unroll
  for (int j = 1; j < EPL; ++j) {
    mn = fminf(mn, x[j]);
    mx = fmaxf(mx, x[j]);
  }
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(FULL, mn, m));
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, m));
  }
  const float scale = fmaxf(__fdiv_rn(__fsub_rn(mx, mn), 15.0f), 1e-6f);
  const float zp = fminf(fmaxf(static_cast<float>(round_half_away(__fdiv_rn(-mn, scale))), 0.f), 15.f);
  const float inv = __fdiv_rn(1.0f, scale);

  uint32_t packed = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const float u = __fadd_rn(__fmul_rn(x[j], inv), zp);
    const float qf = fminf(fmaxf(static_cast<float>(round_half_away(u)), 0.f), 15.f);
    packed |= static_cast<uint32_t>(qf) << (4 * j);
  }

  const long long row = ((slot / p.block_size) * p.block_size + slot % p.block_size) * p.Hk + h;
  uint8_t *cache = is_v ? p.v_cache : p.k_cache;
  uint8_t *dst = cache + row * (D / 2) + l16 * (EPL / 2);
  if constexpr (EPL == 8) {
    *reinterpret_cast<uint32_t *>(dst) = packed;
  } else {
    *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(packed);
  }
  if (l16 == 0) {
    const uint32_t word =
        (__float_as_uint(scale) & 0xFFFFFFF0u) | (static_cast<uint32_t>(static_cast<int>(zp)) & 0xFu);
    (is_v ? p.v_scale : p.k_scale)[row] = word;
  }
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
  const int vec = D / 16;  // elements per vector load
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
  const unsigned grid = static_cast<unsigned>((pairs + 7) / 8);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 128)
    write_int4_kernel<128><<<grid, 256, 0, s>>>(p);
  else
    write_int4_kernel<64><<<grid, 256, 0, s>>>(p);
  return launch_status();
}
