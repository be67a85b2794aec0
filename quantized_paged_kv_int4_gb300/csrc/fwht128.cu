// kvq_fwht128: fused normalised Walsh-Hadamard-128 rotation + per-row power-of-two FP8 quant.
//
// Follows kpool_compress.py, _fwht_quant_kernel / fwht128_quant_fp8: fp32 butterflies (stride
// 1, 2, ..., 64), one multiply by fp32(1/sqrt(128)), a cast to bf16, absmax with a 1e-4 floor,
// scale = 2^ceil(log2(absmax / 448)) (taken as the exact smallest power of two >= the fp32
// product absmax * fp32(1/448)), y = clamp(x / scale, +-448) stored as E4M3FN (round to nearest
// even). The rotated row never leaves registers.
//
// Mapping: 8 lanes per 128-wide row, 16 elements per lane; one warp = 4 rows.

#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {

// Row r of a warp (4 rows per warp) is viewed as 8 x 16: lane l8 of the row holds elements
// 16 l8 .. 16 l8 + 15. Stages h = 1 .. 8 run in the lane; for h = 16, 32, 64 the warp transposes
// its rows through shared memory (lane l8 then holds columns 2 l8, 2 l8 + 1 of all 8 row-blocks),
// runs them in registers and transposes back -- the pages' stage order throughout.
constexpr int kFwRow = 16 + 4;          // padded 16-element block (words)
constexpr int kFwVec = 8 * kFwRow + 16; // padded row: the 4 rows of a warp in two bank halves

// A tile is 32 rows (8 warps x 4 rows); CTAs stride over tiles and fetch the next tile's rows
// before working on the current one.
__global__ void __launch_bounds__(256, 4) fwht128_fp8_kernel(const __nv_bfloat16 *__restrict__ x,
                                                             uint8_t *__restrict__ y,
                                                             float *__restrict__ row_scale,
                                                             long long rows, long long tiles) {
  __shared__ __align__(16) float s_buf[8][4 * kFwVec];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rw = lane >> 3, l8 = lane & 7;
  float *buf = &s_buf[warp][rw * kFwVec];
  auto fetch = [&](long long t, uint4 (&raw)[2]) {
    const long long row = (t * 8 + warp) * 4 + rw;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + row * 128 + 16 * l8);
    raw[0] = row < rows ? __ldg(src) : make_uint4(0, 0, 0, 0);
    raw[1] = row < rows ? __ldg(src + 1) : make_uint4(0, 0, 0, 0);
  };
  uint4 cur[2];
  long long tile = blockIdx.x;
  if (tile < tiles) fetch(tile, cur);
  for (; tile < tiles; tile += gridDim.x) {
    uint4 nxt[2];
    const long long nt = tile + gridDim.x;
    if (nt < tiles) fetch(nt, nxt);
    const long long row = (tile * 8 + warp) * 4 + rw;

    float v[16];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t w[4] = {cur[i].x, cur[i].y, cur[i].z, cur[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
        v[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
      }
    }
    butterfly_local<16>(v);  // h = 1, 2, 4, 8
    __syncwarp();            // the previous tile's reads of buf are done
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4 *>(buf + l8 * kFwRow + 4 * i) = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    __syncwarp();
    float c0[8], c1[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float2 f = *reinterpret_cast<const float2 *>(buf + r * kFwRow + 2 * l8);
      c0[r] = f.x;
      c1[r] = f.y;
    }
    butterfly_local<8>(c0);  // h = 16, 32, 64
    butterfly_local<8>(c1);
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 8; ++r) *reinterpret_cast<float2 *>(buf + r * kFwRow + 2 * l8) = make_float2(c0[r], c1[r]);
    __syncwarp();
    const float kInvSqrt128 = 0x1.6a09e6p-4f;  // 0.08838834764831845 rounded to fp32
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 f = *reinterpret_cast<const float4 *>(buf + l8 * kFwRow + 4 * i);
      v[4 * i] = bf16_round(__fmul_rn(f.x, kInvSqrt128));
      v[4 * i + 1] = bf16_round(__fmul_rn(f.y, kInvSqrt128));
      v[4 * i + 2] = bf16_round(__fmul_rn(f.z, kInvSqrt128));
      v[4 * i + 3] = bf16_round(__fmul_rn(f.w, kInvSqrt128));
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, m));
    amax = fmaxf(amax, 1e-4f);
    const float kInv448 = 0x1.24924ap-9f;  // 1/448 rounded to fp32
    const uint32_t mb = __float_as_uint(__fmul_rn(amax, kInv448));
    // smallest power of two >= m: m itself when its mantissa is zero, else the next binade
    const uint32_t sb = (mb & 0x007FFFFFu) ? (mb & 0x7F800000u) + 0x00800000u : mb;
    const float s = __uint_as_float(sb);
    // x / s == x * (1/s) exactly while s is a power of two below 2^127 (1/s is then one too); an
    // infinite input row (s = inf) keeps the division
    const bool by_inv = sb < 0x7F000000u;
    const float inv = __uint_as_float(0x7F000000u - (by_inv ? sb : 0x3F800000u));
    // the clamp to [-448, 448] is the conversion's own saturation (finite and infinite values)
    if (by_inv) {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], inv);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = __fdiv_rn(v[j], s);
    }
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t p0 = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * k], v[4 * k + 1]), __NV_SATFINITE, __NV_E4M3);
      const uint32_t p1 = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * k + 2], v[4 * k + 3]), __NV_SATFINITE, __NV_E4M3);
      out[k] = p0 | (p1 << 16);
    }
    if (row < rows) {
      reinterpret_cast<uint4 *>(y + row * 128)[l8] = make_uint4(out[0], out[1], out[2], out[3]);
      if (l8 == 0) row_scale[row] = s;
    }
    if (nt < tiles) {
      cur[0] = nxt[0];
      cur[1] = nxt[1];
    }
  }
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_fwht128(const void *x, uint8_t *y_e4m3, float *row_scale, int64_t rows,
                                  kvq_stream_t stream) {
  if (rows < 0) return KVQ_ERR_INVALID_ARG;
  if (rows == 0) return KVQ_OK;
  if (!x || !y_e4m3 || !row_scale || !aligned(x, 16) || !aligned(y_e4m3, 16) || !aligned(row_scale, 4))
    return KVQ_ERR_INVALID_ARG;
  const long long tiles = (rows + 31) / 32;
  static int per_sm = 0;  // resident CTAs per SM, from the occupancy calculator
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwht128_fp8_kernel, 256, 0) != cudaSuccess || n < 1) n = 1;
    per_sm = n;
  }
  const long long cap = static_cast<long long>(sm_count() > 0 ? sm_count() : 1) * per_sm;
  fwht128_fp8_kernel<<<static_cast<unsigned>(tiles < cap ? tiles : cap), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16 *>(x), y_e4m3, row_scale, rows, tiles);
  return launch_status();
}
