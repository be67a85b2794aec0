// kvq_fwht128: fused normalised Walsh-Hadamard-128 rotation + per-row power-of-two FP8 quant.
//
// Follows kpool_compress.py, _fwht_quant_kernel / fwht128_quant_fp8: fp32 butterflies (stride
// 1, 2, ..., 64), one multiply by fp32(1/sqrt(128)), a cast to bf16, absmax with a 1e-4 floor,
// scale = 2^ceil(log2(absmax / 448)) (taken as the exact smallest power of two >= the fp32
// product absmax * fp32(1/448)), y = clamp(x / scale, +-448) stored as E4M3FN (round to nearest
// even). The rotated row never leaves registers.
//
// Mapping: a half-warp per 128-wide row, 8 elements (16 bytes) per lane; one warp = 2 rows.

#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {

__global__ void __launch_bounds__(256) fwht128_fp8_kernel(const __nv_bfloat16 *__restrict__ x,
                                                          uint8_t *__restrict__ y,
                                                          float *__restrict__ row_scale,
                                                          long long rows) {
  const int lane = threadIdx.x & 31;
  const int l16 = lane & 15;
  const long long row = (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * 2 + (lane >> 4);
  const bool live = row < rows;
  float v[8];
  {
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (live) raw = __ldg(reinterpret_cast<const uint4 *>(x + row * 128) + l16);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  butterfly_local<8>(v);  // h = 1, 2, 4
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {  // h = 8, 16, 32, 64
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = butterfly_xor(v[j], l16, m);
  }
  const float kInvSqrt128 = 0x1.6a09e6p-4f;  // 0.08838834764831845 rounded to fp32
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[j] = bf16_round(__fmul_rn(v[j], kInvSqrt128));
    amax = fmaxf(amax, fabsf(v[j]));
  }
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, m));
  amax = fmaxf(amax, 1e-4f);
  const float kInv448 = 0x1.24924ap-9f;  // 1/448 rounded to fp32
  const uint32_t mb = __float_as_uint(__fmul_rn(amax, kInv448));
  // smallest power of two >= m: m itself when its mantissa is zero, else the next binade
  const float s = (mb & 0x007FFFFFu) ? __uint_as_float((mb & 0x7F800000u) + 0x00800000u)
                                     : __uint_as_float(mb);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float a = fminf(fmaxf(__fdiv_rn(v[j], s), -448.f), 448.f);
    const float b = fminf(fmaxf(__fdiv_rn(v[j + 1], s), -448.f), 448.f);
    const uint32_t pair = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    if (j < 4)
      lo |= pair << (8 * j);
    else
      hi |= pair << (8 * (j - 4));
  }
  if (live) {
    reinterpret_cast<uint2 *>(y + row * 128)[l16] = make_uint2(lo, hi);
    if (l16 == 0) row_scale[row] = s;
  }
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_fwht128(const void *x, uint8_t *y_e4m3, float *row_scale, int64_t rows,
                                  kvq_stream_t stream) {
  if (rows < 0) return KVQ_ERR_INVALID_ARG;
  if (rows == 0) return KVQ_OK;
  if (!x || !y_e4m3 || !row_scale || !aligned(x, 16) || !aligned(y_e4m3, 8) || !aligned(row_scale, 4))
    return KVQ_ERR_INVALID_ARG;
  const long long blocks = (rows + 15) / 16;
  if (blocks > 0x7fffffffLL) return KVQ_ERR_UNSUPPORTED;
  fwht128_fp8_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16 *>(x), y_e4m3, row_scale, rows);
  return launch_status();
}
