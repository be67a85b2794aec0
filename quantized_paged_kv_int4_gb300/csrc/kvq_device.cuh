// Device helpers shared by the libkvq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cuda.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kPage = 16;  // tokens per page: one MMA M-tile of the read kernels

// Device-side error flags (kvq_device_error).
enum : unsigned { ERR_BLOCK = 1u, ERR_SEQLEN = 2u, ERR_SLOT = 4u, ERR_TIMEOUT = 8u, ERR_RANGE = 16u };

// 2^k for an integer k in [-126, 127], exact.
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }
// floor(log2 x) of a finite x > 0 from its exponent field (-127 for zero and subnormals, 128
// for inf / NaN).
__device__ __forceinline__ int ilog2f(float x) { return ((__float_as_uint(x) >> 23) & 0xFF) - 127; }

// ---------------------------------------------------------------------------------------------
// Exact fp32 building blocks (IEEE round-to-nearest, never contracted into an FMA).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// round half away from zero, then float -> int32 truncating and saturating (NaN -> 0)
__device__ __forceinline__ int round_half_away(float x) {
  return x >= 0.f ? __float2int_rz(__fadd_rn(x, 0.5f)) : __float2int_rz(__fsub_rn(x, 0.5f));
}

// One butterfly stage across lanes: element i pairs with i ^ (lane_mask * elems_per_lane).
// The lower element keeps a + b, the upper one gets a - b (a = lower, b = upper).
__device__ __forceinline__ float butterfly_xor(float self, int lane, int mask) {
  const float other = __shfl_xor_sync(FULL, self, mask);
  return (lane & mask) ? __fsub_rn(other, self) : __fadd_rn(self, other);
}

// In-register butterfly stages h = 1, 2, ..., N/2 over N consecutive elements.
template <int N>
__device__ __forceinline__ void butterfly_local(float (&x)[N]) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1) {
#pragma unroll
    for (int j = 0; j < N; ++j) {
      if (!(j & h)) {
        const float a = x[j], b = x[j + h];
        x[j] = __fadd_rn(a, b);
        x[j + h] = __fsub_rn(a, b);
      }
    }
  }
}

// ---------------------------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------------------------
// Packed fp32 pairs (the Blackwell f32x2 ALU): add.rn / sub.rn .f32x2 round each component
// exactly like the scalar instruction, so a pair of butterflies costs one instruction with the
// same bits. (A packed multiply that feeds a packed add may be fused into a multiply-add by the
// assembler: where two roundings are required, keep that step scalar.)
__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
  return static_cast<unsigned long long>(__float_as_uint(a)) | (static_cast<unsigned long long>(__float_as_uint(b)) << 32);
}
__device__ __forceinline__ void f2unpack(unsigned long long v, float &a, float &b) {
  a = __uint_as_float(static_cast<uint32_t>(v));
  b = __uint_as_float(static_cast<uint32_t>(v >> 32));
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// butterfly stages h = 1 .. N/2 over N consecutive elements (the pages' order): h = 1 scalar, h >= 2
// on packed pairs (j, j + 1)
template <int N>
__device__ __forceinline__ void butterfly_local2(float (&x)[N]) {
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    const float a = x[j], b = x[j + 1];
    x[j] = __fadd_rn(a, b);
    x[j + 1] = __fsub_rn(a, b);
  }
#pragma unroll
  for (int h = 2; h < N; h <<= 1) {
#pragma unroll
    for (int j = 0; j < N; j += 2) {
      if (!(j & h)) {
        const unsigned long long a = f2pack(x[j], x[j + 1]), b = f2pack(x[j + h], x[j + h + 1]);
        f2unpack(add2(a, b), x[j], x[j + 1]);
        f2unpack(sub2(a, b), x[j + h], x[j + h + 1]);
      }
    }
  }
}
// the same stages over rows of two columns at once: element r of column c is x[c][r]
__device__ __forceinline__ void butterfly_cols2(float (&x)[2][8]) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (!(r & h)) {
        const unsigned long long a = f2pack(x[0][r], x[1][r]), b = f2pack(x[0][r + h], x[1][r + h]);
        f2unpack(add2(a, b), x[0][r], x[1][r]);
        f2unpack(sub2(a, b), x[0][r + h], x[1][r + h]);
      }
    }
  }
}


__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// dst = (a & mask) | magic  in one LOP3
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(magic));
  return d;
}

__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Asynchronous global -> shared copies (LDGSTS). src_bytes == 0 zero-fills without reading.
template <int BYTES>
__device__ __forceinline__ void cp_async(uint32_t dst, const void *src, bool valid) {
  const int n = valid ? BYTES : 0;
  if constexpr (BYTES == 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
                 : "memory");
  } else {
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(dst), "l"(src), "n"(BYTES),
                 "r"(n)
                 : "memory");
  }
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared-memory reads as plain loads: ordered after cp_async_wait by its memory clobber, free to
// be scheduled otherwise.
__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ uint2 lds64(const uint8_t *p) { return *reinterpret_cast<const uint2 *>(p); }
__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

// 2^x with the SFU instruction (relative error ~2^-22; results below 2^-126 flush to zero,
// which for softmax weights exp2(s - max) <= 1 only drops terms under 1e-38)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------------------------
// mbarrier + TMA (cp.async.bulk.tensor) helpers
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Non-blocking probe: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Arrive once on the barrier (release semantics: this thread's earlier accesses come first).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// try_wait that may suspend the thread (up to hint_ns) until the phase completes, instead of
// returning at once: a waiting warp then takes no issue slots from the others.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase with the given parity to complete, giving up after limit_ns of wall time
// (~2 s by default: a copy that never lands is a bug; the caller reports ERR_TIMEOUT instead of
// hanging).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 200000u)) return true;
    if (global_ns() - start > limit_ns) return false;
  }
}
// Shared-memory counter increment with acquire-release semantics at CTA scope; returns the old
// value. Used to find the last of a CTA's warps to finish reading a buffer.
__device__ __forceinline__ unsigned atom_add_acq_rel_cta(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(v)
               : "memory");
  return old;
}
// Order this thread's earlier generic-proxy shared-memory accesses before later async-proxy
// (TMA) writes to the same buffers.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// Byte offset of (row, byte) inside a tile written by TMA with the 64B (rows of 64 bytes) or
// 32B (rows of 32 bytes) swizzle: the 16-byte chunk index is XORed with address bits 7.. of the
// row start. The tile base must be 1024-byte aligned.
template <int ROW_BYTES>
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t byte) {
  constexpr uint32_t mask = ROW_BYTES / 16 - 1;  // 3 (64B swizzle) or 1 (32B swizzle)
  const uint32_t o = row * ROW_BYTES;
  return o + ((((byte >> 4) ^ (o >> 7)) & mask) << 4) + (byte & 15);
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

__device__ __forceinline__ float warp_max_g(float v) {  // over the 8 lanes sharing lane & 3
  v = fmaxf(v, __shfl_xor_sync(FULL, v, 4));
  v = fmaxf(v, __shfl_xor_sync(FULL, v, 8));
  v = fmaxf(v, __shfl_xor_sync(FULL, v, 16));
  return v;
}
__device__ __forceinline__ float warp_sum_g(float v) {
  v += __shfl_xor_sync(FULL, v, 4);
  v += __shfl_xor_sync(FULL, v, 8);
  v += __shfl_xor_sync(FULL, v, 16);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, m));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(FULL, v, m);
  return v;
}

}  // namespace kvq
