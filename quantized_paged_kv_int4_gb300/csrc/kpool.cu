// kvq_kpool_write: kpool compress-and-write -- per pool, the per-dimension softmax (over the pool's
// slots) of slot_score + ape weights the slot keys; the pooled key goes through bf16, the
// normalised Hadamard-128, bf16 again and the per-vector absmax FP8 quantizer, and is written with
// its fp32 scale into the paged indexer cache at loc.
//
// Follows kpool_compress.py, _kpool_softmax_rotate_write_cache_kernel and
// kpool_compress_and_write_cache (WRITE_CACHE, optional write mask, ROUND_SCALE on or off). The
// fp32 operations are the pages' in their order, each rounded to nearest: z = score + ape, the
// max over slots, w = exp(z - max), den += w, acc += k * w (a multiply, then an add), x = acc /
// den. The exponential is written out (exp_pool below: Cody and Waite's range reduction with a
// two-part ln 2, then the Taylor series of e^r to degree 7; within 1 ulp of exp, results below
// the normal range flushed to zero) so the pooled value -- and every FP8 code that depends on it
// -- is reproducible bit for bit.
//
// Mapping (as fwht128.cu): 8 lanes per pool row, 16 dimensions per lane, 4 pools per warp,
// 32 pools per CTA tile; the Hadamard stages h >= 16 go through a per-warp shared-memory
// transpose; CTAs stride over tiles.

#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {

__device__ unsigned g_flags_kpool = 0;

struct KpoolParams {
  uint8_t *cache;                  // [num_blocks, page_size, 128 + 4]
  const __nv_bfloat16 *slot_k;     // [n, pool, 128]
  const float *slot_score;         // [n, pool, 128]
  const float *ape;                // [pool, 128]
  const int64_t *loc;              // [n]
  const uint8_t *write_mask;       // [n] bool or null
  long long n_pools;
  int pool, page_size;
  long long num_blocks;
  bool round_scale;
};

__device__ __forceinline__ float exp_pool(float x) {
  const float kLog2e = 0x1.715476p+0f, kLn2Hi = 0x1.62ep-1f, kLn2Lo = 0x1.0bfbe8p-15f;
  x = fmaxf(x, -104.f);
  const float n = rintf(__fmul_rn(x, kLog2e));
  const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(n, kLn2Hi)), __fmul_rn(n, kLn2Lo));
  float p = 0x1.a01a02p-13f;                                   // 1/7!
  p = __fadd_rn(__fmul_rn(p, r), 0x1.6c16c2p-10f);             // 1/6!
  p = __fadd_rn(__fmul_rn(p, r), 0x1.111112p-7f);              // 1/5!
  p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-5f);              // 1/4!
  p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-3f);              // 1/3!
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  // p * 2^n for n in [-125, 127] (p in [0.7, 1.42], so the product is a normal number and exact):
  // the power of two built from its exponent bits, the same value ldexp gives
  return n <= -126.f ? 0.f : __fmul_rn(p, __int_as_float((static_cast<int>(fminf(n, 127.f)) + 127) << 23));
}

constexpr int kKpRow = 16 + 4;           // padded 16-element block (words)
constexpr int kKpVec = 8 * kKpRow + 16;  // padded row: the 4 rows of a warp in two bank halves

// KP > 0: the pool size as a compile-time constant (the slot loops unroll, so every slot's loads
// are in flight together); KP == 0: any pool size from the parameters. Two CTAs per SM (at most
// 128 registers): at one CTA per SM the unrolled form was slower than the rolled one.
template <int KP>
__global__ void __launch_bounds__(256, 2) kpool_write_kernel(const KpoolParams p, long long tiles) {
  const int pool = KP > 0 ? KP : p.pool;
  __shared__ __align__(16) float s_buf[8][4 * kKpVec];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rw = lane >> 3, l8 = lane & 7;
  float *buf = &s_buf[warp][rw * kKpVec];
  for (long long tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const long long row = (tile * 8 + warp) * 4 + rw;
    const bool live = row < p.n_pools;
    const bool write = live && (p.write_mask == nullptr || p.write_mask[row] != 0);

    // ---- pooled key of dims 16 l8 .. 16 l8 + 15
    float v[16];
    {
      const long long kbase = (live ? row : 0) * pool * 128 + 16 * l8;
      float M[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) M[j] = -INFINITY;
#pragma unroll
      for (int s = 0; s < pool; ++s) {
        const float4 *sc = reinterpret_cast<const float4 *>(p.slot_score + kbase + s * 128);
        const float4 *ap = reinterpret_cast<const float4 *>(p.ape + s * 128 + 16 * l8);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 a = __ldg(sc + i), b = __ldg(ap + i);
          M[4 * i] = fmaxf(M[4 * i], __fadd_rn(a.x, b.x));
          M[4 * i + 1] = fmaxf(M[4 * i + 1], __fadd_rn(a.y, b.y));
          M[4 * i + 2] = fmaxf(M[4 * i + 2], __fadd_rn(a.z, b.z));
          M[4 * i + 3] = fmaxf(M[4 * i + 3], __fadd_rn(a.w, b.w));
        }
      }
      float den[16], acc[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) den[j] = acc[j] = 0.f;
#pragma unroll
      for (int s = 0; s < pool; ++s) {
        const float4 *sc = reinterpret_cast<const float4 *>(p.slot_score + kbase + s * 128);
        const float4 *ap = reinterpret_cast<const float4 *>(p.ape + s * 128 + 16 * l8);
        const uint4 *kr = reinterpret_cast<const uint4 *>(p.slot_k + kbase + s * 128);
        const uint4 kw[2] = {__ldg(kr), __ldg(kr + 1)};
        float z[16], k[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 a = __ldg(sc + i), b = __ldg(ap + i);
          z[4 * i] = __fadd_rn(a.x, b.x);
          z[4 * i + 1] = __fadd_rn(a.y, b.y);
          z[4 * i + 2] = __fadd_rn(a.z, b.z);
          z[4 * i + 3] = __fadd_rn(a.w, b.w);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t w[4] = {kw[i].x, kw[i].y, kw[i].z, kw[i].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            k[8 * i + 2 * q] = __uint_as_float(w[q] << 16);
            k[8 * i + 2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float wgt = exp_pool(__fsub_rn(z[j], M[j]));
          den[j] = __fadd_rn(den[j], wgt);
          acc[j] = __fadd_rn(acc[j], __fmul_rn(k[j], wgt));
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = write ? bf16_round(__fdiv_rn(acc[j], den[j])) : 0.f;
    }

    // ---- normalised Hadamard-128 (stages h = 1 .. 64), bf16, absmax FP8 quantizer
    butterfly_local<16>(v);  // h = 1, 2, 4, 8
    __syncwarp();            // the previous tile's reads of buf are done
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4 *>(buf + l8 * kKpRow + 4 * i) = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    __syncwarp();
    float c0[8], c1[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float2 f = *reinterpret_cast<const float2 *>(buf + r * kKpRow + 2 * l8);
      c0[r] = f.x;
      c1[r] = f.y;
    }
    butterfly_local<8>(c0);  // h = 16, 32, 64
    butterfly_local<8>(c1);
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 8; ++r) *reinterpret_cast<float2 *>(buf + r * kKpRow + 2 * l8) = make_float2(c0[r], c1[r]);
    __syncwarp();
    const float kInvSqrt128 = 0x1.6a09e6p-4f;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 f = *reinterpret_cast<const float4 *>(buf + l8 * kKpRow + 4 * i);
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
    const float m448 = __fmul_rn(amax, 0x1.24924ap-9f);  // * fp32(1/448)
    float s;
    if (p.round_scale) {  // smallest power of two >= m448; divide by multiplying with its exact inverse
      const uint32_t mb = __float_as_uint(m448);
      const uint32_t sb = (mb & 0x007FFFFFu) ? (mb & 0x7F800000u) + 0x00800000u : mb;
      s = __uint_as_float(sb);
      const float inv = __uint_as_float(0x7F000000u - sb);  // sb < 2^127: amax is finite here
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], inv);
    } else {
      s = m448;
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = __fdiv_rn(v[j], s);
    }
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // the +-448 clamp is the conversion's saturation
      const uint32_t p0 = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * k], v[4 * k + 1]), __NV_SATFINITE, __NV_E4M3);
      const uint32_t p1 = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * k + 2], v[4 * k + 3]), __NV_SATFINITE, __NV_E4M3);
      out[k] = p0 | (p1 << 16);
    }
    if (write) {
      const long long loc = p.loc[row];
      if (loc < 0 || loc >= p.num_blocks * p.page_size) {
        if (l8 == 0) atomicOr(&g_flags_kpool, ERR_SLOT);
      } else {
        const long long page = loc / p.page_size, off = loc - page * p.page_size;
        uint8_t *pg = p.cache + page * p.page_size * 132;
        reinterpret_cast<uint4 *>(pg + off * 128)[l8] = make_uint4(out[0], out[1], out[2], out[3]);
        if (l8 == 0) reinterpret_cast<float *>(pg + p.page_size * 128)[off] = s;
      }
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Tail ring: prefill seeding and the batched decode-step update (kpool_compress.py,
// _kpool_tail_seed_kernel and _kpool_decode_update_batched_kernel). The tail cache is bf16
// [blocks][2][ring][128] addressed through its block and half strides (it may alias a padded
// cache); half 0 holds keys, half 1 gate scores.
// ---------------------------------------------------------------------------------------------

struct TailArgs {
  __nv_bfloat16 *tail;
  long long block_stride, half_stride;  // elements
  int ring;
  long long blocks;
};

// One warp per token; lane l copies key / score elements 4l .. 4l + 3 (8 bytes each).
__global__ void __launch_bounds__(256) kpool_seed_tail_kernel(const TailArgs ta, const __nv_bfloat16 *__restrict__ key,
                                                              const __nv_bfloat16 *__restrict__ score,
                                                              const int32_t *__restrict__ tslot, long long n,
                                                              int kpool) {
  const long long i = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n) return;
  const long long t = tslot[i];
  if (t < 0) return;
  const long long blk = t / ta.ring;
  const long long ahead = i + kpool < n ? tslot[i + kpool] : -1;
  if (ahead >= 0 && ahead / ta.ring == blk) return;  // not among the request's last kpool tokens
  if (blk >= ta.blocks) {
    if (lane == 0) atomicOr(&g_flags_kpool, ERR_SLOT);
    return;
  }
  __nv_bfloat16 *dst = ta.tail + blk * ta.block_stride + (t % ta.ring) * 128 + 4 * lane;
  *reinterpret_cast<uint2 *>(dst) = __ldg(reinterpret_cast<const uint2 *>(key + i * 128) + lane);
  *reinterpret_cast<uint2 *>(dst + ta.half_stride) = __ldg(reinterpret_cast<const uint2 *>(score + i * 128) + lane);
}

struct DecodeUpdateArgs {
  uint8_t *cache;
  int page_size;
  long long num_blocks;
  const int32_t *tail_slot, *slot_mapping, *positions;  // [R, next_n]
  const __nv_bfloat16 *key, *score;
  long long key_sb, key_st, score_sb, score_st;         // strides (elements)
  const float *ape;                                     // [pool, 128]
  int R, next_n, pool;
  bool round_scale;
};

__device__ __forceinline__ void load_bf16x4(const __nv_bfloat16 *p, float (&v)[4]) {
  const uint2 w = *reinterpret_cast<const uint2 *>(p);
  v[0] = __uint_as_float(w.x << 16);
  v[1] = __uint_as_float(w.x & 0xffff0000u);
  v[2] = __uint_as_float(w.y << 16);
  v[3] = __uint_as_float(w.y & 0xffff0000u);
}

// One warp per request, its next_n tokens in order; lane l owns dimensions 4l .. 4l + 3. A pool
// completion reads ring entries that earlier tokens of this warp stashed -- each lane its own
// dimensions, so program order makes them visible.
__global__ void __launch_bounds__(256) kpool_decode_update_kernel(const DecodeUpdateArgs a, const TailArgs ta) {
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= a.R) return;
  for (int t = 0; t < a.next_n; ++t) {
    const long long idx = static_cast<long long>(r) * a.next_n + t;
    const long long loc = a.slot_mapping[idx];
    const int pos = a.positions[idx];
    const long long ts = a.tail_slot[idx];
    const int safe_pos = max(pos, 0);
    const int slot = safe_pos % a.pool;
    const long long blk = max(ts, 0LL) / ta.ring;
    const bool blk_ok = blk < ta.blocks;
    float key[4], sc[4];
    load_bf16x4(a.key + r * a.key_sb + t * a.key_st + 4 * lane, key);
    load_bf16x4(a.score + r * a.score_sb + t * a.score_st + 4 * lane, sc);
    const __nv_bfloat16 *ring_k = ta.tail + (blk_ok ? blk : 0) * ta.block_stride + 4 * lane;
    const __nv_bfloat16 *ring_s = ring_k + ta.half_stride;

    if (loc >= 0 && pos >= 0 && slot == a.pool - 1) {
      if (!blk_ok || loc >= a.num_blocks * a.page_size) {
        if (lane == 0) atomicOr(&g_flags_kpool, ERR_SLOT);
      } else {
        const int start = safe_pos - slot;
        float M[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        for (int j = 0; j < a.pool; ++j) {
          float z[4];
          if (j == slot) {
#pragma unroll
            for (int e = 0; e < 4; ++e) z[e] = sc[e];
          } else {
            load_bf16x4(ring_s + ((start + j) % ta.ring) * 128, z);
          }
          const float4 ap = __ldg(reinterpret_cast<const float4 *>(a.ape + j * 128 + 4 * lane));
          M[0] = fmaxf(M[0], __fadd_rn(z[0], ap.x));
          M[1] = fmaxf(M[1], __fadd_rn(z[1], ap.y));
          M[2] = fmaxf(M[2], __fadd_rn(z[2], ap.z));
          M[3] = fmaxf(M[3], __fadd_rn(z[3], ap.w));
        }
        float den[4] = {0.f, 0.f, 0.f, 0.f}, acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < a.pool; ++j) {
          float z[4], k[4];
          if (j == slot) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              z[e] = sc[e];
              k[e] = key[e];
            }
          } else {
            const int phys = (start + j) % ta.ring;
            load_bf16x4(ring_s + phys * 128, z);
            load_bf16x4(ring_k + phys * 128, k);
          }
          const float4 ap = __ldg(reinterpret_cast<const float4 *>(a.ape + j * 128 + 4 * lane));
          const float zz[4] = {__fadd_rn(z[0], ap.x), __fadd_rn(z[1], ap.y), __fadd_rn(z[2], ap.z), __fadd_rn(z[3], ap.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float w = exp_pool(__fsub_rn(zz[e], M[e]));
            den[e] = __fadd_rn(den[e], w);
            acc[e] = __fadd_rn(acc[e], __fmul_rn(k[e], w));
          }
        }
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = bf16_round(__fdiv_rn(acc[e], den[e]));
        // Hadamard-128: stages h = 1, 2 in the lane, h = 4 .. 64 across lanes (partner lane ^ h/4)
        butterfly_local<4>(v);
#pragma unroll
        for (int mask = 1; mask < 32; mask <<= 1) {
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = butterfly_xor(v[e], lane, mask);
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[e] = bf16_round(__fmul_rn(v[e], 0x1.6a09e6p-4f));
          amax = fmaxf(amax, fabsf(v[e]));
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, m));
        amax = fmaxf(amax, 1e-4f);
        const float m448 = __fmul_rn(amax, 0x1.24924ap-9f);
        float s;
        if (a.round_scale) {
          const uint32_t mb = __float_as_uint(m448);
          const uint32_t sb = (mb & 0x007FFFFFu) ? (mb & 0x7F800000u) + 0x00800000u : mb;
          s = __uint_as_float(sb);
          const float inv = __uint_as_float(0x7F000000u - sb);
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = __fmul_rn(v[e], inv);
        } else {
          s = m448;
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = __fdiv_rn(v[e], s);
        }
        const uint32_t c01 = __nv_cvt_float2_to_fp8x2(make_float2(v[0], v[1]), __NV_SATFINITE, __NV_E4M3);
        const uint32_t c23 = __nv_cvt_float2_to_fp8x2(make_float2(v[2], v[3]), __NV_SATFINITE, __NV_E4M3);
        const long long page = loc / a.page_size, off = loc - page * a.page_size;
        uint8_t *pg = a.cache + page * a.page_size * 132;
        reinterpret_cast<uint32_t *>(pg + off * 128)[lane] = c01 | (c23 << 16);
        if (lane == 0) reinterpret_cast<float *>(pg + a.page_size * 128)[off] = s;
      }
    }
    // stash the current token after any completion read
    if (pos >= 0 && ts >= 0) {
      if (!blk_ok) {
        if (lane == 0) atomicOr(&g_flags_kpool, ERR_SLOT);
      } else {
        __nv_bfloat16 *dk = ta.tail + blk * ta.block_stride + (pos % ta.ring) * 128 + 4 * lane;
        *reinterpret_cast<uint2 *>(dk) = *reinterpret_cast<const uint2 *>(a.key + r * a.key_sb + t * a.key_st + 4 * lane);
        *reinterpret_cast<uint2 *>(dk + ta.half_stride) =
            *reinterpret_cast<const uint2 *>(a.score + r * a.score_sb + t * a.score_st + 4 * lane);
      }
    }
  }
}

bool take_flags_kpool(cudaStream_t stream, unsigned *host_word) {
  static const unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(host_word, g_flags_kpool, sizeof(unsigned), 0, cudaMemcpyDeviceToHost,
                                stream) != cudaSuccess)
    return false;
  return cudaMemcpyToSymbolAsync(g_flags_kpool, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, stream) ==
         cudaSuccess;
}

}  // namespace kvq

using namespace kvq;

namespace kvq {
template <int KP>
static kvq_status launch_kpool_write(const KpoolParams &p, long long tiles, cudaStream_t s) {
  static int per_sm = 0;  // resident CTAs per SM, from the occupancy calculator
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kpool_write_kernel<KP>, 256, 0) != cudaSuccess || n < 1) n = 1;
    per_sm = n;
  }
  const long long cap = static_cast<long long>(sm_count() > 0 ? sm_count() : 1) * per_sm;
  kpool_write_kernel<KP><<<static_cast<unsigned>(tiles < cap ? tiles : cap), 256, 0, s>>>(p, tiles);
  return launch_status();
}
}  // namespace kvq

extern "C" kvq_status kvq_kpool_write(uint8_t *kv_cache, const void *slot_k, const float *slot_score,
                                      const float *ape, const int64_t *loc, const uint8_t *write_mask,
                                      int64_t n_pools, int32_t pool_size, int32_t head_dim, int32_t page_size,
                                      int64_t num_blocks, int32_t round_scale, kvq_stream_t stream) {
  if (n_pools < 0 || pool_size < 1 || page_size < 1 || num_blocks < 1) return KVQ_ERR_INVALID_ARG;
  if (head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (page_size % 4 != 0) return KVQ_ERR_UNSUPPORTED;  // 16-byte aligned rows of codes in every page
  if (n_pools == 0) return KVQ_OK;
  if (!kv_cache || !slot_k || !slot_score || !ape || !loc) return KVQ_ERR_INVALID_ARG;
  if (!aligned(kv_cache, 16) || !aligned(slot_k, 16) || !aligned(slot_score, 16) || !aligned(ape, 16) ||
      !aligned(loc, 8))
    return KVQ_ERR_INVALID_ARG;
  KpoolParams p;
  p.cache = kv_cache;
  p.slot_k = static_cast<const __nv_bfloat16 *>(slot_k);
  p.slot_score = slot_score;
  p.ape = ape;
  p.loc = loc;
  p.write_mask = write_mask;
  p.n_pools = n_pools;
  p.pool = pool_size;
  p.page_size = page_size;
  p.num_blocks = num_blocks;
  p.round_scale = round_scale != 0;
  const long long tiles = (n_pools + 31) / 32;
  switch (pool_size) {  // the common pool sizes unrolled
    case 4: return launch_kpool_write<4>(p, tiles, reinterpret_cast<cudaStream_t>(stream));
    case 2: return launch_kpool_write<2>(p, tiles, reinterpret_cast<cudaStream_t>(stream));
    default: return launch_kpool_write<0>(p, tiles, reinterpret_cast<cudaStream_t>(stream));
  }
}

extern "C" kvq_status kvq_kpool_seed_tail(void *tail, int64_t tail_block_stride, int64_t tail_half_stride,
                                          int32_t ring, int64_t tail_blocks, const void *key,
                                          const void *gate_score, const int32_t *tslot, int64_t n_tokens,
                                          int32_t kpool, int32_t head_dim, kvq_stream_t stream) {
  if (n_tokens < 0 || ring < 1 || tail_blocks < 1 || kpool < 1) return KVQ_ERR_INVALID_ARG;
  if (head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (n_tokens == 0) return KVQ_OK;
  if (!tail || !key || !gate_score || !tslot) return KVQ_ERR_INVALID_ARG;
  if (!aligned(tail, 8) || !aligned(key, 8) || !aligned(gate_score, 8) || !aligned(tslot, 4) ||
      tail_block_stride % 4 || tail_half_stride % 4 || tail_block_stride < 2LL * ring * 128 ||
      tail_half_stride < static_cast<long long>(ring) * 128)
    return KVQ_ERR_INVALID_ARG;
  TailArgs ta{static_cast<__nv_bfloat16 *>(tail), tail_block_stride, tail_half_stride, ring, tail_blocks};
  kpool_seed_tail_kernel<<<static_cast<unsigned>((n_tokens + 7) / 8), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      ta, static_cast<const __nv_bfloat16 *>(key), static_cast<const __nv_bfloat16 *>(gate_score), tslot, n_tokens,
      kpool);
  return launch_status();
}

extern "C" kvq_status kvq_kpool_decode_update(uint8_t *kv_cache, int32_t page_size, int64_t num_blocks, void *tail,
                                              int64_t tail_block_stride, int64_t tail_half_stride, int32_t ring,
                                              int64_t tail_blocks, const int32_t *tail_slot_mapping, const void *key,
                                              int64_t key_stride_b, int64_t key_stride_t, const void *slot_score,
                                              int64_t score_stride_b, int64_t score_stride_t, const float *ape,
                                              const int32_t *slot_mapping, const int32_t *positions,
                                              int32_t num_requests, int32_t next_n, int32_t pool_size,
                                              int32_t head_dim, int32_t round_scale, kvq_stream_t stream) {
  if (num_requests < 0 || next_n < 0 || pool_size < 1 || page_size < 1 || num_blocks < 1 || tail_blocks < 1)
    return KVQ_ERR_INVALID_ARG;
  if (head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (ring < pool_size || ring % pool_size != 0) return KVQ_ERR_INVALID_ARG;
  if (page_size % 4 != 0) return KVQ_ERR_UNSUPPORTED;
  if (num_requests == 0 || next_n == 0) return KVQ_OK;
  if (!kv_cache || !tail || !tail_slot_mapping || !key || !slot_score || !ape || !slot_mapping || !positions)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned(kv_cache, 16) || !aligned(tail, 8) || !aligned(key, 8) || !aligned(slot_score, 8) ||
      !aligned(ape, 16) || !aligned(tail_slot_mapping, 4) || !aligned(slot_mapping, 4) || !aligned(positions, 4) ||
      key_stride_b % 4 || key_stride_t % 4 || score_stride_b % 4 || score_stride_t % 4 || tail_block_stride % 4 ||
      tail_half_stride % 4 || tail_block_stride < 2LL * ring * 128 || tail_half_stride < static_cast<long long>(ring) * 128)
    return KVQ_ERR_INVALID_ARG;
  DecodeUpdateArgs a;
  a.cache = kv_cache;
  a.page_size = page_size;
  a.num_blocks = num_blocks;
  a.tail_slot = tail_slot_mapping;
  a.slot_mapping = slot_mapping;
  a.positions = positions;
  a.key = static_cast<const __nv_bfloat16 *>(key);
  a.score = static_cast<const __nv_bfloat16 *>(slot_score);
  a.key_sb = key_stride_b;
  a.key_st = key_stride_t;
  a.score_sb = score_stride_b;
  a.score_st = score_stride_t;
  a.ape = ape;
  a.R = num_requests;
  a.next_n = next_n;
  a.pool = pool_size;
  a.round_scale = round_scale != 0;
  TailArgs ta{static_cast<__nv_bfloat16 *>(tail), tail_block_stride, tail_half_stride, ring, tail_blocks};
  kpool_decode_update_kernel<<<static_cast<unsigned>((num_requests + 7) / 8), 256, 0,
                               reinterpret_cast<cudaStream_t>(stream)>>>(a, ta);
  return launch_status();
}
