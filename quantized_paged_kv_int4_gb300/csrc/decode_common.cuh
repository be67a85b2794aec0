// Split-KV plumbing shared by the INT4 and TurboQuant decode kernels: work partition,
// partial-result layout, and the log-sum-exp merge (+ optional inverse rotation), fused into the
// decode kernel as a "last CTA to finish a sequence merges it" epilogue.
//
// Partition. A CTA covers the kv heads [blockIdx.y * heads_per_cta, +heads_per_cta) of one
// contiguous piece of one or more sequences:
//   * fixed splits (num_splits = S > 0): CTA x handles sequence x / S, split x % S, i.e. the
//     positions [s * ceil(L/S), min((s + 1) * ceil(L/S), L)) -- the split range of
//     triton_turboquant_decode.py, _tq_decode_stage1; partial slot = x;
//   * balanced (num_splits = 0): the 16-token pages of the whole batch, concatenated in
//     sequence order, are cut into gridDim.x runs whose lengths differ by at most one page
//     (longer runs first, so the CTAs that touch a sequence are consecutive); CTA c walks its
//     run and emits one partial per sequence piece, at slot c + b.
// Inside a CTA, warp w serves kv head w % heads_per_cta and, when heads_per_cta < 8, every
// warps_per_head-th page of the piece (warps_per_head = 8 / heads_per_cta). Every warp writes
// its own partial (sub-slot w / heads_per_cta): o = acc / l and lse = m + log2(l) in the base-2
// domain (scores are pre-multiplied by log2(e)); an empty warp writes lse = -inf.
//
// Merge. After a piece, the CTA publishes its partials (__threadfence) and takes a ticket on
// the sequence's counter; the CTA that draws the last ticket (it never waits for anyone) resets
// the counter and combines sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M) over all partials of
// the sequence -- the stage-2 reduction that triton_turboquant_decode.py (_fwd_kernel_stage2) and
// int4_per_token_head.py (reduce_segments) call but do not show -- then, for the INT4 cache,
// applies H(o) * d1 / D (int4_per_token_head.py, unified_attention_int4: inverse single_rht
// divided by head_size) and writes the output row. With the grid over head groups, the ticket
// counts (sequence, head group) pairs and the merge covers the group's query heads.
#pragma once

#include "kvq_device.cuh"

namespace kvq {

struct SplitArgs {
  const int32_t *seq_lens;
  int32_t max_blocks;
  int32_t num_splits;  // 0 = balanced
  int32_t B, Hq, Hk, G;
  int32_t heads_per_cta, warps_per_head;
  long long slots;     // partial slots in the workspace (before the warps_per_head factor)
  float *part_o;       // [(slots * warps_per_head), Hq, D]
  float *part_lse;     // [(slots * warps_per_head), Hq]
  int32_t *counters;   // [B * head_groups], zero between calls
  const float *signs;  // inverse rotation of the merged output when non-null
  void *out;           // [B, Hq, D] of out_dtype
  int32_t out_dtype;
};

__device__ __forceinline__ int clamped_len(const SplitArgs &a, int b, unsigned *flags) {
  int L = __ldg(a.seq_lens + b);
  const int cap = a.max_blocks * kPage;
  if (L > cap) {
    if (flags != nullptr) atomicOr(flags, ERR_SEQLEN);
    L = cap;
  }
  return L < 0 ? 0 : L;
}

// Block-wide inclusive scan of one int64 per thread (256 threads); returns the inclusive
// prefix and writes the block total to *total.
__device__ __forceinline__ long long block_scan_256(long long v, long long *scratch, long long *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(FULL, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  long long before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const long long s = scratch[w];
    if (w < warp) before += s;
    all += s;
  }
  __syncthreads();
  *total = all;
  return v + before;
}

template <int D>
__device__ __forceinline__ void store_out(const SplitArgs &a, long long row, int lane, const float (&o)[D / 32]) {
#pragma unroll
  for (int j = 0; j < D / 32; ++j) {
    const long long e = row * D + lane + 32 * j;
    if (a.out_dtype == KVQ_F32)
      static_cast<float *>(a.out)[e] = o[j];
    else if (a.out_dtype == KVQ_BF16)
      static_cast<__nv_bfloat16 *>(a.out)[e] = __float2bfloat16_rn(o[j]);
    else
      static_cast<__half *>(a.out)[e] = __float2half_rn(o[j]);
  }
}

// Merge the partials of (b, hq) in slots [s_lo, s_hi) and write the output row (one warp).
// Partials come from other CTAs: read through L2 (ld.global.cg), never a stale L1 line.
template <int D>
__device__ void merge_row(const SplitArgs &a, int b, int hq, long long s_lo, long long s_hi, int lane) {
  constexpr int J = D / 32;
  const int W = a.warps_per_head;
  const long long n = (s_hi - s_lo) * W, r0 = s_lo * W;  // rows (s * W + w) are contiguous
  const float *lse = a.part_lse + hq;
  float M = -INFINITY;
  for (long long i = lane; i < n; i += 32) M = fmaxf(M, __ldcg(lse + (r0 + i) * a.Hq));
#pragma unroll
  for (int mask = 16; mask >= 1; mask >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, mask));
  float o[J];
#pragma unroll
  for (int j = 0; j < J; ++j) o[j] = 0.f;
  float den = 0.f;
  for (long long i0 = 0; i0 < n; i0 += 32) {
    float wgt = 0.f;
    if (i0 + lane < n) {
      const float x = __ldcg(lse + (r0 + i0 + lane) * a.Hq);
      wgt = x == -INFINITY ? 0.f : exp2f(x - M);
    }
    den += wgt;
    const int cnt = static_cast<int>(min(32LL, n - i0));
#pragma unroll 4
    for (int k = 0; k < cnt; ++k) {
      const float wk = __shfl_sync(FULL, wgt, k);
      const float *src = a.part_o + ((r0 + i0 + k) * a.Hq + hq) * D;
#pragma unroll
      for (int j = 0; j < J; ++j) o[j] = fmaf(wk, __ldcg(src + lane + 32 * j), o[j]);
    }
  }
#pragma unroll
  for (int mask = 16; mask >= 1; mask >>= 1) den += __shfl_xor_sync(FULL, den, mask);
  const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
  for (int j = 0; j < J; ++j) o[j] *= inv;
  if (a.signs != nullptr) {
#pragma unroll
    for (int mask = 1; mask < 32; mask <<= 1) {
#pragma unroll
      for (int j = 0; j < J; ++j) o[j] = butterfly_xor(o[j], lane, mask);
    }
    butterfly_local<J>(o);
#pragma unroll
    for (int j = 0; j < J; ++j) o[j] *= __ldg(a.signs + lane + 32 * j) * (1.0f / D);
  }
  store_out<D>(a, static_cast<long long>(b) * a.Hq + hq, lane, o);
}

// Rows of the query heads this CTA's head group owns: [h0 * G, (h0 + heads_per_cta) * G).
template <int D>
__device__ void merge_sequence(const SplitArgs &a, int b, long long s_lo, long long s_hi) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.y * a.heads_per_cta * a.G, nq = a.heads_per_cta * a.G;
  s_lo = max(0LL, min(s_lo, a.slots));  // never index outside the workspace
  s_hi = max(s_lo, min(s_hi, a.slots));
  for (int i = warp; i < nq; i += 8) merge_row<D>(a, b, q0 + i, s_lo, s_hi, lane);
}

template <int D>
__device__ void zero_sequence(const SplitArgs &a, int b) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.y * a.heads_per_cta * a.G, nq = a.heads_per_cta * a.G;
  float z[D / 32];
#pragma unroll
  for (int j = 0; j < D / 32; ++j) z[j] = 0.f;
  for (int i = warp; i < nq; i += 8) store_out<D>(a, static_cast<long long>(b) * a.Hq + q0 + i, lane, z);
}

// After a piece of sequence b (slot range of the sequence [s_lo, s_hi), nseg CTAs in total):
// publish, take a ticket, and merge if this CTA is the last of the sequence.
template <int D>
__device__ void arrive_and_merge(const SplitArgs &a, int b, long long s_lo, long long s_hi, int nseg) {
  __shared__ int s_last;
  __syncthreads();  // every warp of the CTA has written its partial
  if (threadIdx.x == 0) {
    int last = 1;
    if (nseg > 1) {
      int *ctr = a.counters + static_cast<long long>(b) * gridDim.y + blockIdx.y;
      __threadfence();  // release: this CTA's partials before its ticket
      last = atomicAdd(ctr, 1) == nseg - 1;
      if (last) {
        *ctr = 0;         // every other CTA of the sequence has taken its ticket
        __threadfence();  // acquire: the other CTAs' partials after their tickets
      }
    }
    s_last = last;
  }
  __syncthreads();
  if (s_last) merge_sequence<D>(a, b, s_lo, s_hi);
}

// CTA index of global page x under the balanced cut of P pages into C runs (q = P / C,
// r = P % C: runs 0..r-1 have q + 1 pages, the others q).
__device__ __forceinline__ long long cta_of_page(long long x, long long q, long long r) {
  const long long big = r * (q + 1);
  return x < big ? x / (q + 1) : r + (x - big) / q;
}

// Calls seg(b, t0, t1, slot) for every sequence piece of this CTA (all threads, same order),
// each followed by the fused merge; also writes the zero rows of empty sequences.
template <int D, typename SegFn>
__device__ __forceinline__ void for_each_piece(const SplitArgs &a, unsigned *flags, SegFn &&seg) {
  if (a.num_splits > 0) {
    const int S = a.num_splits;
    const int b = blockIdx.x / S, s = blockIdx.x % S;
    const int L = clamped_len(a, b, flags);
    if (L == 0) {
      if (s == 0) zero_sequence<D>(a, b);
      return;
    }
    const int span = (L + S - 1) / S;
    const int t0 = s * span;
    const int t1 = min(t0 + span, L);
    if (t0 >= t1) return;
    seg(b, t0, t1, static_cast<long long>(blockIdx.x));
    const int nseg = (L + span - 1) / span;
    arrive_and_merge<D>(a, b, static_cast<long long>(b) * S, static_cast<long long>(b) * S + nseg, nseg);
    return;
  }
  __shared__ long long s_scan[8];
  __shared__ long long s_first_p;
  __shared__ int s_first_b;
  const long long C = gridDim.x, c = blockIdx.x;
  long long P_tot = 0;
  for (int base = 0; base < a.B; base += 256) {
    const int b = base + threadIdx.x;
    const long long np = b < a.B ? (clamped_len(a, b, flags) + kPage - 1) / kPage : 0;
    long long chunk;
    block_scan_256(np, s_scan, &chunk);
    P_tot += chunk;
  }
  for (long long b = c; b < a.B; b += C)  // empty sequences: CTA b % C writes their zero rows
    if (clamped_len(a, static_cast<int>(b), nullptr) == 0) zero_sequence<D>(a, static_cast<int>(b));
  const long long q = P_tot / C, r = P_tot % C;
  const long long pb = c * q + min(c, r), pe = pb + q + (c < r ? 1 : 0);
  if (pb >= pe) return;
  if (threadIdx.x == 0) s_first_b = -1;
  __syncthreads();
  long long running = 0;
  for (int base = 0; base < a.B; base += 256) {
    const int b = base + threadIdx.x;
    const long long np = b < a.B ? (clamped_len(a, b, nullptr) + kPage - 1) / kPage : 0;
    long long chunk;
    const long long incl = block_scan_256(np, s_scan, &chunk) + running;
    const long long excl = incl - np;
    if (np > 0 && excl <= pb && pb < incl) {
      s_first_b = b;
      s_first_p = excl;
    }
    running += chunk;
    __syncthreads();
    if (s_first_b >= 0) break;
  }
  int b = s_first_b;
  long long P = s_first_p;
  while (P < pe && b < a.B) {
    const int L = clamped_len(a, b, nullptr);
    const long long np = (L + kPage - 1) / kPage;
    if (np > 0) {
      const long long lo = max(pb, P) - P, hi = min(pe, P + np) - P;
      const int t0 = static_cast<int>(lo * kPage);
      const int t1 = static_cast<int>(min(hi * kPage, static_cast<long long>(L)));
      seg(b, t0, t1, c + b);
      const long long c_first = cta_of_page(P, q, r), c_last = cta_of_page(P + np - 1, q, r);
      arrive_and_merge<D>(a, b, c_first + b, c_last + b + 1, static_cast<int>(c_last - c_first + 1));
    }
    P += np;
    ++b;
  }
}

// Writes one warp's partial: thread (g, t) holds, for heads 2t and 2t + 1, the D/8 consecutive
// dims [g * D/8, (g+1) * D/8) in o0 / o1; lse in base 2.
template <int D>
__device__ __forceinline__ void store_partial(const SplitArgs &a, long long slot, int sub, int h,
                                              int lane, const float (&o0)[D / 8],
                                              const float (&o1)[D / 8], float lse0, float lse1) {
  const int g = lane >> 2, t = lane & 3;
  const long long row = (slot * a.warps_per_head + sub) * a.Hq + static_cast<long long>(h) * a.G;
  const int n0 = 2 * t, n1 = 2 * t + 1;
  if (n0 < a.G) {
    float4 *dst = reinterpret_cast<float4 *>(a.part_o + (row + n0) * D + g * (D / 8));
#pragma unroll
    for (int i = 0; i < D / 32; ++i) dst[i] = make_float4(o0[4 * i], o0[4 * i + 1], o0[4 * i + 2], o0[4 * i + 3]);
    if (g == 0) a.part_lse[row + n0] = lse0;
  }
  if (n1 < a.G) {
    float4 *dst = reinterpret_cast<float4 *>(a.part_o + (row + n1) * D + g * (D / 8));
#pragma unroll
    for (int i = 0; i < D / 32; ++i) dst[i] = make_float4(o1[4 * i], o1[4 * i + 1], o1[4 * i + 2], o1[4 * i + 3]);
    if (g == 0) a.part_lse[row + n1] = lse1;
  }
}

}  // namespace kvq
