// Split-KV plumbing shared by the INT4 and TurboQuant decode kernels: work partition,
// partial-result layout, and the log-sum-exp merge (+ optional inverse rotation) kernel.
//
// Partition. A CTA covers the kv heads [blockIdx.y * heads_per_cta, +heads_per_cta) of one
// contiguous piece of one or more sequences:
//   * fixed splits (num_splits = S > 0): CTA x handles sequence x / S, split x % S, i.e. the
//     positions [s * ceil(L/S), min((s + 1) * ceil(L/S), L)) -- the split range of
//     triton_turboquant_decode.py, _tq_decode_stage1; partial slot = x;
//   * balanced (num_splits = 0): the 16-token pages of the whole batch, concatenated in
//     sequence order, are cut into gridDim.x runs whose lengths differ by at most one page
//     (longer runs first, so the CTAs that touch a sequence are consecutive and non-empty);
//     CTA c walks its run and emits one partial per sequence piece, at slot c + b.
//     seg_first[b] / seg_last[b] record the first and last CTA that touched sequence b.
// Inside a CTA, warp w serves kv head w % heads_per_cta and, when heads_per_cta < 8, every
// warps_per_head-th page of the piece (warps_per_head = 8 / heads_per_cta). Every warp writes
// its own partial (sub-slot w / heads_per_cta): o = acc / l and lse = m + log2(l) in the base-2
// domain (scores are pre-multiplied by log2(e)); an empty warp writes lse = -inf.
//
// Merge (a second kernel, launched as a programmatic dependent of the first so that its launch
// overlaps the split kernel's tail): sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M) -- the stage-2
// reduction that triton_turboquant_decode.py (_fwd_kernel_stage2) and int4_per_token_head.py
// (reduce_segments) call but do not show; then, for the INT4 cache, H(o) * d1 / D
// (int4_per_token_head.py, unified_attention_int4: inverse single_rht divided by head_size).
// On request the merged log-sum-exp (M + log2 sum_s 2^(lse_s - M)) ln 2 of each row is written too
// (the lse_buf of triton_turboquant_decode.py, triton_turboquant_decode_attention).
#pragma once

#include "kvq_device.cuh"

namespace kvq {

struct SplitArgs {
  const int32_t *seq_lens;
  int32_t max_blocks;
  int32_t num_splits;  // 0 = balanced
  int32_t B, Hq, Hk, G;  // Hq: output rows per sequence (Q tokens x heads); G: heads per kv head
  int32_t Q;             // query tokens per sequence (multi-token decode; 1 otherwise)
  // Multi-token decode: the "sequences" are virtual -- vseq[v] = {block-table row, key end L (the
  // last query token's position + 1), first query / output row, query tokens (<= Q)}; Q is then
  // the largest block of query tokens one pass serves (8 / G). Null: sequence b is itself.
  const int4 *vseq;
  int32_t heads_per_cta, warps_per_head;
  int32_t seg_ctas;    // the split kernel's gridDim.x
  long long slots;     // partial slots in the workspace (before the warps_per_head factor)
  float *part_o;       // [(slots * warps_per_head), Hq, D]
  float *part_lse;     // [(slots * warps_per_head), Hq]
  int32_t *seg_first;  // [B] first / last CTA of each sequence (balanced only)
  int32_t *seg_last;
  const float *signs;  // inverse rotation of the merged output when non-null
  int32_t window;      // sliding window: keys at positions >= L - window (0 = all keys)
  const float *sinks;  // [Hq] sink logits joining each head's softmax denominator, or null
  void *out;           // [B, Hq, D] of out_dtype
  int32_t out_dtype;
  float *lse_out;      // [B, Hq] merged log-sum-exp (natural log) of every row's scores, or null
};

// ---------------------------------------------------------------------------------------------
// Range of the fp16 tensor-core operands (all decode kernels).
//
// Queries: the fp16 query operand is the query times 2^-k, k chosen per (piece, kv head) from the
// largest |q| so that no element can reach 2^15; 2^k goes into the score scale. The shift is a
// power of two, so every element keeps its value exactly.
//
// Weights: softmax is invariant to the reference it is taken against, so each query column keeps
// a reference m that is not the running maximum of its scores but a value chosen for the fp16
// P.V operands P_v = 2^(S - m) * s_v (s_v the token's value scale): l = sum 2^(S - m),
// acc = sum P_v (...), o = acc / l and lse = m + log2 l hold for any m. A step moves m (upwards
// only, rescaling l and acc by 2^(m_old - m_new)) when one of its weights passes kWeightHi or a
// score passes m + kScoreCap; the new m puts the step's largest P_v into [1, 2), and never below
// the step's largest score - kScoreCap (so 2^(S - m) <= 2^64 and l cannot overflow). Then no
// weight overflows fp16, and a token whose weight is within 2^-29 of the largest seen keeps a
// normal fp16 weight, for value scales of any magnitude.
// ---------------------------------------------------------------------------------------------
constexpr float kWeightHi = 32768.f;
constexpr float kScoreCap = 64.f;

// 3-bit value indices as P.V MMA operands (the TurboQuant layouts). s[0..3]: the index streams
// of tokens 2t, 2t + 1, 2t + 8, 2t + 9 (LSB first), the lane's dim j at bits 3j .. 3j + 2. Row r
// of m-tile mt is the lane's dim 2 mt + r, and each A register holds that dim's indices of two
// tokens as exact fp16 subnormals idx * 2^(p - 24), p = 3 (2 mt + r) mod 8 <= 7: the 16-bit
// window of each stream that holds the field is moved into the register's half by one byte
// permute and the field is masked where it lies. v3_scale(mt, r) = 2^(24 - p) undoes the scale.
__device__ __forceinline__ void v3_windows(const unsigned long long (&s)[4], uint32_t (&win)[4][3]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // stream bytes 0..3, 2..5, 4..7
    const uint32_t lo = static_cast<uint32_t>(s[i]), hi = static_cast<uint32_t>(s[i] >> 32);
    win[i][0] = lo;
    win[i][1] = __funnelshift_r(lo, hi, 16);
    win[i][2] = hi;
  }
}
__device__ __forceinline__ void v3_frag(const uint32_t (&win)[4][3], int mt, uint32_t (&a)[4]) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int bit = 3 * (2 * mt + r), jb = bit >> 3, p = bit & 7;
    const int w = jb <= 1 ? 0 : (jb <= 3 ? 1 : 2), o = jb - 2 * w;  // window and byte in it
    const uint32_t sel = o | (o + 1) << 4 | (o + 4) << 8 | (o + 5) << 12;
    const uint32_t mask = (7u << p) * 0x10001u;
#pragma unroll
    for (int tp = 0; tp < 2; ++tp) a[2 * tp + r] = __byte_perm(win[2 * tp][w], win[2 * tp + 1][w], sel) & mask;
  }
}
__host__ __device__ constexpr float v3_scale(int mt, int r) {
  return static_cast<float>(1u << (24 - ((3 * (2 * mt + r)) & 7)));
}

// Starting point of a column's new reference: the step's largest score ms for a column with no
// keys yet (ref = -inf), else the old reference raised to at least ms - kScoreCap.
__device__ __forceinline__ float ref_base(float ref, float ms) {
  return ref == -INFINITY ? ms : fmaxf(ref, ms - kScoreCap);
}
// The new reference, given the column's largest P_v wb against `base`: base + floor(log2 wb),
// at least ms - kScoreCap. A weight beyond fp32 raises ERR_RANGE.
__device__ __forceinline__ float ref_new(float base, float ms, float wb, unsigned *flags) {
  int k = 0;
  if (wb > 0.f) {
    if (!(wb < INFINITY)) atomicOr(flags, ERR_RANGE);
    k = min(ilog2f(wb), 127);
  }
  return fmaxf(base + static_cast<float>(k), ms - kScoreCap);
}

// k of the query shift for a largest element maxabs whose products may grow by up to 2^extra
// (the unnormalised Hadamard rotation: extra = log2 D): every |q| * 2^extra * 2^-k stays below
// 2^15. k is kept within [-100, 100]; a clamp at the top (|q| beyond ~2^100) raises ERR_RANGE.
// flags may be null (no report).
__device__ __forceinline__ int query_shift(float maxabs, int extra, unsigned *flags) {
  const int k = ilog2f(maxabs) + 1 + extra - 15;
  if ((k > 100 || !(maxabs < INFINITY)) && flags != nullptr) atomicOr(flags, ERR_RANGE);
  return max(-100, min(100, k));
}

__device__ __forceinline__ int clamped_len(const SplitArgs &a, int b, unsigned *flags) {
  if (a.vseq != nullptr) return a.vseq[b].y;  // clamped (and flagged) when the list was built
  int L = __ldg(a.seq_lens + b);
  const int cap = a.max_blocks * kPage;
  if (L > cap) {
    if (flags != nullptr) atomicOr(flags, ERR_SEQLEN);
    L = cap;
  }
  return L < 0 ? 0 : L;
}

// The keys of sequence b that a decode reads: positions [lo, L), lo = max(0, L - window) under a
// sliding window (unified_attention_int4, SLIDING_WINDOW) -- for nq query tokens the first one's
// window, max(0, L - nq + 1 - window) -- on the sequence's pages f .. f + np - 1.
struct SeqSpan {
  int L, lo, f, np;
};

// WIN = false: the caller's kernel runs without a window (a.window == 0), all keys are read.
template <bool WIN = true>
__device__ __forceinline__ SeqSpan seq_span(const SplitArgs &a, int b, unsigned *flags) {
  SeqSpan s;
  s.L = clamped_len(a, b, flags);
  const int nq = a.vseq != nullptr ? a.vseq[b].w : 1;
  s.lo = WIN && a.window > 0 ? max(0, s.L - nq + 1 - a.window) : 0;
  s.f = s.lo / kPage;
  s.np = s.L > 0 ? (s.L - 1) / kPage - s.f + 1 : 0;
  return s;
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

// Output rows: lane owns the D/32 consecutive dims [lane * D/32, (lane + 1) * D/32).
template <int D>
__device__ __forceinline__ void store_out(const SplitArgs &a, long long row, int lane, const float (&o)[D / 32]) {
  constexpr int V = D / 32;
  const long long e = row * D + lane * V;
  if (a.out_dtype == KVQ_F32) {
    if constexpr (V == 4)
      *reinterpret_cast<float4 *>(static_cast<float *>(a.out) + e) = make_float4(o[0], o[1], o[2], o[3]);
    else
      *reinterpret_cast<float2 *>(static_cast<float *>(a.out) + e) = make_float2(o[0], o[1]);
  } else if (a.out_dtype == KVQ_BF16) {
#pragma unroll
    for (int j = 0; j < V; j += 2)
      *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(a.out) + e + j) = __floats2bfloat162_rn(o[j], o[j + 1]);
  } else {
#pragma unroll
    for (int j = 0; j < V; j += 2)
      *reinterpret_cast<__half2 *>(static_cast<__half *>(a.out) + e + j) = __floats2half2_rn(o[j], o[j + 1]);
  }
}

// Merge the partials of (b, hq) in slots [s_lo, s_hi) and write the output row (one warp).
// Up to 16 partial rows per round trip: their log-sum-exps and their vectors are all requested
// before any is used, then combined online (running max M, weights 2^(lse - M)). Partials come
// from the split kernel's CTAs: read through L2 (ld.global.cg). sg: this lane's rotation signs
// (used when a.signs is set); sink2: the head's sink logit in base 2 (-inf: none), a partial with
// lse = sink2 and a zero vector.
template <int D>
__device__ __forceinline__ void merge_row(const SplitArgs &a, int b, int hq, long long orow, long long s_lo,
                                          long long s_hi, int lane, const float (&sg)[D / 32], float sink2) {
  constexpr int V = D / 32, R = 16;
  const int W = a.warps_per_head;
  const long long n = (s_hi - s_lo) * W, r0 = s_lo * W;  // rows (s * W + w) are contiguous
  float o[V];
#pragma unroll
  for (int j = 0; j < V; ++j) o[j] = 0.f;
  float M = -INFINITY, den = 0.f;
  for (long long i0 = 0; i0 < n; i0 += R) {
    const int cnt = static_cast<int>(min(static_cast<long long>(R), n - i0));
    const float lse = lane < cnt ? __ldcg(a.part_lse + (r0 + i0 + lane) * a.Hq + hq) : -INFINITY;
    float v[R][V];
#pragma unroll
    for (int k = 0; k < R; ++k) {
      if (k < cnt) {
        const float *src = a.part_o + ((r0 + i0 + k) * a.Hq + hq) * D + lane * V;
        if constexpr (V == 4) {
          const float4 x = __ldcg(reinterpret_cast<const float4 *>(src));
          v[k][0] = x.x; v[k][1] = x.y; v[k][2] = x.z; v[k][3] = x.w;
        } else {
          const float2 x = __ldcg(reinterpret_cast<const float2 *>(src));
          v[k][0] = x.x; v[k][1] = x.y;
        }
      }
    }
    float cm = lse;
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) cm = fmaxf(cm, __shfl_xor_sync(FULL, cm, mask));
    const float nM = fmaxf(M, cm);
    if (nM != -INFINITY) {
      const float f = M == -INFINITY ? 0.f : exp2f(M - nM);
#pragma unroll
      for (int j = 0; j < V; ++j) o[j] *= f;
      den *= f;
      M = nM;
    }
    const float w = lse == -INFINITY ? 0.f : exp2f(lse - M);
    float ws = w;
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) ws += __shfl_xor_sync(FULL, ws, mask);
    den += ws;
#pragma unroll
    for (int k = 0; k < R; ++k) {
      if (k < cnt) {
        const float wk = __shfl_sync(FULL, w, k);
#pragma unroll
        for (int j = 0; j < V; ++j) o[j] = fmaf(wk, v[k][j], o[j]);
      }
    }
  }
  if (sink2 > -INFINITY) {  // USE_SINKS: one more term of the denominator, nothing in the sum
    const float nM = fmaxf(M, sink2);
    const float f = M == -INFINITY ? 0.f : exp2f(M - nM);
#pragma unroll
    for (int j = 0; j < V; ++j) o[j] *= f;
    den = den * f + exp2f(sink2 - nM);
    M = nM;
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
  for (int j = 0; j < V; ++j) o[j] *= inv;
  if (a.lse_out != nullptr && lane == 0)  // ln(sum of e^S) = (M + log2 den) ln 2
    a.lse_out[orow] = den > 0.f ? (M + log2f(den)) * 0.6931471805599453f : -INFINITY;
  if (a.signs != nullptr) {
    // element e = lane * V + j: stages h < V inside the lane, h = V .. D/2 across lanes
    butterfly_local<V>(o);
#pragma unroll
    for (int mask = 1; mask < 32; mask <<= 1) {
#pragma unroll
      for (int j = 0; j < V; ++j) o[j] = butterfly_xor(o[j], lane, mask);
    }
#pragma unroll
    for (int j = 0; j < V; ++j) o[j] *= sg[j] * (1.0f / D);
  }
  store_out<D>(a, orow, lane, o);
}

// Calls seg(b, t0, t1, slot) for every sequence piece of this CTA (all threads, same order).
template <typename SegFn>
__device__ __forceinline__ void for_each_piece(const SplitArgs &a, unsigned *flags, SegFn &&seg) {
  if (a.num_splits > 0) {
    const int b = blockIdx.x / a.num_splits, s = blockIdx.x % a.num_splits;
    const int L = clamped_len(a, b, flags);
    const int span = (L + a.num_splits - 1) / a.num_splits;
    const int t0 = s * span;
    const int t1 = min(t0 + span, L);
    if (t0 < t1) seg(b, t0, t1, static_cast<long long>(blockIdx.x));
    return;
  }
  __shared__ long long s_scan[8];
  __shared__ long long s_first_p;
  __shared__ int s_first_b;
  long long P_tot = 0;
  for (int base = 0; base < a.B; base += 256) {
    const int b = base + threadIdx.x;
    const long long np = b < a.B ? (clamped_len(a, b, flags) + kPage - 1) / kPage : 0;
    long long chunk;
    block_scan_256(np, s_scan, &chunk);
    P_tot += chunk;
  }
  const long long C = gridDim.x, c = blockIdx.x;
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
      if (threadIdx.x == 0 && blockIdx.y == 0) {
        if (P >= pb) a.seg_first[b] = static_cast<int>(c);
        if (P + np <= pe) a.seg_last[b] = static_cast<int>(c);
      }
      seg(b, t0, t1, c + b);
    }
    P += np;
    ++b;
  }
}

// Writes one warp's partial: thread (g, t) holds, for heads 2t and 2t + 1, the D/8 consecutive
// dims [g * D/8, (g+1) * D/8) in o0 / o1; lse in base 2.
// MULTI: a.Q may exceed 1 (multi-token decode); otherwise column n is head h * G + n.
template <int D, bool MULTI = false, bool STRIDED = false>
__device__ __forceinline__ void store_partial(const SplitArgs &a, long long slot, int sub, int h,
                                              int lane, const float (&o0)[D / 8],
                                              const float (&o1)[D / 8], float lse0, float lse1) {
  const int g = lane >> 2, t = lane & 3;
  const long long row = (slot * a.warps_per_head + sub) * a.Hq;
  const int n0 = 2 * t, n1 = 2 * t + 1, ncol = MULTI ? a.G * a.Q : a.G;
  // MMA column n = query token n / G, head h * G + n % G of it
  auto row_of = [&](int n) {
    return !MULTI || a.Q == 1 ? row + static_cast<long long>(h) * a.G + n
                              : row + (n / a.G) * (a.Hq / a.Q) + static_cast<long long>(h) * a.G + n % a.G;
  };
  if (n0 < ncol) {
    const long long r0 = row_of(n0);
    float *base = a.part_o + r0 * D;
#pragma unroll
    for (int i = 0; i < D / 32; ++i)  // STRIDED: float4 i holds dims 32 i + 4 g ..; else dims g D/8 + 4 i ..
      *reinterpret_cast<float4 *>(base + (STRIDED ? 32 * i + 4 * g : g * (D / 8) + 4 * i)) =
          make_float4(o0[4 * i], o0[4 * i + 1], o0[4 * i + 2], o0[4 * i + 3]);
    if (g == 0) a.part_lse[r0] = lse0;
  }
  if (n1 < ncol) {
    const long long r1 = row_of(n1);
    float *base = a.part_o + r1 * D;
#pragma unroll
    for (int i = 0; i < D / 32; ++i)  // STRIDED: float4 i holds dims 32 i + 4 g ..; else dims g D/8 + 4 i ..
      *reinterpret_cast<float4 *>(base + (STRIDED ? 32 * i + 4 * g : g * (D / 8) + 4 * i)) =
          make_float4(o1[4 * i], o1[4 * i + 1], o1[4 * i + 2], o1[4 * i + 3]);
    if (g == 0) a.part_lse[r1] = lse1;
  }
}

// The CTA of the balanced split that holds page X of the concatenated pages: runs are
// [c q + min(c, r), ...) with q = P_tot / C, r = P_tot % C (the first r runs one page longer).
__device__ __forceinline__ long long run_of_page(long long X, long long q, long long r) {
  return X < r * (q + 1) ? X / (q + 1) : r + (X - r * (q + 1)) / q;
}

// One warp per output row (b, hq). Launched as a programmatic dependent of the split kernel:
// everything that does not depend on its results -- lengths, slot ranges (recomputed from the
// partition for B <= 256, else read from seg_first / seg_last), the rotation signs -- is done
// before griddepcontrol.wait, which holds the kernel until that grid has finished and its writes
// are visible; after it, one round trip for the partials.
template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const SplitArgs a) {
  constexpr int V = D / 32;
  __shared__ long long s_scan[8];
  __shared__ long long s_first_page[256];
  const int lane = threadIdx.x & 31;
  const long long idx = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const bool live = idx < static_cast<long long>(a.B) * a.Hq;
  const int b = live ? static_cast<int>(idx / a.Hq) : 0, hq = live ? static_cast<int>(idx % a.Hq) : 0;
  const bool scan = a.num_splits == 0 && a.B <= 256;  // uniform over the grid
  long long P_tot = 0;
  if (scan) {
    const int t = threadIdx.x;
    const long long np = t < a.B ? seq_span(a, t, nullptr).np : 0;
    const long long incl = block_scan_256(np, s_scan, &P_tot);
    s_first_page[t] = incl - np;
    __syncthreads();
  }
  float sg[V];
#pragma unroll
  for (int j = 0; j < V; ++j) sg[j] = a.signs != nullptr ? __ldg(a.signs + lane * V + j) : 0.f;
  const float sink2 = live && a.sinks != nullptr ? __ldg(a.sinks + hq % (a.Hq / a.Q)) * 1.4426950408889634f : -INFINITY;
  const SeqSpan sp = live ? seq_span(a, b, nullptr) : SeqSpan{0, 0, 0, 0};  // the split kernel already flagged it
  // the output row: row (b, hq) itself, or for a virtual sequence query token hq / heads of its
  // block (rows past its tokens belong to no query)
  long long orow = idx;
  bool owns = live;
  if (a.vseq != nullptr && live) {
    const int heads = a.Hq / a.Q, i = hq / heads;
    const int4 vs = a.vseq[b];
    owns = i < vs.w;
    orow = (static_cast<long long>(vs.z) + i) * heads + hq % heads;
  }
  const int L = sp.L;
  long long s_lo = 0, s_hi = 0;                           // slot range [s_lo, s_hi)
  bool ranged = false;
  if (L > 0 && a.num_splits > 0) {
    const int n = L - sp.lo, span = (n + a.num_splits - 1) / a.num_splits;
    s_lo = static_cast<long long>(b) * a.num_splits;
    s_hi = s_lo + (n + span - 1) / span;
    ranged = true;
  } else if (L > 0 && scan) {
    const long long C = a.seg_ctas, q = P_tot / C, r = P_tot % C;
    const long long P0 = s_first_page[b], np = sp.np;
    s_lo = run_of_page(P0, q, r) + b;
    s_hi = run_of_page(P0 + np - 1, q, r) + b + 1;
    ranged = true;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!owns) return;
  if (L == 0) {
    float z[V];
#pragma unroll
    for (int j = 0; j < V; ++j) z[j] = 0.f;
    store_out<D>(a, orow, lane, z);
    if (a.lse_out != nullptr && lane == 0)  // no key: the sink alone, if any
      a.lse_out[orow] = sink2 > -INFINITY ? sink2 * 0.6931471805599453f : -INFINITY;
    return;
  }
  if (!ranged) {
    s_lo = static_cast<long long>(a.seg_first[b]) + b;
    s_hi = static_cast<long long>(a.seg_last[b]) + b + 1;
  }
  s_lo = max(0LL, min(s_lo, a.slots));  // never index outside the workspace
  s_hi = max(s_lo, min(s_hi, a.slots));
  merge_row<D>(a, b, hq, orow, s_lo, s_hi, lane, sg, sink2);
}

}  // namespace kvq
