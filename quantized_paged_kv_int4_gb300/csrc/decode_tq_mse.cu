// kvq_decode_tq_mse: split-KV paged decode attention over the TurboQuant combined slot with MSE
// keys (key_bits-bit centroid indices + an fp16 norm) and 4-bit or 3-bit uniform values.
//
// Follows triton_turboquant_decode.py, _tq_decode_stage1 with KEY_FP8 = 0 and
// triton_turboquant_decode_attention with key_fp8 = False: q_rot = q @ Pi^T (the launcher's
// GEMM; here rotate_q_kernel, fp32), per key the LSB-first index stream from byte 0 of the slot,
// the centroid gather c_d = centroids[idx_d], with NORM_CORRECTION c / sqrt(sum c^2 + 1e-16), the
// fp16 norm at byte MSE_BYTES, score = ATTN_SCALE * norm * (q_rot . c); the values start at byte
// key_packed_size (KPS) and dequantize as idx * scale + zero like the FP8-key layout; the splits
// are merged by log-sum-exp (decode_common.cuh).
//
// GB300 design: the FP8-key kernel's structure (one warp per kv head and run of pages, a per-warp
// ring of (page, head) tiles brought by one tensor-memory-accelerator box each, mma.m16n8k16 for
// both contractions), with each slot's used bytes staged as one row: KPS is usually not a multiple
// of 4 (MSE_BYTES + 2), so the fields are read from shared memory at any byte offset (aligned
// words + funnel shifts). Centroids go to the
// tensor cores as fp16 hi + lo parts: a pair table in shared memory maps two adjacent indices to
// the hi pair and the lo pair of an A-fragment register in one 8-byte load; q as fp16 hi + lo as
// in the FP8 path; three MMAs per k-step (hi.hi, hi.lo, lo.hi) keep ~22 bits of the product.

#include "decode_common.cuh"
#include "kvq_host.h"

namespace kvq {

__device__ unsigned g_flags_decode_tq_mse = 0;

struct TqMseParams {
  SplitArgs s;
  CUtensorMap map;         // the slot pool as {slot_bytes, 16, Hk, num_blocks}, box {row bytes, 16, 1, 1}
  const float *q_rot;      // [B, Hq, D] fp32 (written by rotate_q_kernel into the workspace)
  const int32_t *block_table;
  const float *centroids;  // [2^key_bits]
  int32_t kps, norm_correction;
  float sc_log2;           // attn_scale * log2(e)
  int64_t num_blocks;
  unsigned long long wait_ns;  // limit of every bounded wait on a ring slot
  int32_t withhold;            // error-path tests only: warp 0 of CTA (0, 0) never issues its ring tile `withhold`
};

constexpr uint32_t kLoMse = 0x000F000Fu;
constexpr uint32_t kHiMse = 0x00F000F0u;

template <int D, int KB, int VB>
struct MseGeom {
  static constexpr int MSE = (D * KB + 7) / 8;      // MSE_BYTES
  static constexpr int KCH = D / 4;                 // dims per lane (t) in the score MMA's k order
  static constexpr int KW = (KCH * KB + 31) / 32;   // index words per lane and row
  static constexpr int VDB = (D * VB + 7) / 8;
  static constexpr int KSTEPS = D / 16;
  static constexpr int MT = D / 16;
  static constexpr int NPAIR = 1 << (2 * KB);       // index pairs
  // pair table: entry (i0 | i1 << KB) = {fp16 hi(c_i0) | hi(c_i1) << 16, lo(c_i0) | lo(c_i1) << 16},
  // in COPIES copies side by side (entry e of copy c at byte 8 (e COPIES + c): lane l reads copy
  // l % COPIES, so lanes of a half-warp with different copies never share a bank), then the fp32
  // sums c_i0^2 + c_i1^2 (NORM_CORRECTION)
  static constexpr int COPIES = KB == 3 ? 16 : 4;   // 8 KB either way
  static constexpr int PSH = 3 + (KB == 3 ? 4 : 2); // entry index -> byte offset shift
  static constexpr int TABLE = NPAIR * 8 * COPIES + NPAIR * 4;
};

// Staged bytes of a slot holding its `used` bytes: a multiple of 16 (a box row) whose word stride
// is 4 mod 8 (rows g and g + 8 of a fragment fall in different banks), i.e. an odd multiple of 16,
// and at least used + 4: the unaligned 32-bit read of the last field (two aligned words) may take
// up to 4 bytes past it, which must stay inside the row. Bytes past the slot's end are out of the
// tensor and filled with zeros by the copy.
inline int mse_row_bytes(int used) {
  int rs = (used + 4 + 15) / 16 * 16;
  while (((rs / 4) & 7) != 4) rs += 16;
  return rs;
}

// Per-warp ring state carried from piece to piece: tiles issued so far (ring slot and mbarrier
// phase of tile K are K % NSTAGE and (K / NSTAGE) & 1), and whether a wait ran out.
struct MseRing {
  const uint8_t *ring_p;  // the warp's first ring slot
  uint32_t ring;          // its shared-window address
  uint32_t bar;           // shared address of its first mbarrier (8 bytes each)
  uint32_t used;
  bool failed;
};

// 32 bits of a shared-memory row starting at any byte offset o (two aligned words, funnel shift)
__device__ __forceinline__ uint32_t lds32_at(const uint8_t *row, int o) {
  const uint32_t *w = reinterpret_cast<const uint32_t *>(row + (o & ~3));
  return __funnelshift_r(w[0], w[1], 8 * (o & 3));
}

// N consecutive 32-bit values of a shared-memory row starting at any byte offset o (N + 1 aligned
// words, N funnel shifts)
template <int N>
__device__ __forceinline__ void lds_words_at(const uint8_t *row, int o, uint32_t (&out)[N]) {
  const uint32_t *w = reinterpret_cast<const uint32_t *>(row + (o & ~3));
  const int sh = 8 * (o & 3);
  uint32_t prev = w[0];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const uint32_t next = w[i + 1];
    out[i] = __funnelshift_r(prev, next, sh);
    prev = next;
  }
}

__device__ __forceinline__ uint32_t lds16_at(const uint8_t *row, int o) {
  return *reinterpret_cast<const uint16_t *>(row + o);  // o even
}

// q_rot[r][d] = sum_e q[r][e] * Pi[d][e] (fp32, e in order) for R = 16 rows per CTA: Pi goes to
// shared memory transposed (row e of the copy holds Pi[.][e], padded to D + 1 words so that both
// the transposing stores and the reads across d are free of bank conflicts), the R query rows as
// [e][r]; thread (d, group) accumulates rows group * RPT .. + RPT - 1 of output dim d.
constexpr int kRotRows = 16;

template <int D>
constexpr size_t rotate_q_smem() {
  return (static_cast<size_t>(D) * (D + 1) + static_cast<size_t>(D) * kRotRows) * sizeof(float);
}

template <int D>
__global__ void __launch_bounds__(256) rotate_q_kernel(const float *__restrict__ q, const float *__restrict__ Pi,
                                                       float *__restrict__ q_rot, long long rows) {
  asm volatile("griddepcontrol.launch_dependents;");  // the decode kernel may start its prologue
  constexpr int R = kRotRows, RPT = R * D / 256;  // rows per thread
  extern __shared__ __align__(16) float s_rot[];
  float *pt = s_rot, *qs = s_rot + D * (D + 1);
  const long long r0 = static_cast<long long>(blockIdx.x) * R;
#pragma unroll 4
  for (int i = threadIdx.x; i < D * D / 4; i += 256) {  // Pi[d][4 j .. 4 j + 3] -> pt[4 j + k][d]
    const int d = i / (D / 4), j = i % (D / 4);
    const float4 v = __ldg(reinterpret_cast<const float4 *>(Pi) + i);
    pt[(4 * j) * (D + 1) + d] = v.x;
    pt[(4 * j + 1) * (D + 1) + d] = v.y;
    pt[(4 * j + 2) * (D + 1) + d] = v.z;
    pt[(4 * j + 3) * (D + 1) + d] = v.w;
  }
  for (int i = threadIdx.x; i < R * D; i += 256) {
    const int r = i / D, e = i % D;
    qs[e * R + r] = r0 + r < rows ? q[(r0 + r) * D + e] : 0.f;
  }
  __syncthreads();
  const int d = threadIdx.x % D, grp = threadIdx.x / D;
  float acc[RPT];
#pragma unroll
  for (int r = 0; r < RPT; ++r) acc[r] = 0.f;
#pragma unroll 8
  for (int e = 0; e < D; ++e) {
    const float pv = pt[e * (D + 1) + d];
    const float *qe = qs + e * R + grp * RPT;
#pragma unroll
    for (int r = 0; r < RPT; ++r) acc[r] = fmaf(qe[r], pv, acc[r]);
  }
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    const long long row = r0 + grp * RPT + r;
    if (row < rows) q_rot[row * D + d] = acc[r];
  }
}

// the 2 KB-bit field at bit `bit` (a compile-time constant) of the index words w, shifted to bit
// PSH and masked: the byte offset of its pair-table entry in copy 0
template <int KB, int PSH>
__device__ __forceinline__ uint32_t pair_offset(const uint32_t *w, int bit) {
  constexpr uint32_t mask = ((1u << (2 * KB)) - 1) << PSH;
  const int wi = bit >> 5, sh = bit & 31;
  if (sh >= PSH) return __funnelshift_r(w[wi], w[wi + 1], sh - PSH) & mask;
  return (w[wi] << (PSH - sh)) & mask;
}

// PACKQ (G <= 4): the q hi parts of the G heads fill MMA columns 0..3 and the lo parts columns
// 4..7, and the MMA rows are 8 tokens' centroid hi parts (rows 0..7) and lo parts (rows 8..15),
// so one MMA per 8 tokens and k-step covers all four products; rows g and g + 8 are added, and a
// shuffle adds column n + 4 into column n (columns 4..7 then repeat heads 0..3 and are dropped).
// ctab: the power of two the table's centroids were divided by (2^kc, decode_tq_mse_kernel).
template <int D, int KB, int VB, int NSTAGE, bool PACKQ>
__device__ __forceinline__ void tq_mse_piece(const TqMseParams &p, MseRing &rg, const uint2 *table,
                                             const float *sq, float ctab, int RS, int b, int h, int sub,
                                             int t0, int t1, long long slot) {
  using Gm = MseGeom<D, KB, VB>;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.s.G, WPH = p.s.warps_per_head;
  const int KPS = p.kps;
  const int TILE = kPage * RS;
  const uint8_t *tb = reinterpret_cast<const uint8_t *>(table);
  const uint32_t copy_off = (lane & (Gm::COPIES - 1)) << 3;

  const int pg0 = t0 / kPage, pglast = (t1 - 1) / kPage;
  const int first = pg0 + sub;
  const int n_my = first <= pglast ? (pglast - first) / WPH + 1 : 0;
  const int32_t *bt_row = p.block_table + static_cast<long long>(b) * p.s.max_blocks;
  auto load_bids = [&](int batch) -> int {
    const int k = batch * 32 + lane;
    return k < n_my ? __ldg(bt_row + first + k * WPH) : 0;
  };
  int bids_cur = load_bids(0);
  int bids_next = load_bids(1);

  const uint32_t K0 = rg.used;  // this piece's tile k is ring tile K0 + k
  // tile k of the piece into its ring slot: lane 0 arms the slot's mbarrier with the tile's bytes
  // and starts the box copy (the warp has finished reading the slot: __syncwarp before the call)
  auto issue = [&](int k) {
    if (k >= n_my) return;
    const int kk = k & 31;
    if (k > 0 && kk == 0) {
      bids_cur = bids_next;
      bids_next = load_bids((k >> 5) + 1);
    }
    const int blk = __shfl_sync(FULL, bids_cur, kk);
    const bool withheld = K0 + k == static_cast<uint32_t>(p.withhold) && blockIdx.x == 0 && blockIdx.y == 0 &&
                          threadIdx.x < 32;  // its wait runs out: the error-path test
    if (lane == 0 && !withheld) {
      const bool ok = blk >= 0 && blk < p.num_blocks;
      if (!ok) atomicOr(&g_flags_decode_tq_mse, ERR_BLOCK);
      const uint32_t sl = (K0 + k) % NSTAGE;
      const uint32_t bar = rg.bar + 8 * sl;
      fence_proxy_async();  // earlier reads of the slot come before the copy that refills it
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(TILE));
      tma_load_4d(rg.ring + sl * TILE, &p.map, 0, 0, h, ok ? blk : 0, bar);
    }
  };

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float pz0 = 0.f, pz1 = 0.f;
  float acc[Gm::MT][4];
#pragma unroll
  for (int i = 0; i < Gm::MT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

#pragma unroll
  for (int k = 0; k < NSTAGE - 1; ++k) issue(k);

  // -------- q_rot -> fp16 hi / lo parts in shared memory, then B fragments. The first page
  // copies are already on their way; q_rot is written by the rotation kernel this one may
  // overlap (a programmatic dependent launch), so wait for that grid first.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float sc2;  // score scale of the piece: attn_scale * log2 e * 2^k (q shift) * 2^kc (table shift)
  // q_rot -> fp16 hi / lo B fragments, straight from global memory: lane (g, t) holds column g
  // (head g, or PACKQ: head g % 4, its hi part for g < 4 and its lo part for g >= 4) at the dims
  // KCH t .. KCH t + KCH - 1, k-step ks taking dims KCH t + 4 ks .. + 3
  uint32_t qhi[Gm::KSTEPS][2], qlo[PACKQ ? 1 : Gm::KSTEPS][2];
  {
    const int head = PACKQ ? (g & 3) : g;
    const bool live = head < G;
    const float4 *src = reinterpret_cast<const float4 *>(
        p.q_rot + (static_cast<long long>(b) * p.s.Hq + static_cast<long long>(h) * G + (live ? head : 0)) * D +
        t * Gm::KCH);
    float qv[Gm::KCH];
#pragma unroll
    for (int j = 0; j < Gm::KCH / 4; ++j) {
      const float4 v = live ? src[j] : make_float4(0.f, 0.f, 0.f, 0.f);  // written by the pre-kernel: no __ldg
      qv[4 * j] = v.x;
      qv[4 * j + 1] = v.y;
      qv[4 * j + 2] = v.z;
      qv[4 * j + 3] = v.w;
    }
    float qmax = 0.f;
#pragma unroll
    for (int j = 0; j < Gm::KCH; ++j) qmax = fmaxf(qmax, fabsf(qv[j]));
    const int qk = query_shift(warp_max(qmax), 0, &g_flags_decode_tq_mse);
    const float qdiv = pow2i(-qk);
    sc2 = p.sc_log2 * pow2i(qk) * ctab;
#pragma unroll
    for (int ks = 0; ks < Gm::KSTEPS; ++ks) {
      __half hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = qv[4 * ks + e] * qdiv;
        hi[e] = __float2half_rn(x);
        lo[e] = __float2half_rn(x - __half2float(hi[e]));
      }
      if constexpr (PACKQ) {
        const bool use_lo = g >= 4;
        qhi[ks][0] = h2_as_u32(use_lo ? __halves2half2(lo[0], lo[1]) : __halves2half2(hi[0], hi[1]));
        qhi[ks][1] = h2_as_u32(use_lo ? __halves2half2(lo[2], lo[3]) : __halves2half2(hi[2], hi[3]));
      } else {
        qhi[ks][0] = h2_as_u32(__halves2half2(hi[0], hi[1]));
        qhi[ks][1] = h2_as_u32(__halves2half2(hi[2], hi[3]));
        qlo[ks][0] = h2_as_u32(__halves2half2(lo[0], lo[1]));
        qlo[ks][1] = h2_as_u32(__halves2half2(lo[2], lo[3]));
      }
    }
  }

  int k = 0;
  for (; k < n_my; ++k) {
    issue(k + NSTAGE - 1);
    {
      const uint32_t K = K0 + k;
      const uint32_t bar = rg.bar + 8 * (K % NSTAGE), par = (K / NSTAGE) & 1;
      if (!__all_sync(FULL, mbar_try_wait(bar, par)) && !__all_sync(FULL, mbar_wait(bar, par, p.wait_ns))) {
        if (lane == 0) atomicOr(&g_flags_decode_tq_mse, ERR_TIMEOUT);
        rg.failed = true;
        break;
      }
    }
    const uint8_t *st = rg.ring_p + ((K0 + k) % NSTAGE) * TILE;
    const int nb = (first + k * WPH) * kPage;
    const bool ok0 = nb + g >= t0 && nb + g < t1;
    const bool ok1 = nb + g + 8 >= t0 && nb + g + 8 < t1;
    const uint8_t *row0 = st + g * RS, *row1 = st + (g + 8) * RS;

    // ---- scores: the lane's KCH dims of rows g, g + 8 as centroid hi / lo fp16 pairs
    uint32_t w0[Gm::KW + 1], w1[Gm::KW + 1];
    {
      uint32_t x0[Gm::KW], x1[Gm::KW];
      lds_words_at(row0, t * (Gm::KCH * KB / 8), x0);
      lds_words_at(row1, t * (Gm::KCH * KB / 8), x1);
#pragma unroll
      for (int i = 0; i < Gm::KW; ++i) {
        w0[i] = x0[i];
        w1[i] = x1[i];
      }
    }
    w0[Gm::KW] = w1[Gm::KW] = 0u;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    float ca[4] = {0.f, 0.f, 0.f, 0.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};  // PACKQ: tokens g, g + 8
    float ss0 = 0.f, ss1 = 0.f;  // sum of c^2 over the lane's dims (NORM_CORRECTION)
#pragma unroll
    for (int ks = 0; ks < Gm::KSTEPS; ++ks) {
      uint2 e0[2], e1[2];  // elements (4 ks + 2 j, + 1) of rows g, g + 8: one pair-table entry each
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int bit = (4 * ks + 2 * j) * KB;
        const uint32_t o0 = pair_offset<KB, Gm::PSH>(w0, bit), o1 = pair_offset<KB, Gm::PSH>(w1, bit);
        e0[j] = *reinterpret_cast<const uint2 *>(tb + (o0 | copy_off));
        e1[j] = *reinterpret_cast<const uint2 *>(tb + (o1 | copy_off));
        if (p.norm_correction) {
          ss0 += sq[o0 >> Gm::PSH];
          ss1 += sq[o1 >> Gm::PSH];
        }
      }
      if constexpr (PACKQ) {
        // MMA rows = 8 tokens x (centroid hi, centroid lo): a pair-table entry is exactly the
        // (row g, row g + 8) half of an A fragment, so the loads feed the MMAs directly
        mma_f16_16816(ca, e0[0].x, e0[0].y, e0[1].x, e0[1].y, qhi[ks][0], qhi[ks][1]);
        mma_f16_16816(cb, e1[0].x, e1[0].y, e1[1].x, e1[1].y, qhi[ks][0], qhi[ks][1]);
      } else {
        mma_f16_16816(c, e0[0].x, e1[0].x, e0[1].x, e1[1].x, qhi[ks][0], qhi[ks][1]);
        mma_f16_16816(c, e0[0].x, e1[0].x, e0[1].x, e1[1].x, qlo[ks][0], qlo[ks][1]);
        mma_f16_16816(c, e0[0].y, e1[0].y, e0[1].y, e1[1].y, qhi[ks][0], qhi[ks][1]);
      }
    }
    if constexpr (PACKQ) {
      c[0] = ca[0] + ca[2];  // token g: centroid hi + lo rows
      c[1] = ca[1] + ca[3];
      c[2] = cb[0] + cb[2];  // token g + 8
      c[3] = cb[1] + cb[3];
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] += __shfl_xor_sync(FULL, c[i], 2);  // q hi (t < 2) + q lo (t >= 2)
    }
    // per-token factor: attn_scale * log2(e) * norm (/ |c| under NORM_CORRECTION)
    float f0 = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16_at(row0, Gm::MSE)))) * sc2;
    float f1 = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16_at(row1, Gm::MSE)))) * sc2;
    if (p.norm_correction) {
      ss0 += __shfl_xor_sync(FULL, ss0, 1);
      ss0 += __shfl_xor_sync(FULL, ss0, 2);
      ss1 += __shfl_xor_sync(FULL, ss1, 1);
      ss1 += __shfl_xor_sync(FULL, ss1, 2);
      f0 *= rsqrtf(ss0 + 1e-16f);
      f1 *= rsqrtf(ss1 + 1e-16f);
    }
    const float s00 = ok0 ? c[0] * f0 : -INFINITY;
    const float s01 = ok0 ? c[1] * f0 : -INFINITY;
    const float s10 = ok1 ? c[2] * f1 : -INFINITY;
    const float s11 = ok1 ? c[3] * f1 : -INFINITY;

    // value scale and zero of tokens g, g + 8 (fp16 pair at KPS + VDB)
    const uint32_t sz0 = lds32_at(row0, KPS + Gm::VDB), sz1 = lds32_at(row1, KPS + Gm::VDB);
    const float2 szf0 = __half22float2(u32_as_h2(sz0)), szf1 = __half22float2(u32_as_h2(sz1));

    // online softmax against the columns' references (decode_common.cuh): p = 2^(S - m), P_v =
    // p * scale; a warp vote finds the rare step that must raise a reference
    float p00, p01, p10, p11, w00, w01, w10, w11;
    auto weights = [&](float q0, float q1) {
      p00 = fast_exp2(s00 - q0);
      p10 = fast_exp2(s10 - q0);
      p01 = fast_exp2(s01 - q1);
      p11 = fast_exp2(s11 - q1);
      w00 = ok0 ? p00 * szf0.x : 0.f;
      w01 = ok0 ? p01 * szf0.x : 0.f;
      w10 = ok1 ? p10 * szf1.x : 0.f;
      w11 = ok1 ? p11 * szf1.x : 0.f;
    };
    weights(m0 == -INFINITY ? 0.f : m0, m1 == -INFINITY ? 0.f : m1);
    const float ml0 = fmaxf(s00, s10), ml1 = fmaxf(s01, s11);
    if (__any_sync(FULL, ml0 > m0 + kScoreCap || ml1 > m1 + kScoreCap ||
                             fmaxf(fmaxf(w00, w10), fmaxf(w01, w11)) > kWeightHi)) {
      // every lane takes part in every reduction (no shuffle inside a conditional expression)
      const float ms0 = warp_max_g(ml0), ms1 = warp_max_g(ml1);
      const float wc0 = warp_max_g(fmaxf(w00, w10)), wc1 = warp_max_g(fmaxf(w01, w11));
      const bool tr0 = ms0 > m0 + kScoreCap || wc0 > kWeightHi;
      const bool tr1 = ms1 > m1 + kScoreCap || wc1 > kWeightHi;
      const float b0 = tr0 ? ref_base(m0, ms0) : m0, b1 = tr1 ? ref_base(m1, ms1) : m1;
      weights(b0 == -INFINITY ? 0.f : b0, b1 == -INFINITY ? 0.f : b1);
      const float x0 = warp_max_g(fmaxf(w00, w10)), x1 = warp_max_g(fmaxf(w01, w11));
      const float n0 = tr0 ? ref_new(b0, ms0, x0, &g_flags_decode_tq_mse) : m0;
      const float n1 = tr1 ? ref_new(b1, ms1, x1, &g_flags_decode_tq_mse) : m1;
      const float al0 = tr0 ? fast_exp2(m0 - n0) : 1.f, al1 = tr1 ? fast_exp2(m1 - n1) : 1.f;
      m0 = n0;
      m1 = n1;
      l0 *= al0;
      l1 *= al1;
      pz0 *= al0;
      pz1 *= al1;
#pragma unroll
      for (int i = 0; i < Gm::MT; ++i) {
        acc[i][0] *= al0;
        acc[i][1] *= al1;
        acc[i][2] *= al0;
        acc[i][3] *= al1;
      }
      weights(n0 == -INFINITY ? 0.f : n0, n1 == -INFINITY ? 0.f : n1);
      if (fmaxf(fmaxf(w00, w10), fmaxf(w01, w11)) > kWeightHi) atomicOr(&g_flags_decode_tq_mse, ERR_RANGE);
    }
    l0 += p00 + p10;
    l1 += p01 + p11;
    pz0 += (ok0 ? p00 * szf0.y : 0.f) + (ok1 ? p10 * szf1.y : 0.f);
    pz1 += (ok0 ? p01 * szf0.y : 0.f) + (ok1 ? p11 * szf1.y : 0.f);
    const __half2 X0 = __floats2half2_rn(w00, w10);
    const __half2 X1 = __floats2half2_rn(w01, w11);
    const int src0 = 8 * t + (g >> 1), src1 = src0 + 4;
    const uint32_t x0 = h2_as_u32(X0), x1 = h2_as_u32(X1);
    const uint32_t y0 = __shfl_sync(FULL, x0, src0), y1 = __shfl_sync(FULL, x1, src0);
    const uint32_t z0 = __shfl_sync(FULL, x0, src1), z1 = __shfl_sync(FULL, x1, src1);
    const uint32_t ya = (g & 1) ? y1 : y0, za = (g & 1) ? z1 : z0;
    const uint32_t b01 = __byte_perm(ya, za, 0x5410), b23 = __byte_perm(ya, za, 0x7632);

    // ---- O^T += V^T . P_v^T over tokens 2t, 2t+1, 2t+8, 2t+9 (rows of this stage)
    const uint8_t *ra = st + (2 * t) * RS, *rb = ra + RS, *rc = ra + 8 * RS, *rd = ra + 9 * RS;
    if constexpr (VB == 4) {
      constexpr int VW = D / 64;  // value words per lane per token (dims 8 g .. of D / 8 per lane)
      uint32_t wa[VW], wb[VW], wc[VW], wd[VW];
      const int o = KPS + g * (D / 16);
      lds_words_at(ra, o, wa);
      lds_words_at(rb, o, wb);
      lds_words_at(rc, o, wc);
      lds_words_at(rd, o, wd);
#pragma unroll
      for (int wi = 0; wi < VW; ++wi) {
        const uint32_t va = wa[wi], vb = wb[wi], vc = wc[wi], vd = wd[wi];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t sel = hf ? 0x7632u : 0x5410u;
          const uint32_t x = __byte_perm(va, vb, sel), y = __byte_perm(vc, vd, sel);
          const int mt = 4 * wi + 2 * hf;
          mma_f16_16816(acc[mt], x & kLoMse, x & kHiMse, y & kLoMse, y & kHiMse, b01, b23);
          const uint32_t x8 = x >> 8, y8 = y >> 8;
          mma_f16_16816(acc[mt + 1], x8 & kLoMse, x8 & kHiMse, y8 & kLoMse, y8 & kHiMse, b01, b23);
        }
      }
    } else {
      // 3-bit: the lane's D/8 indices per token, LSB first, from bit 3 (D/8) g of the value data
      constexpr int kV3Bytes = 3 * D / 64;
      const int off = KPS + kV3Bytes * g;
      unsigned long long w[4];
      const uint8_t *rows[4] = {ra, rb, rc, rd};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t x[2];
        lds_words_at(rows[i], off, x);
        w[i] = (static_cast<unsigned long long>(x[1]) << 32) | x[0];
      }
      uint32_t win[4][3];
      v3_windows(w, win);
#pragma unroll
      for (int mt = 0; mt < Gm::MT; ++mt) {
        uint32_t a[4];
        v3_frag(win, mt, a);
        mma_f16_16816(acc[mt], a[0], a[1], a[2], a[3], b01, b23);
      }
    }
    __syncwarp();
  }
  rg.used = K0 + static_cast<uint32_t>(n_my);
  if (rg.failed) {  // let the copies already issued land (bounded) before the CTA can exit
    for (int j = k; j < n_my && j < k + NSTAGE; ++j) {
      const uint32_t K = K0 + j;
      mbar_wait(rg.bar + 8 * (K % NSTAGE), (K / NSTAGE) & 1, 100000000ull);
    }
    return;
  }

  l0 = warp_sum_g(l0);
  l1 = warp_sum_g(l1);
  pz0 = warp_sum_g(pz0);
  pz1 = warp_sum_g(pz1);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  float o0[D / 8], o1[D / 8];
#pragma unroll
  for (int mt = 0; mt < Gm::MT; ++mt) {  // 4-bit: high nibbles enter 16x larger; 3-bit: v3_scale
    const float s0 = VB == 4 ? 16777216.f : v3_scale(mt, 0), s1 = VB == 4 ? 1048576.f : v3_scale(mt, 1);
    o0[2 * mt] = (acc[mt][0] * s0 + pz0) * inv0;
    o1[2 * mt] = (acc[mt][1] * s0 + pz1) * inv1;
    o0[2 * mt + 1] = (acc[mt][2] * s1 + pz0) * inv0;
    o1[2 * mt + 1] = (acc[mt][3] * s1 + pz1) * inv1;
  }
  const float lse0 = l0 > 0.f ? m0 + log2f(l0) : -INFINITY;
  const float lse1 = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
  store_partial<D>(p.s, slot, sub, h, lane, o0, o1, lse0, lse1);
}

extern __shared__ __align__(128) uint8_t kvq_mse_dsmem[];

template <int D, int KB, int VB, int NSTAGE, bool PACKQ>
__global__ void __launch_bounds__(256, 2) decode_tq_mse_kernel(const __grid_constant__ TqMseParams p, int RS) {
  uint8_t *smem = kvq_mse_dsmem;
  __shared__ __align__(8) uint64_t s_bar[8][NSTAGE];
  asm volatile("griddepcontrol.launch_dependents;");  // let the merge kernel's launch begin early
  using Gm = MseGeom<D, KB, VB>;
  const int warp = threadIdx.x >> 5;
  // the pair table (MseGeom::TABLE): centroids times 2^-kc (kc from the largest |centroid|, so no
  // entry can reach 2^15) split into fp16 hi + lo, two per entry
  uint2 *table = reinterpret_cast<uint2 *>(smem);
  float *sq = reinterpret_cast<float *>(smem + Gm::NPAIR * 8 * Gm::COPIES);
  float cmax = 0.f;
#pragma unroll
  for (int i = 0; i < (1 << KB); ++i) cmax = fmaxf(cmax, fabsf(__ldg(p.centroids + i)));
  const int kc = query_shift(cmax, 0, threadIdx.x == 0 ? &g_flags_decode_tq_mse : nullptr);
  const float cdiv = pow2i(-kc);
  for (int i = threadIdx.x; i < Gm::NPAIR * Gm::COPIES; i += 256) {
    const int e = i / Gm::COPIES;
    const float c0 = __ldg(p.centroids + (e & ((1 << KB) - 1))), c1 = __ldg(p.centroids + (e >> KB));
    const float d0 = c0 * cdiv, d1 = c1 * cdiv;
    const __half h0 = __float2half_rn(d0), h1 = __float2half_rn(d1);
    const __half l0 = __float2half_rn(d0 - __half2float(h0)), l1 = __float2half_rn(d1 - __half2float(h1));
    table[i] = make_uint2(static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16),
                          static_cast<uint32_t>(__half_as_ushort(l0)) | (static_cast<uint32_t>(__half_as_ushort(l1)) << 16));
    if (i % Gm::COPIES == 0) sq[e] = c0 * c0 + c1 * c1;
  }
  // ring slots: after the table, from its first 128-byte aligned offset; each warp inits its barriers
  const uint32_t dbase = smem_u32(smem);
  const uint32_t off = ((dbase + Gm::TABLE + 127u) & ~127u) - dbase + warp * NSTAGE * kPage * RS;
  MseRing rg;
  rg.ring_p = smem + off;
  rg.ring = dbase + off;
  rg.bar = smem_u32(&s_bar[warp][0]);
  rg.used = 0;
  rg.failed = false;
  if ((threadIdx.x & 31) == 0) {
    for (int i = 0; i < NSTAGE; ++i) mbar_init(rg.bar + 8 * i, 1);
    mbar_init_fence();
  }
  __syncthreads();
  const int hl = warp % p.s.heads_per_cta;
  const int sub = warp / p.s.heads_per_cta;
  const int h = blockIdx.y * p.s.heads_per_cta + hl;
  for_each_piece(p.s, &g_flags_decode_tq_mse, [&](int b, int t0, int t1, long long slot) {
    if (!rg.failed) tq_mse_piece<D, KB, VB, NSTAGE, PACKQ>(p, rg, table, sq, pow2i(kc), RS, b, h, sub, t0, t1, slot);
  });
}

constexpr int kStagesMse = 4;

bool take_flags_decode_tq_mse(cudaStream_t stream, unsigned *host_word) {
  static const unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(host_word, g_flags_decode_tq_mse, sizeof(unsigned), 0,
                                cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return false;
  return cudaMemcpyToSymbolAsync(g_flags_decode_tq_mse, &zero, sizeof(unsigned), 0,
                                 cudaMemcpyHostToDevice, stream) == cudaSuccess;
}

template <int D, int KB, int VB, bool PACKQ>
static kvq_status launch_tq_mse(TqMseParams &p, const SplitPlan &plan, const float *q, const float *Pi,
                                float *q_rot, const uint8_t *cache, int slot_bytes, int Hk, cudaStream_t s) {
  using Gm = MseGeom<D, KB, VB>;
  const int RS = mse_row_bytes(p.kps + Gm::VDB + 4);  // key part, values, scale and zero
  if (RS > 256) return KVQ_ERR_UNSUPPORTED;
  if (!tq_tensor_map(cache, p.num_blocks, Hk, slot_bytes, RS, &p.map)) return KVQ_ERR_CUDA;
  const size_t smem = Gm::TABLE + 128 + 8 * static_cast<size_t>(kStagesMse * kPage * RS);
  if (smem > 227 * 1024) return KVQ_ERR_UNSUPPORTED;
  static size_t attr_done[kMaxDevices] = {};  // the size depends on slot_bytes: the largest set so far
  if (ensure_dynamic_smem(decode_tq_mse_kernel<D, KB, VB, kStagesMse, PACKQ>, smem, attr_done) != cudaSuccess)
    return KVQ_ERR_CUDA;
  const long long rows = static_cast<long long>(p.s.B) * p.s.Hq;
  static size_t rot_done[kMaxDevices] = {};
  if (ensure_dynamic_smem(rotate_q_kernel<D>, rotate_q_smem<D>(), rot_done) != cudaSuccess) return KVQ_ERR_CUDA;
  rotate_q_kernel<D><<<static_cast<unsigned>((rows + kRotRows - 1) / kRotRows), 256, rotate_q_smem<D>(), s>>>(q, Pi, q_rot,
                                                                                                               rows);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  const dim3 grid(plan.seg_ctas, plan.head_groups);
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_tq_mse_kernel<D, KB, VB, kStagesMse, PACKQ>, p, RS) != cudaSuccess)
      return KVQ_ERR_CUDA;
  }
  if (launch_dependent(merge_kernel<D>, dim3(static_cast<unsigned>((rows + 7) / 8)), dim3(256), s, p.s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return launch_status();
}

}  // namespace kvq

using namespace kvq;

extern "C" size_t kvq_decode_tq_mse_workspace_bytes(int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                                    int32_t num_splits) {
  if (B < 0 || Hq < 1 || Hk < 1 || Hq % Hk || (D != 64 && D != 128)) return 0;
  SplitPlan plan;
  if (!make_plan(B, Hk, num_splits, &plan)) return 0;
  const size_t qbytes = (static_cast<size_t>(B) * Hq * D * sizeof(float) + 255) / 256 * 256;
  return qbytes + workspace_bytes(B, Hq, D, plan);
}

extern "C" kvq_status kvq_decode_tq_mse(const float *q, const float *rotation, const float *centroids,
                                        const uint8_t *kv_cache, int32_t slot_bytes, int32_t key_bits,
                                        int32_t key_packed_size, int32_t value_bits, int32_t norm_correction,
                                        const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens,
                                        float attn_scale, int32_t num_splits, void *workspace,
                                        size_t workspace_bytes_, float *out, int32_t B, int32_t Hq, int32_t Hk,
                                        int32_t D, int32_t block_size, int64_t num_blocks,
                                        kvq_stream_t stream) {
  if (B < 0 || Hq < 1 || Hk < 1 || max_blocks < 0 || num_splits < 0 || num_blocks < 1)
    return KVQ_ERR_INVALID_ARG;
  if (Hq % Hk != 0) return KVQ_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if ((key_bits != 3 && key_bits != 4) || (value_bits != 3 && value_bits != 4)) return KVQ_ERR_UNSUPPORTED;
  if (block_size != kPage || Hq / Hk > 8) return KVQ_ERR_UNSUPPORTED;
  const int mse = (D * key_bits + 7) / 8, vdb = (D * value_bits + 7) / 8;
  if (key_packed_size < mse + 2 || key_packed_size % 2 != 0) return KVQ_ERR_INVALID_ARG;
  if (slot_bytes % 16 != 0 || slot_bytes < key_packed_size + vdb + 4 || slot_bytes > 512) return KVQ_ERR_INVALID_ARG;
  if (!(attn_scale > 0.f) || !(attn_scale < INFINITY)) return KVQ_ERR_INVALID_ARG;
  SplitPlan plan;
  if (!make_plan(B, Hk, num_splits, &plan)) return KVQ_ERR_UNSUPPORTED;
  if (B == 0) return KVQ_OK;
  if (!q || !rotation || !centroids || !kv_cache || !block_table || !seq_lens || !out || !workspace)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(rotation, 16) || !aligned(centroids, 4) || !aligned(kv_cache, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(out, 16) || !aligned(workspace, 256))
    return KVQ_ERR_INVALID_ARG;
  if (max_blocks < 1) return KVQ_ERR_INVALID_ARG;
  if (workspace_bytes_ < kvq_decode_tq_mse_workspace_bytes(B, Hq, Hk, D, num_splits)) return KVQ_ERR_WORKSPACE;

  float *q_rot = static_cast<float *>(workspace);
  void *rest = static_cast<uint8_t *>(workspace) + (static_cast<size_t>(B) * Hq * D * sizeof(float) + 255) / 256 * 256;
  TqMseParams p;
  SplitArgs &sa = p.s;
  sa.seq_lens = seq_lens;
  sa.max_blocks = max_blocks;
  sa.num_splits = num_splits;
  sa.B = B;
  sa.Hq = Hq;
  sa.Hk = Hk;
  sa.G = Hq / Hk;
  sa.Q = 1;
  sa.heads_per_cta = plan.heads_per_cta;
  sa.warps_per_head = plan.warps_per_head;
  sa.seg_ctas = plan.seg_ctas;
  sa.slots = plan.slots;
  workspace_carve(rest, B, Hq, D, plan, &sa.part_o, &sa.part_lse, &sa.seg_first, &sa.seg_last);
  sa.signs = nullptr;
  sa.window = 0;
  sa.sinks = nullptr;
  sa.vseq = nullptr;
  sa.lse_out = nullptr;
  sa.out = out;
  sa.out_dtype = KVQ_F32;
  p.q_rot = q_rot;
  p.block_table = block_table;
  p.wait_ns = debug_wait_ns();
  p.withhold = debug_take_withhold();  // one call only
  p.centroids = centroids;
  p.kps = key_packed_size;
  p.norm_correction = norm_correction != 0;
  p.sc_log2 = static_cast<float>(static_cast<double>(attn_scale) * 1.4426950408889634);
  p.num_blocks = num_blocks;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool packq = sa.G <= 4;
#define KVQ_MSE_CASE(DD, KK, VV)                                                                     \
  if (D == DD && key_bits == KK && value_bits == VV)                                                 \
    return packq ? launch_tq_mse<DD, KK, VV, true>(p, plan, q, rotation, q_rot, kv_cache, slot_bytes, Hk, s) \
                 : launch_tq_mse<DD, KK, VV, false>(p, plan, q, rotation, q_rot, kv_cache, slot_bytes, Hk, s);
  KVQ_MSE_CASE(128, 3, 4)
  KVQ_MSE_CASE(128, 4, 4)
  KVQ_MSE_CASE(128, 3, 3)
  KVQ_MSE_CASE(128, 4, 3)
  KVQ_MSE_CASE(64, 3, 4)
  KVQ_MSE_CASE(64, 4, 4)
  KVQ_MSE_CASE(64, 3, 3)
  KVQ_MSE_CASE(64, 4, 3)
#undef KVQ_MSE_CASE
  return KVQ_ERR_UNSUPPORTED;
}
