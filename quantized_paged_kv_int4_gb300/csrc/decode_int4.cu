// kvq_decode_int4: split-KV paged decode attention over the INT4 per-(token, head) cache.
//
// Follows int4_per_token_head.py, unified_attention_int4 and _attn_packed in its decode (3D,
// segment) mode: q is rotated like the cache (bf16(H(q * d1))), the softmax scale is divided by
// D, every page of the block table is walked, nibbles are used as plain integers with the
// zero-point applied through the split-dot correction
//     S = (sum_d q_d n_d - zp * sum_d q_d) * scale_k * sm,
// values enter the P.V product as P_v = p * scale_v with the correction - sum(P_v * zp_v), and
// the per-split results are merged by log-sum-exp and rotated back (decode_common.cuh, a second
// kernel launched as a programmatic dependent).
//
// GB300 design. A CTA owns HB = min(Hk, 8) kv heads and a run of pages (balanced split: an
// equal share of all the batch's pages; fixed split: one piece of one sequence). It streams
// the run through an NS-deep ring of stages in shared memory. A stage holds 8 (page, head)
// tiles -- W = 8 / HB consecutive pages of the run, each with the CTA's HB heads -- loaded by
// four TMA copies per page: one 4-D box of the K pool (HB heads x 16 tokens x D/2 bytes, stored
// [head][token][row] with the 64B/32B swizzle that keeps the fragment reads conflict-free), the
// same for V, and the page's two blocks of scale words. Warp w reads tile w of every stage
// (head w % HB of page w / HB); the last of the 8 warps to finish with a stage refills its slot
// at once (a shared counter), so no warp waits for another to notice a free slot and there is
// no producer warp and no block-wide barrier after setup. Waits on the stage barriers are
// bounded and report a flag. Both contractions run on the tensor cores (mma.m16n8k16, fp16 operands,
// fp32 accumulation) on exact operands: a nibble pair masked into an fp16 pair with a zero
// exponent field IS the pair of fp16 subnormals n * 2^-24 (low nibble) or n * 2^-20 (high
// nibble), so one LOP3 turns 2 nibbles into MMA operands; the power of two goes into the
// per-token scale, and the zero-point is applied as the split-dot correction of the pages:
//   * S^T[16 tokens x 8 heads] = K[16 x D] . Q^T  (q of a high-nibble dim pre-divided by 16);
//   * O^T[D x 8 heads] += V^T[D x 16 tokens] . P_v^T with P_v = 2^(S - m) * scale_v in fp16, m a
//     per-column softmax reference kept so that P_v stays inside fp16 for any value scale
//     (decode_common.cuh); the V^T fragments come from ldmatrix.x4.trans.
// q enters as fp16 times a per-(sequence, kv head) power of two 2^-k (so no element can overflow),
// and 2^k joins the score scale. A pre-kernel rotates q and builds these fragments once per
// (sequence, kv head) -- per virtual sequence in multi-token calls; the split kernel, its
// programmatic dependent, sets up its run and issues its first page copies meanwhile and then
// copies the fragments (2.4 KB) at each piece start.
// The G query heads of a kv head share every K/V byte loaded (GQA); with G <= 4 in single-token
// calls the MMA's other columns score a second page (combined columns, int4_pages), otherwise
// the columns past G are padding.

#include <atomic>
#include <mutex>

#include "decode_common.cuh"
#include "kvq_host.h"

namespace kvq {

__device__ unsigned g_flags_decode_int4 = 0;

struct Int4Params {
  Int4Maps maps;  // TMA descriptors of the K / V pools and their scale words (64-byte aligned)
  SplitArgs s;
  const __nv_bfloat16 *q;
  const int32_t *block_table;
  int32_t bt_rows;  // rows of block_table (the real sequences; s.B counts virtual ones in multi-token calls)
  float sm_log2;  // softmax scale (divided by D when rotating) times log2(e)
  int64_t num_blocks;
  float softcap2;       // USE_SOFTCAP: the cap in base-2 units (cap * log2 e), 0 = off
  float inv_softcap2;
  const float *alibi;   // USE_ALIBI_SLOPES: [Hq] slopes, or null
  uint32_t *qfrag;      // the query fragments of rotate_q_int4_kernel [B][Hk][QWORDS][32 lanes]
                        // (B: the call's sequences, virtual ones in multi-token calls)
  unsigned long long wait_ns;  // limit of every bounded wait on a stage barrier
  int32_t withhold;     // error-path tests only: CTA (0, 0) never issues stage `withhold` (-1: none)
};

constexpr uint32_t kLo = 0x000F000Fu;  // low nibbles of bytes 0 and 2 -> fp16 subnormal pair n * 2^-24
constexpr uint32_t kHi = 0x00F000F0u;  // high nibbles -> fp16 subnormal pair n * 2^-20
constexpr float kTwo24 = 16777216.0f;
constexpr float kTwo20 = 1048576.0f;

template <int D>
struct Int4Geom {
  static constexpr int RB = D / 2;        // bytes per token row of one head
  static constexpr int VCH = D / 16;      // V bytes per lane per token
  static constexpr int TILE = 16 * RB;    // one (page, head) tile of one pool
  static constexpr int VOFF = 8 * TILE;   // stage layout: 8 K tiles, 8 V tiles,
  static constexpr int SOFF = 16 * TILE;  //   K scale blocks (<= 1 KB), V scale blocks (<= 1 KB)
  static constexpr int SCPOOL = 1024;
  static constexpr int STAGE = 16 * TILE + 2 * SCPOOL;  // a multiple of 1024
  static constexpr int WPR = D / 32;      // K words per lane per row
  static constexpr int KSTEPS = D / 16;
  static constexpr int MT = D / 16;       // m-tiles of the PV product
  static constexpr int QWORDS = 2 * (D / 16) + 3;   // query words per lane: qf, qs0, qs1, qmul
  static constexpr int QBYTES = (8 * D * 2 + 64) > QWORDS * 128 ? (8 * D * 2 + 64) : QWORDS * 128;
};

// One sequence of the walk over a CTA's run: index b, global index of its first read page
// (balanced split) or 0 (fixed split), its read page count, its clamped length, its first read
// key lo and the sequence page f holding it (balanced split; 0 in a fixed split, whose page
// numbers are the sequence's own).
struct SeqCursor {
  int b;
  int np;
  long long P;
  int L;
  int lo, f;
};

template <bool WIN>
__device__ __forceinline__ void seq_next(const SplitArgs &a, SeqCursor &c) {
  do {
    c.P += c.np;
    ++c.b;
    const SeqSpan sp = c.b < a.B ? seq_span<WIN>(a, c.b, nullptr) : SeqSpan{0, 0, 0, 0};
    c.L = sp.L;
    c.lo = sp.lo;
    c.f = sp.f;
    c.np = sp.np;
  } while (c.np == 0 && c.b < a.B);
}

// The CTA's run of pages (identical in all threads). Run page x is page base + x of the
// concatenation of all sequences' pages (balanced) or page base + x of sequence first.b
// (fixed split, token range [t0, t1)).
struct PageRun {
  long long base, end;  // run pages are base .. end - 1 (same numbering as SeqCursor::P)
  int n;
  bool fixed;
  int t0, t1;
  SeqCursor first;
};

template <bool WIN>
__device__ __forceinline__ bool page_run(const SplitArgs &a, unsigned *flags, PageRun *run) {
  if (a.num_splits > 0) {
    const int b = blockIdx.x / a.num_splits, s = blockIdx.x % a.num_splits;
    const SeqSpan sp = seq_span<WIN>(a, b, flags);
    const int L = sp.L;
    const int span = (L - sp.lo + a.num_splits - 1) / a.num_splits;
    const int t0 = sp.lo + s * span, t1 = min(t0 + span, L);
    if (t0 >= t1) return false;
    run->fixed = true;
    run->t0 = t0;
    run->t1 = t1;
    run->base = t0 / kPage;
    run->n = (t1 - 1) / kPage - t0 / kPage + 1;
    run->end = run->base + run->n;
    run->first.b = b;
    run->first.P = 0;
    run->first.np = 0x3fffffff;  // never left
    run->first.L = L;
    run->first.lo = sp.lo;
    run->first.f = 0;
    return true;
  }
  __shared__ long long s_scan[8];
  __shared__ long long s_first_p;
  __shared__ int s_first_b;
  const long long C = gridDim.x, c = blockIdx.x;
  if (a.B <= 256) {  // one scan finds both the total and the sequence holding the run's first page
    const int b = threadIdx.x;
    const long long np = b < a.B ? seq_span<WIN>(a, b, flags).np : 0;
    long long P_tot;
    const long long incl = block_scan_256(np, s_scan, &P_tot);
    const long long q = P_tot / C, r = P_tot % C;
    const long long pb = c * q + min(c, r), pe = pb + q + (c < r ? 1 : 0);
    if (pb >= pe) return false;
    if (np > 0 && incl - np <= pb && pb < incl) {
      s_first_b = b;
      s_first_p = incl - np;
    }
    __syncthreads();
    run->fixed = false;
    run->base = pb;
    run->end = pe;
    run->n = static_cast<int>(pe - pb);
    run->first.b = s_first_b;
    run->first.P = s_first_p;
    const SeqSpan sp = seq_span<WIN>(a, s_first_b, nullptr);
    run->first.L = sp.L;
    run->first.lo = sp.lo;
    run->first.f = sp.f;
    run->first.np = sp.np;
    return true;
  }
  long long P_tot = 0;
  for (int base = 0; base < a.B; base += 256) {
    const int b = base + threadIdx.x;
    const long long np = b < a.B ? seq_span<WIN>(a, b, flags).np : 0;
    long long chunk;
    block_scan_256(np, s_scan, &chunk);
    P_tot += chunk;
  }
  const long long q = P_tot / C, r = P_tot % C;
  const long long pb = c * q + min(c, r), pe = pb + q + (c < r ? 1 : 0);
  if (pb >= pe) return false;
  if (threadIdx.x == 0) s_first_b = -1;
  __syncthreads();
  long long running = 0;
  for (int base = 0; base < a.B; base += 256) {
    const int b = base + threadIdx.x;
    const long long np = b < a.B ? seq_span<WIN>(a, b, nullptr).np : 0;
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
  run->fixed = false;
  run->base = pb;
  run->end = pe;
  run->n = static_cast<int>(pe - pb);
  run->first.b = s_first_b;
  run->first.P = s_first_p;
  const SeqSpan sp = seq_span<WIN>(a, s_first_b, nullptr);
  run->first.L = sp.L;
  run->first.lo = sp.lo;
  run->first.f = sp.f;
  run->first.np = sp.np;
  return true;
}

// Online-softmax state of one warp for one sequence piece: per query column (2t, 2t + 1) the
// softmax reference m (decode_common.cuh), the weight sum l and the zero-point sum pz = sum P_v zp_v.
template <int D>
struct PieceState {
  float m0, m1, l0, l1, pz0, pz1;
  float acc[D / 16][4];
  __device__ __forceinline__ void reset() {
    m0 = m1 = -INFINITY;
    l0 = l1 = pz0 = pz1 = 0.f;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  }
};

// q_rot = bf16(H(q * d1)) for the G heads of kv head h of sequence b, as the fp16 B fragments
// of the score MMA (odd dims pre-divided by 16) and the per-head sums of the q the products use.
// Start copying the G * Q raw query rows of (sequence b, kv head h) -- for each of the Q query
// tokens G contiguous rows, G * D bf16 -- into this warp's area (16-byte cp.async per lane), row
// i * G + g for token i, head h * G + g; load_query waits for them.
template <int D, bool MTOK>
__device__ __forceinline__ void fetch_query(const Int4Params &p, uint8_t *qarea, int b, int h, int lane) {
  const int G = p.s.G, per = G * D / 8;
  const uint32_t dst = smem_u32(qarea);
  if (!MTOK || p.s.vseq == nullptr) {  // one token: G contiguous rows
    const uint8_t *src = reinterpret_cast<const uint8_t *>(
        p.q + (static_cast<long long>(b) * p.s.Hq + static_cast<long long>(h) * G) * D);
    for (int c = lane; c < per; c += 32) cp_async<16>(dst + 16 * c, src + 16 * c, true);
    cp_async_commit();
    return;
  }
  // a virtual sequence: its nq query tokens are q rows row0 .. row0 + nq - 1; the rows of the
  // block's other (Q - nq) tokens are zero-filled
  const int heads = p.s.Hq / p.s.Q;
  const int4 vs = p.s.vseq[b];
  for (int c = lane; c < p.s.Q * per; c += 32) {
    const int i = c / per, w = c - i * per;
    const bool ok = i < vs.w;
    const uint8_t *src = ok ? reinterpret_cast<const uint8_t *>(
                                  p.q + ((static_cast<long long>(vs.z) + i) * heads + static_cast<long long>(h) * G) * D) + 16 * w
                            : reinterpret_cast<const uint8_t *>(p.q);
    cp_async<16>(dst + 16 * c, src, ok);
  }
  cp_async_commit();
}

// qmul receives 2^k, the power of two the fp16 operands were divided by (query_shift).
template <int D, bool MTOK>
__device__ __forceinline__ void load_query(const Int4Params &p, uint8_t *qarea, int b, int h, int lane,
                                           uint32_t (&qf)[D / 16][2], float &qs0, float &qs1, float &qmul,
                                           bool fetched) {
  using Gm = Int4Geom<D>;
  constexpr int J = D / 32;
  const int g = lane >> 2, t = lane & 3, G = MTOK ? p.s.G * p.s.Q : p.s.G;  // MMA columns in use
  __half *qh = reinterpret_cast<__half *>(qarea);
  float *qsum = reinterpret_cast<float *>(qarea + 8 * D * 2);
  // The raw rows land in this warp's area (fetch_query, issued early when possible); each head is
  // then rotated and converted in place (a lane rewrites exactly the elements it read).
  __syncwarp();
  if (!fetched) {
    cp_async_wait<0>();  // a prefetch of another sequence's rows may still be landing here
    fetch_query<D, MTOK>(p, qarea, b, h, lane);
  }
  cp_async_wait<0>();
  float sg[J];
#pragma unroll
  for (int j = 0; j < J; ++j) sg[j] = p.s.signs != nullptr ? __ldg(p.s.signs + lane + 32 * j) : 1.f;
  __syncwarp();
  const __nv_bfloat16 *qraw = reinterpret_cast<const __nv_bfloat16 *>(qarea);
  // |H(q d1)| <= D max |q|: the shift that keeps every operand below 2^15 (exact)
  uint32_t qbits = 0;  // the largest |q| as bf16 bits (sign cleared: ordered like the values)
  {
    const uint32_t *qw = reinterpret_cast<const uint32_t *>(qarea);
#pragma unroll
    for (int i = 0; i < 8 * D / 64; ++i) {
      const int wi = lane + 32 * i;  // word wi holds dims 2 wi, 2 wi + 1 of the raw rows
      if (wi < G * D / 2) {
        const uint32_t v = qw[wi] & 0x7FFF7FFFu;
        qbits = max(qbits, max(v & 0xFFFFu, v >> 16));
      }
    }
  }
  const float qmax = warp_max(__uint_as_float(qbits << 16));
  const int qk = query_shift(qmax, p.s.signs != nullptr ? (D == 128 ? 7 : 6) : 0, &g_flags_decode_int4);
  qmul = pow2i(qk);
  const float qdiv = pow2i(-qk), qdiv16 = pow2i(-qk - 4);
  // four heads at a time, interleaved: their shuffle chains overlap instead of running back to back
  for (int n0 = 0; n0 < G; n0 += 4) {
    float x[4][J];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int j = 0; j < J; ++j)
        x[i][j] = n0 + i < G ? __bfloat162float(qraw[(n0 + i) * D + lane + 32 * j]) * sg[j] : 0.f;
    }
    if (p.s.signs != nullptr) {
#pragma unroll
      for (int mask = 1; mask < 32; mask <<= 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int j = 0; j < J; ++j) x[i][j] = butterfly_xor(x[i][j], lane, mask);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        butterfly_local<J>(x[i]);
#pragma unroll
        for (int j = 0; j < J; ++j) x[i][j] = bf16_round(x[i][j]);
      }
    }
    // odd dims meet high nibbles, which enter the MMA 16x larger: pre-divide q by 16 (exact);
    // the operands (and their sums) are in units of 2^k
    float eff[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      eff[i] = 0.f;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        const __half v = __float2half_rn(x[i][j] * ((e & 1) ? qdiv16 : qdiv));
        if (n0 + i < G) qh[(n0 + i) * D + e] = v;
        eff[i] += (e & 1) ? __half2float(v) * 16.f : __half2float(v);
      }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i) eff[i] += __shfl_xor_sync(FULL, eff[i], m);
    }
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (n0 + i < G) qsum[n0 + i] = eff[i] * (1.0f / kTwo24);  // sum of the q the products use
    }
  }
  for (int n = G; n < 8; ++n) {  // padded MMA columns
#pragma unroll
    for (int j = 0; j < J; ++j) qh[n * D + lane + 32 * j] = __float2half_rn(0.f);
    if (lane == 0) qsum[n] = 0.f;
  }
  __syncwarp();
  // B fragment of k-step ks = 2m + s: the dims a K word's nibbles occupy after the LOP3 split
  // (word j = WPR * t + m: low nibbles 8j + 2s, 8j + 4 + 2s; high nibbles one dim up)
  const __half *qr = qh + g * D;
#pragma unroll
  for (int ks = 0; ks < Gm::KSTEPS; ++ks) {
    const int j = Gm::WPR * t + (ks >> 1), s2 = 2 * (ks & 1);
    qf[ks][0] = h2_as_u32(__halves2half2(qr[8 * j + s2], qr[8 * j + 4 + s2]));
    qf[ks][1] = h2_as_u32(__halves2half2(qr[8 * j + 1 + s2], qr[8 * j + 5 + s2]));
  }
  qs0 = qsum[2 * t];
  qs1 = qsum[2 * t + 1];
  __syncwarp();
}

// The query fragments of (sequence b, kv head h) written by rotate_q_int4_kernel: QWORDS words per
// lane, word w of lane l at ((b Hk + h) QWORDS + w) 32 + l -- copied into the warp's query area
// (16-byte cp.async), then read by each lane.
template <int D>
__device__ __forceinline__ void fetch_frag(const Int4Params &p, uint8_t *qarea, int b, int h, int lane) {
  using Gm = Int4Geom<D>;
  const uint8_t *src = reinterpret_cast<const uint8_t *>(
      p.qfrag + (static_cast<long long>(b) * p.s.Hk + h) * Gm::QWORDS * 32);
  const uint32_t dst = smem_u32(qarea);
  for (int c = lane; c < Gm::QWORDS * 8; c += 32) cp_async<16>(dst + 16 * c, src + 16 * c, true);
  cp_async_commit();
}
template <int D>
__device__ __forceinline__ void load_frag(const Int4Params &p, uint8_t *qarea, int b, int h, int lane,
                                          uint32_t (&qf)[D / 16][2], float &qs0, float &qs1, float &qmul,
                                          bool fetched) {
  using Gm = Int4Geom<D>;
  __syncwarp();
  if (!fetched) {
    cp_async_wait<0>();
    fetch_frag<D>(p, qarea, b, h, lane);
  }
  cp_async_wait<0>();
  __syncwarp();
  const uint32_t *w = reinterpret_cast<const uint32_t *>(qarea);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    qf[k][0] = w[(2 * k) * 32 + lane];
    qf[k][1] = w[(2 * k + 1) * 32 + lane];
  }
  qs0 = __uint_as_float(w[(Gm::QWORDS - 3) * 32 + lane]);
  qs1 = __uint_as_float(w[(Gm::QWORDS - 2) * 32 + lane]);
  qmul = __uint_as_float(w[(Gm::QWORDS - 1) * 32 + lane]);
  __syncwarp();
}

// One warp per (sequence, kv head) -- virtual sequence in multi-token calls, whose MMA columns are
// its query tokens' heads -- rotates the query and builds its fp16 MMA fragments (load_query) once,
// for every CTA that walks the sequence; the split kernel is launched as its programmatic
// dependent, so the split kernel's setup and first page copies overlap this kernel, and a piece
// change inside a CTA's run costs a 2.4 KB copy instead of a rotation.
template <int D, bool MTOK>
__global__ void __launch_bounds__(256) rotate_q_int4_kernel(const __grid_constant__ Int4Params p) {
  using Gm = Int4Geom<D>;
  extern __shared__ __align__(16) uint8_t qsm[];
  asm volatile("griddepcontrol.launch_dependents;");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gw = static_cast<long long>(blockIdx.x) * 8 + warp;
  if (gw >= static_cast<long long>(p.s.B) * p.s.Hk) return;
  const int b = static_cast<int>(gw / p.s.Hk), h = static_cast<int>(gw % p.s.Hk);
  uint8_t *qarea = qsm + warp * Gm::QBYTES;
  uint32_t qf[D / 16][2];
  float qs0, qs1, qmul;
  load_query<D, MTOK>(p, qarea, b, h, lane, qf, qs0, qs1, qmul, false);
  uint32_t *dst = p.qfrag + gw * Gm::QWORDS * 32 + lane;
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    dst[(2 * k) * 32] = qf[k][0];
    dst[(2 * k + 1) * 32] = qf[k][1];
  }
  dst[(Gm::QWORDS - 3) * 32] = __float_as_uint(qs0);
  dst[(Gm::QWORDS - 2) * 32] = __float_as_uint(qs1);
  dst[(Gm::QWORDS - 1) * 32] = __float_as_uint(qmul);
}

// What a lane needs from one page after the score MMAs: its base-2 logits for tokens g, g+8 x
// heads 2t, 2t+1, and the V scale / zero-point of tokens g, g+8.
struct PageIn {
  float s[4];  // (g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
  float sv0, sv1, zv0, zv1;
};

// Shared-memory reads at 32-bit offsets from the dynamic buffer (the compiler folds constant
// parts of an offset into the instruction).
extern __shared__ __align__(16) uint8_t kvq_dsmem[];
__device__ __forceinline__ uint4 ld_s128(uint32_t o) { return *reinterpret_cast<const uint4 *>(kvq_dsmem + o); }
__device__ __forceinline__ uint2 ld_s64(uint32_t o) { return *reinterpret_cast<const uint2 *>(kvq_dsmem + o); }
__device__ __forceinline__ uint32_t ld_s32(uint32_t o) { return *reinterpret_cast<const uint32_t *>(kvq_dsmem + o); }

// This lane's fixed offsets inside a stage (stage-relative): K row g of its tile, V row 2t of its
// tile, and its K scale word of token g. The other rows it reads sit at constant distances:
// K row g+8 = +8 rows; V rows 2t+1, 2t+8, 2t+9 = +1, +8, +9 rows (the swizzle pattern repeats
// every 8 rows and is the same for rows 2t and 2t+1); token g+8's word = +8 * HB words.
template <int D>
struct LaneOffsets {
  uint32_t k, v, s;
  uint32_t vm[D / 64];  // shared address (minus the stage offset) of this lane's ldmatrix row, per load
};

template <int D, int W>
__device__ __forceinline__ LaneOffsets<D> lane_offsets(int warp, int sub, int hl, int lane) {
  using Gm = Int4Geom<D>;
  constexpr int HB = 8 / W;
  constexpr int SCP = 64 * HB < 128 ? 128 : 64 * HB;
  const int g = lane >> 2, t = lane & 3;
  LaneOffsets<D> o;
  o.k = warp * Gm::TILE + swz<Gm::RB>(g, Gm::WPR * 4 * t);
  o.v = Gm::VOFF + warp * Gm::TILE + swz<Gm::RB>(2 * t, (Gm::VCH) * g);
  o.s = Gm::SOFF + sub * SCP + (g * HB + hl) * 4;
  // ldmatrix.x4.trans load i: lanes 8m .. 8m + 7 address the 8 token rows of matrix m = (token
  // half m & 1, 16-byte chunk 2i + (m >> 1)) of the warp's V tile
  const int mi = lane >> 3, tok = (lane & 7) + 8 * (mi & 1);
#pragma unroll
  for (int i = 0; i < D / 64; ++i)
    o.vm[i] = smem_u32(kvq_dsmem) + Gm::VOFF + warp * Gm::TILE + swz<Gm::RB>(tok, 16 * (2 * i + (mi >> 1)));
  return o;
}

// c += sum_d q_d n_d (the score MMAs, all 8 columns) for the (page, head) tile at stage offset so.
template <int D>
__device__ __forceinline__ void score_mma(float (&c)[4], uint32_t so, const LaneOffsets<D> &lo,
                                          const uint32_t (&qf)[D / 16][2]) {
  using Gm = Int4Geom<D>;
  uint32_t wa[Gm::WPR], wb[Gm::WPR];
  const uint32_t ko = so + lo.k;
  if constexpr (Gm::WPR == 4) {
    const uint4 a4 = ld_s128(ko), b4 = ld_s128(ko + 8 * Gm::RB);
    wa[0] = a4.x; wa[1] = a4.y; wa[2] = a4.z; wa[3] = a4.w;
    wb[0] = b4.x; wb[1] = b4.y; wb[2] = b4.z; wb[3] = b4.w;
  } else {
    const uint2 a2 = ld_s64(ko), b2 = ld_s64(ko + 8 * Gm::RB);
    wa[0] = a2.x; wa[1] = a2.y;
    wb[0] = b2.x; wb[1] = b2.y;
  }
#pragma unroll
  for (int m = 0; m < Gm::WPR; ++m) {
    const uint32_t xa = wa[m] >> 8, xb = wb[m] >> 8;
    mma_f16_16816(c, wa[m] & kLo, wb[m] & kLo, wa[m] & kHi, wb[m] & kHi, qf[2 * m][0], qf[2 * m][1]);
    mma_f16_16816(c, xa & kLo, xb & kLo, xa & kHi, xb & kHi, qf[2 * m + 1][0], qf[2 * m + 1][1]);
  }
}

// S = (sum_d q_d n_d - zp sum_d q_d) * scale_k * sm from the MMA sums c of tokens g, g + 8, and
// their V scales / zero-points; sk = the stage offset of token g's K scale word (this lane's page).
template <int D, int HB>
__device__ __forceinline__ void score_epilogue(PageIn &pg, const float (&c)[4], uint32_t sk, float qs0, float qs1,
                                               float sm24) {
  using Gm = Int4Geom<D>;
  const uint32_t kw0 = ld_s32(sk), kw1 = ld_s32(sk + 32 * HB);
  const uint32_t vw0 = ld_s32(sk + Gm::SCPOOL), vw1 = ld_s32(sk + Gm::SCPOOL + 32 * HB);
  const float ck0 = __uint_as_float(kw0 & ~0xFu) * sm24, ck1 = __uint_as_float(kw1 & ~0xFu) * sm24;
  const float zk0 = static_cast<float>(kw0 & 0xFu), zk1 = static_cast<float>(kw1 & 0xFu);
  pg.s[0] = (c[0] - zk0 * qs0) * ck0;
  pg.s[1] = (c[1] - zk0 * qs1) * ck0;
  pg.s[2] = (c[2] - zk1 * qs0) * ck1;
  pg.s[3] = (c[3] - zk1 * qs1) * ck1;
  pg.sv0 = __uint_as_float(vw0 & ~0xFu);
  pg.sv1 = __uint_as_float(vw1 & ~0xFu);
  pg.zv0 = static_cast<float>(vw0 & 0xFu);
  pg.zv1 = static_cast<float>(vw1 & 0xFu);
}

// S = (sum_d q_d n_d - zp sum_d q_d) * scale_k * sm for one (page, head) tile at stage offset so.
template <int D, int W>
__device__ __forceinline__ void page_scores(PageIn &pg, uint32_t so, const LaneOffsets<D> &lo,
                                            const uint32_t (&qf)[D / 16][2], float qs0, float qs1, float sm24) {
  float c[4] = {0.f, 0.f, 0.f, 0.f};
  score_mma<D>(c, so, lo, qf);
  score_epilogue<D, 8 / W>(pg, c, so + lo.s, qs0, qs1, sm24);
}

// O^T += V^T . P_v^T for one (page, head) tile at stage offset so; x0 / x1 = this lane's fp16
// P_v pairs (tokens g, g+8) of heads 2t / 2t+1.
// B fragment of P_v^T from the lanes' P_v pairs: this lane needs MMA column g at tokens 2t, 2t+1
// (b01) and 2t+8, 2t+9 (b23).
__device__ __forceinline__ void pv_bfrag(uint32_t x0, uint32_t x1, int lane, uint32_t &b01, uint32_t &b23) {
  const int g = lane >> 2, t = lane & 3;
  const int src0 = 8 * t + (g >> 1), src1 = src0 + 4;
  const uint32_t y0 = __shfl_sync(FULL, x0, src0), y1 = __shfl_sync(FULL, x1, src0);
  const uint32_t z0 = __shfl_sync(FULL, x0, src1), z1 = __shfl_sync(FULL, x1, src1);
  const uint32_t ya = (g & 1) ? y1 : y0, za = (g & 1) ? z1 : z0;
  b01 = __byte_perm(ya, za, 0x5410);
  b23 = __byte_perm(ya, za, 0x7632);
}

// O^T += V^T . P_v^T for the (page, head) tile at stage offset so, given the B fragment.
template <int D>
__device__ __forceinline__ void pv_mma(float (&acc)[D / 16][4], uint32_t so, const LaneOffsets<D> &lo,
                                       uint32_t b01, uint32_t b23) {
  // V^T fragments: ldmatrix.trans gives this lane word 8q + g of tokens (2t, 2t+1) [x] and
  // (2t+8, 2t+9) [y]; its low / high nibbles of byte 0 (then byte 1) are A rows g / g + 8
#pragma unroll
  for (int i = 0; i < D / 64; ++i) {
    uint32_t r[4];
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(lo.vm[i] + so));
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t x = r[2 * e], y = r[2 * e + 1];
      const int mt = 2 * (2 * i + e);
      mma_f16_16816(acc[mt], x & kLo, x & kHi, y & kLo, y & kHi, b01, b23);
      const uint32_t x8 = x >> 8, y8 = y >> 8;
      mma_f16_16816(acc[mt + 1], x8 & kLo, x8 & kHi, y8 & kLo, y8 & kHi, b01, b23);
    }
  }
}

template <int D>
__device__ __forceinline__ void page_pv(float (&acc)[D / 16][4], uint32_t so, const LaneOffsets<D> &lo,
                                        uint32_t x0, uint32_t x1, int lane) {
  uint32_t b01, b23;
  pv_bfrag(x0, x1, lane, b01, b23);
  pv_mma<D>(acc, so, lo, b01, b23);
}

// tanh(y) = 1 - 2 / (e^(2y) + 1) with the hardware base-2 exponential; |y| is limited to 10
// (tanh(10) rounds to 1 in fp32). The absolute error (a few 1e-7) is what the soft cap passes on.
__device__ __forceinline__ float tanh_fast(float y) {
  const float e = fast_exp2(fminf(fmaxf(y, -10.f), 10.f) * 2.8853900817779268f);  // e^(2y)
  return 1.f - __fdividef(2.f, e + 1.f);
}

// Score modifiers of one warp (unified_attention_int4's USE_SOFTCAP and USE_ALIBI_SLOPES), in
// base-2 units: S = cap2 tanh(S / cap2) (cap2 and its inverse stay in the kernel parameters),
// then S += slope2 * (n - qpos) for the lane's two columns, qpos the position of the column's
// query token.
struct ScoreMods {
  float sl0, sl1;
  int qp0, qp1;
};

// NP consecutive pages of this warp (stage offsets so[0..NP-1]) inside one piece: scores, one
// online softmax step over their 16 * NP tokens, P.V.
// COMB (single-token decode with G <= 4 heads per kv head): the MMA's 8 columns carry the G heads
// twice (columns n and n + 4 hold head n), and a pair of pages is split over them -- columns 0..3
// score the first page, columns 4..7 the second -- so each lane's softmax handles 4 live scores
// instead of 8 of which half are padding. Columns 0..3 and 4..7 are two independent softmax
// streams over the piece's pages (a single page, MASKED, goes to columns 0..3 only), combined by
// comb_merge at the end of the piece. MASKED: some rows of the (single) page lie
// outside [t0, t1) -- the ragged end of a sequence, a fixed split boundary or the start of a
// sliding window -- and may hold never-written scale words (NaN): they are selected away, never
// multiplied; in multi-token decode a column's keys are also limited to its own query token's
// range [lw0, lim0) / [lw1, lim1) for the lane's columns 2t / 2t + 1 (causal limit, window).
// MODS: apply the score modifiers md (page i's row 0 is at position nb + 16 W i).
template <int D, int W, int NP, bool MASKED, bool MODS, bool MTOK, bool COMB>
__device__ __forceinline__ void int4_pages(PieceState<D> &st, const uint32_t (&so)[2], const LaneOffsets<D> &lo,
                                           const uint32_t (&qf)[D / 16][2], float qs0, float qs1, float sm24,
                                           int lane, int nb, int t0, int t1, int lim0, int lim1, int lw0,
                                           int lw1, const Int4Params &p, const ScoreMods &md) {
  using Gm = Int4Geom<D>;
  static_assert(!COMB || !MTOK, "combined columns: single-token decode only");
  constexpr bool PAIRED = COMB && NP == 2;  // two pages over the two column halves
  constexpr int NQ = PAIRED ? 1 : NP;       // pages of softmax operands per lane
  const int g = lane >> 2;
  const bool hi_half = (lane & 3) >= 2;  // this lane's columns are 4..7
  PageIn pg[NQ];
  if constexpr (PAIRED) {
    float ca[4] = {0.f, 0.f, 0.f, 0.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};
    score_mma<D>(ca, so[0], lo, qf);
    score_mma<D>(cb, so[1], lo, qf);
    float c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = hi_half ? cb[j] : ca[j];
    score_epilogue<D, 8 / W>(pg[0], c, (hi_half ? so[1] : so[0]) + lo.s, qs0, qs1, sm24);
  } else {
#pragma unroll
    for (int i = 0; i < NP; ++i) page_scores<D, W>(pg[i], so[i], lo, qf, qs0, qs1, sm24);
  }
  if constexpr (MODS) {
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      if (p.softcap2 > 0.f) {
#pragma unroll
        for (int j = 0; j < 4; ++j) pg[i].s[j] = p.softcap2 * tanh_fast(pg[i].s[j] * p.inv_softcap2);
      }
      if (p.alibi != nullptr) {
        // token g's position (token g + 8: n + 8); a paired lane of columns 4..7 scores the second page
        const int n = nb + (PAIRED ? (hi_half ? W * kPage : 0) : i * W * kPage) + g;
        const float e0 = static_cast<float>(n - md.qp0), e1 = static_cast<float>(n - md.qp1);
        pg[i].s[0] = fmaf(md.sl0, e0, pg[i].s[0]);
        pg[i].s[1] = fmaf(md.sl1, e1, pg[i].s[1]);
        pg[i].s[2] = fmaf(md.sl0, e0 + 8.f, pg[i].s[2]);
        pg[i].s[3] = fmaf(md.sl1, e1 + 8.f, pg[i].s[3]);
      }
    }
  }
  bool ok00 = true, ok01 = true, ok10 = true, ok11 = true;  // (token g / g + 8, column 2t / 2t + 1)
  if (MASKED) {
    const bool ok0 = nb + g >= t0 && nb + g < t1;
    const bool ok1 = nb + g + 8 >= t0 && nb + g + 8 < t1;
    ok00 = ok01 = ok0;
    ok10 = ok11 = ok1;
    if constexpr (MTOK) {  // multi-token decode: each column's own key range
      ok00 = ok00 && nb + g < lim0 && nb + g >= lw0;
      ok01 = ok01 && nb + g < lim1 && nb + g >= lw1;
      ok10 = ok10 && nb + g + 8 < lim0 && nb + g + 8 >= lw0;
      ok11 = ok11 && nb + g + 8 < lim1 && nb + g + 8 >= lw1;
    }
    if constexpr (COMB) {  // a single page belongs to columns 0..3
      ok00 = ok00 && !hi_half;
      ok01 = ok01 && !hi_half;
      ok10 = ok10 && !hi_half;
      ok11 = ok11 && !hi_half;
    }
    pg[0].s[0] = ok00 ? pg[0].s[0] : -INFINITY;
    pg[0].s[1] = ok01 ? pg[0].s[1] : -INFINITY;
    pg[0].s[2] = ok10 ? pg[0].s[2] : -INFINITY;
    pg[0].s[3] = ok11 ? pg[0].s[3] : -INFINITY;
  }
  // ---- online softmax (base 2): weights p = 2^(S - m) and P.V operands w = p * scale_v against
  // each column's reference m (decode_common.cuh); one warp vote finds a step in which a score
  // passes m + kScoreCap or a weight passes kWeightHi, and only then (rarely) are the columns'
  // maxima reduced, their references raised and the running sums rescaled.
  uint32_t X0[NQ], X1[NQ];  // this lane's fp16 P_v pairs (tokens g, g+8) of columns 2t, 2t+1
  float ls0, ls1, wm0, wm1;  // the step's weight sums and largest P_v per column
  auto weights = [&](float q0, float q1) {
    ls0 = ls1 = wm0 = wm1 = 0.f;
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      const float p00 = fast_exp2(pg[i].s[0] - q0), p10 = fast_exp2(pg[i].s[2] - q0);
      const float p01 = fast_exp2(pg[i].s[1] - q1), p11 = fast_exp2(pg[i].s[3] - q1);
      ls0 += p00 + p10;
      ls1 += p01 + p11;
      float w00 = p00 * pg[i].sv0, w10 = p10 * pg[i].sv1, w01 = p01 * pg[i].sv0, w11 = p11 * pg[i].sv1;
      if (MASKED) {  // never-written rows may hold NaN scale words: select them away
        w00 = ok00 ? w00 : 0.f;
        w01 = ok01 ? w01 : 0.f;
        w10 = ok10 ? w10 : 0.f;
        w11 = ok11 ? w11 : 0.f;
      }
      wm0 = fmaxf(wm0, fmaxf(w00, w10));
      wm1 = fmaxf(wm1, fmaxf(w01, w11));
      X0[i] = h2_as_u32(__floats2half2_rn(w00, w10));
      X1[i] = h2_as_u32(__floats2half2_rn(w01, w11));
    }
  };
  weights(st.m0 == -INFINITY ? 0.f : st.m0, st.m1 == -INFINITY ? 0.f : st.m1);
  float ml0 = fmaxf(pg[0].s[0], pg[0].s[2]), ml1 = fmaxf(pg[0].s[1], pg[0].s[3]);
#pragma unroll
  for (int i = 1; i < NQ; ++i) {
    ml0 = fmaxf(ml0, fmaxf(pg[i].s[0], pg[i].s[2]));
    ml1 = fmaxf(ml1, fmaxf(pg[i].s[1], pg[i].s[3]));
  }
  if (__builtin_expect(__any_sync(FULL, ml0 > st.m0 + kScoreCap || ml1 > st.m1 + kScoreCap || fmaxf(wm0, wm1) > kWeightHi), 0)) {
    // every lane takes part in every reduction (no shuffle inside a conditional expression)
    const float ms0 = warp_max_g(ml0), ms1 = warp_max_g(ml1);
    const float wc0 = warp_max_g(wm0), wc1 = warp_max_g(wm1);
    const bool tr0 = ms0 > st.m0 + kScoreCap || wc0 > kWeightHi;
    const bool tr1 = ms1 > st.m1 + kScoreCap || wc1 > kWeightHi;
    const float b0 = tr0 ? ref_base(st.m0, ms0) : st.m0, b1 = tr1 ? ref_base(st.m1, ms1) : st.m1;
    const float q0 = b0 == -INFINITY ? 0.f : b0, q1 = b1 == -INFINITY ? 0.f : b1;
    float x0 = 0.f, x1 = 0.f;  // the largest P_v per column against the bases
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      const float a00 = fast_exp2(pg[i].s[0] - q0) * pg[i].sv0, a10 = fast_exp2(pg[i].s[2] - q0) * pg[i].sv1;
      const float a01 = fast_exp2(pg[i].s[1] - q1) * pg[i].sv0, a11 = fast_exp2(pg[i].s[3] - q1) * pg[i].sv1;
      x0 = fmaxf(x0, fmaxf(ok00 ? a00 : 0.f, ok10 ? a10 : 0.f));
      x1 = fmaxf(x1, fmaxf(ok01 ? a01 : 0.f, ok11 ? a11 : 0.f));
    }
    x0 = warp_max_g(x0);
    x1 = warp_max_g(x1);
    const float n0 = tr0 ? ref_new(b0, ms0, x0, &g_flags_decode_int4) : st.m0;
    const float n1 = tr1 ? ref_new(b1, ms1, x1, &g_flags_decode_int4) : st.m1;
    const float al0 = tr0 ? fast_exp2(st.m0 - n0) : 1.f;  // 0 for a column that had no keys yet
    const float al1 = tr1 ? fast_exp2(st.m1 - n1) : 1.f;
    st.m0 = n0;
    st.m1 = n1;
    st.l0 *= al0;
    st.l1 *= al1;
    st.pz0 *= al0;
    st.pz1 *= al1;
#pragma unroll
    for (int i = 0; i < Gm::MT; ++i) {
      st.acc[i][0] *= al0;
      st.acc[i][1] *= al1;
      st.acc[i][2] *= al0;
      st.acc[i][3] *= al1;
    }
    weights(n0 == -INFINITY ? 0.f : n0, n1 == -INFINITY ? 0.f : n1);
    if (fmaxf(wm0, wm1) > kWeightHi) atomicOr(&g_flags_decode_int4, ERR_RANGE);
  }
  st.l0 += ls0;
  st.l1 += ls1;
#pragma unroll
  for (int i = 0; i < NQ; ++i) {  // sum P_v * zp_v (the fp16 P_v the products use)
    const float2 f0 = __half22float2(u32_as_h2(X0[i])), f1 = __half22float2(u32_as_h2(X1[i]));
    st.pz0 += f0.x * pg[i].zv0 + f0.y * pg[i].zv1;
    st.pz1 += f1.x * pg[i].zv0 + f1.y * pg[i].zv1;
  }
  // ---- O^T += V^T . P_v^T
  if constexpr (PAIRED) {  // columns 0..3 take the first page's V, columns 4..7 the second's
    uint32_t b01, b23;
    pv_bfrag(X0[0], X1[0], lane, b01, b23);
    const bool lo_col = g < 4;  // this lane supplies MMA column g of the B fragment
    pv_mma<D>(st.acc, so[0], lo, lo_col ? b01 : 0u, lo_col ? b23 : 0u);
    pv_mma<D>(st.acc, so[1], lo, lo_col ? 0u : b01, lo_col ? 0u : b23);
  } else {
#pragma unroll
    for (int i = 0; i < NP; ++i) page_pv<D>(st.acc, so[i], lo, X0[i], X1[i], lane);
  }
}

// Epilogue of one piece: undo the subnormal scaling, apply the zero-point term, normalise, and
// write the warp's partial (an empty piece writes zeros with lse = -inf).
// COMB: fold the softmax stream of columns 4..7 into columns 0..3 (lanes t and t ^ 2 hold the
// same heads): each side is rescaled from its reference to the larger one (a side with no keys,
// reference -inf, contributes nothing).
template <int D>
__device__ __forceinline__ void comb_merge(PieceState<D> &st) {
  auto fold = [&](float &m, float &l, float &pz, int j0, int j1) {
    const float mo = __shfl_xor_sync(FULL, m, 2), lo = __shfl_xor_sync(FULL, l, 2);
    const float pzo = __shfl_xor_sync(FULL, pz, 2);
    const float mn = fmaxf(m, mo);
    const float a = m == -INFINITY ? 0.f : fast_exp2(m - mn), ao = mo == -INFINITY ? 0.f : fast_exp2(mo - mn);
    m = mn;
    l = l * a + lo * ao;
    pz = pz * a + pzo * ao;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      const float x0 = __shfl_xor_sync(FULL, st.acc[i][j0], 2), x1 = __shfl_xor_sync(FULL, st.acc[i][j1], 2);
      st.acc[i][j0] = st.acc[i][j0] * a + x0 * ao;
      st.acc[i][j1] = st.acc[i][j1] * a + x1 * ao;
    }
  };
  fold(st.m0, st.l0, st.pz0, 0, 2);  // column 2t: acc[.][0] (row g), acc[.][2] (row g + 8)
  fold(st.m1, st.l1, st.pz1, 1, 3);  // column 2t + 1
}

template <int D, bool MTOK, bool COMB>
__device__ __forceinline__ void int4_finish(const SplitArgs &a, PieceState<D> &st, long long slot, int sub,
                                            int h, int lane) {
  using Gm = Int4Geom<D>;
  if constexpr (COMB) comb_merge<D>(st);
  const float l0 = warp_sum_g(st.l0), l1 = warp_sum_g(st.l1);
  const float pz0 = warp_sum_g(st.pz0), pz1 = warp_sum_g(st.pz1);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  float o0[D / 8], o1[D / 8];
#pragma unroll
  for (int mt = 0; mt < Gm::MT; ++mt) {
    o0[2 * mt] = (st.acc[mt][0] * kTwo24 - pz0) * inv0;
    o1[2 * mt] = (st.acc[mt][1] * kTwo24 - pz1) * inv1;
    o0[2 * mt + 1] = (st.acc[mt][2] * kTwo20 - pz0) * inv0;
    o1[2 * mt + 1] = (st.acc[mt][3] * kTwo20 - pz1) * inv1;
  }
  const float lse0 = l0 > 0.f ? st.m0 + log2f(l0) : -INFINITY;
  const float lse1 = l1 > 0.f ? st.m1 + log2f(l1) : -INFINITY;
  store_partial<D, MTOK, true>(a, slot, sub, h, lane, o0, o1, lse0, lse1);
}

// W = warps per kv head (8 / heads per CTA). Stage k of the ring (slot k % NS) holds run pages
// k * W .. k * W + W - 1 for the CTA's HB = 8 / W heads; warp w reads tile w of it.
// Ring protocol: s_full[slot] completes when a stage's copies have landed (one arrival: the
// expect_tx of the issuing lane 0, plus the copies' bytes). Every warp done with a stage adds 1 to
// s_done[slot] (acquire-release); the warp whose addition completes a multiple of 8 is the last
// reader and issues stage k + NS into the slot. Warp 0 issues the first stages and keeps the
// CTA's block ids in a shared ring two batches of 32 pages ahead of its own position (a refill
// is at most NS * W <= 32 pages ahead of the slowest warp).
// VAR 0: plain; 1: score modifiers (window, soft cap, ALiBi; multi-token decode allowed);
// 2: multi-token decode only; 3: plain with combined columns (G <= 4, see int4_pages);
// 4: score modifiers, single-token, combined columns (G <= 4).
template <int D, int NS, int W, int VAR>
__global__ void __launch_bounds__(256, 2) decode_int4_kernel(const __grid_constant__ Int4Params p) {
  constexpr bool MODS = VAR == 1 || VAR == 4, MTOK = VAR == 1 || VAR == 2, COMB = VAR == 3 || VAR == 4;
  using Gm = Int4Geom<D>;
  constexpr int HB = 8 / W;
  constexpr int SCP = 64 * HB < 128 ? 128 : 64 * HB;  // one page's scale block, 128-byte aligned slots
  static_assert(NS >= 2 && NS * W <= 32, "refills read at most two batches of block ids ahead");
  __shared__ __align__(8) uint64_t s_full[NS];
  __shared__ unsigned s_done[NS];   // warps done with each slot, counted up forever (mod 8 = this round)
  __shared__ int s_bids[128];       // block ids of run pages: batch c (32 pages) at (c % 4) * 32
  asm volatile("griddepcontrol.launch_dependents;");  // let the merge kernel's launch begin early
  // stages start at the first 1024-byte aligned offset of the dynamic buffer (swizzled TMA tiles)
  const uint32_t dbase = smem_u32(kvq_dsmem);
  const uint32_t base = (1024u - (dbase & 1023u)) & 1023u;
  const SplitArgs &a = p.s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = warp % HB, sub = warp / HB;
  const int h0 = blockIdx.y * HB, h = h0 + hl;
  const bool split_heads = a.Hk > 8;

  {  // pull the block table into L2 while the run is planned (each CTA a slice of 128-byte lines)
    const long long bytes = static_cast<long long>(p.bt_rows) * a.max_blocks * 4;
    const long long lines = (bytes + 127) / 128, per = (lines + gridDim.x - 1) / gridDim.x;
    const long long l0 = static_cast<long long>(blockIdx.x) * per;
    for (long long l = l0 + threadIdx.x; l < l0 + per && l < lines; l += blockDim.x)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(p.block_table) + l * 128));
  }
  PageRun run;
  if (!page_run<MODS>(a, &g_flags_decode_int4, &run)) return;  // uniform over the CTA
  const int n_stages = (run.n + W - 1) / W;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      s_done[i] = 0;
    }
    mbar_init_fence();
  }

  // ---- producer state (warp 0): block ids, 32 run pages per batch, lane l of a batch register
  // holding run page 32 * batch + l; each lane walks its own sequence cursor (monotone).
  SeqCursor lc = run.first;
  auto load_batch = [&](int k) -> int {
    const int x = k * 32 + lane;
    if (x >= run.n) return 0;
    const long long X = run.base + x;
    while (X >= lc.P + lc.np && lc.b < a.B) seq_next<MODS>(a, lc);
    if (lc.b >= a.B) return -1;
    const long long row = a.vseq != nullptr ? a.vseq[lc.b].x : lc.b;  // a virtual sequence: its sequence's row
    return __ldg(p.block_table + row * a.max_blocks + (X - lc.P + lc.f));
  };
  auto store_batch = [&](int c) {  // warp 0: block ids of batch c into the shared ring
    if (c * 32 < run.n) s_bids[(c & 3) * 32 + lane] = load_batch(c);
  };
  // Stage k into ring slot `slot`: lane i copies page k * W + i (expect_tx first, by lane 0).
  auto issue = [&](int k, int slot) {  // warp-wide
    if (k == p.withhold && blockIdx.x == 0 && blockIdx.y == 0) return;  // its full barrier never completes
    const int x0 = k * W, npg = min(W, run.n - x0);
    const uint32_t bar = smem_u32(&s_full[slot]);
    const uint32_t stg = dbase + base + slot * Gm::STAGE;
    const int xi = x0 + (lane < npg ? lane : 0);
    const int raw = s_bids[((xi >> 5) & 3) * 32 + (xi & 31)];
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(npg * (2 * HB * Gm::TILE + 2 * 64 * HB)));
    __syncwarp();
    if (lane < npg) {
      const bool ok = raw >= 0 && raw < p.num_blocks;
      if (!ok) atomicOr(&g_flags_decode_int4, ERR_BLOCK);
      const int blk = ok ? raw : 0;  // out of range: flagged, page 0 read instead
      fence_proxy_async();  // the earlier reads of this slot come before the copies that refill it
      tma_load_4d(stg + lane * HB * Gm::TILE, &p.maps.k, 0, 0, h0, blk, bar);
      tma_load_4d(stg + Gm::VOFF + lane * HB * Gm::TILE, &p.maps.v, 0, 0, h0, blk, bar);
      const uint32_t ks = stg + Gm::SOFF + lane * SCP, vs = ks + Gm::SCPOOL;
      if (split_heads) {
        tma_load_3d(ks, &p.maps.ks, h0, 0, blk, bar);
        tma_load_3d(vs, &p.maps.vs, h0, 0, blk, bar);
      } else {
        tma_load_2d(ks, &p.maps.ks, 0, blk, bar);
        tma_load_2d(vs, &p.maps.vs, 0, blk, bar);
      }
    }
  };
  // the first piece's query fragments (written by the pre-kernel) are fetched after the first
  // page copies are out: waiting for that kernel must not delay them
  uint8_t *qarea = kvq_dsmem + base + NS * Gm::STAGE + warp * Gm::QBYTES;
  int q_prefetched = -1;  // sequence whose query fragments are being copied
  auto prefetch_first = [&]() {
    if (sub >= run.n) return;
    SeqCursor c0 = run.first;
    const long long X0 = run.base + sub;
    while (X0 >= c0.P + c0.np && c0.b < a.B) seq_next<MODS>(a, c0);
    if (c0.b >= a.B) return;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the fragments of the pre-kernel
    fetch_frag<D>(p, qarea, c0.b, h, lane);
    q_prefetched = c0.b;
  };
  int cb = 0;        // warp 0: the batch of block ids its consumption has reached
  bool rest = false;  // warp 0: stages 2 .. NS - 1 issued
  if (warp == 0) {
    store_batch(0);
    store_batch(1);
    __syncwarp();
    // Only the first two stages now: at launch every CTA requests its first stages at once and
    // DRAM serves them interleaved, so a shorter first request lands sooner; the other slots
    // are filled once this warp has its first stage.
    for (int k = 0; k < 2 && k < n_stages; ++k) issue(k, k);
  }
  __syncthreads();  // barrier init and the first block ids, before any other warp can refill
  prefetch_first();
  // A slot is refilled by the last warp done with it (the shared counter's old value is 7 mod 8):
  // no warp waits for another to notice the slot is free.
  auto release = [&](int k, int slot) {
    __syncwarp();
    unsigned old = 0;
    if (lane == 0) old = atom_add_acq_rel_cta(&s_done[slot], 1u);
    old = __shfl_sync(FULL, old, 0);
    if ((old & 7u) == 7u && k + NS < n_stages) issue(k + NS, slot);
  };

  // ---- consumer side: warp w takes run page k * W + sub of every stage k
  const LaneOffsets<D> lo = lane_offsets<D, W>(warp, sub, hl, lane);
  SeqCursor cur = run.first;
  PieceState<D> st;
  st.reset();
  uint32_t qf[Gm::KSTEPS][2];
  float qs0 = 0.f, qs1 = 0.f;
  bool have_q = false, abort = false;
  float sm24 = 0.f;  // score scale of the piece: sm * log2 e * 2^24 (K operands) * 2^k (q shift)
  ScoreMods md{};
  if constexpr (MODS) {  // MMA column n is query token n / G, head h G + n % G of it (COMB: head n % 4)
    const int c0 = COMB ? 2 * (lane & 1) : 2 * (lane & 3), G = a.G;
    const float lg2e = 1.4426950408889634f;
    md.sl0 = p.alibi != nullptr && c0 < G * a.Q ? __ldg(p.alibi + h * G + c0 % G) * lg2e : 0.f;
    md.sl1 = p.alibi != nullptr && c0 + 1 < G * a.Q ? __ldg(p.alibi + h * G + (c0 + 1) % G) * lg2e : 0.f;
  }
  // per piece: the lane's columns' key ranges [lw, lim) and the first query token's limit limf
  // (pages below it, and at or above the last token's window start lwl, need no masks). Columns
  // past the block's query tokens repeat its last token (their rows are never read).
  int lim0 = 0, lim1 = 0, lw0 = 0, lw1 = 0, limf = 0, lwl = 0;
  auto columns = [&]() {
    const int nq = a.vseq != nullptr ? a.vseq[cur.b].w : 1;
    const int k0 = min((2 * (lane & 3)) / a.G, nq - 1), k1 = min((2 * (lane & 3) + 1) / a.G, nq - 1);
    md.qp0 = cur.L - nq + k0;
    md.qp1 = cur.L - nq + k1;
    lim0 = md.qp0 + 1;
    lim1 = md.qp1 + 1;
    lw0 = a.window > 0 ? max(0, md.qp0 + 1 - a.window) : 0;
    lw1 = a.window > 0 ? max(0, md.qp1 + 1 - a.window) : 0;
    limf = cur.L - nq + 1;
    lwl = a.window > 0 ? max(0, cur.L - a.window) : 0;
  };
  // the current piece in run coordinates: its pages are run pages < pe_x, run page x is page
  // x + off of sequence cur.b, and its tokens are [t0, t1)
  int pe_x = 0, off = 0, t0 = 0, t1 = 0;
  auto bounds = [&]() {
    off = static_cast<int>(run.base - cur.P) + cur.f;
    if (run.fixed) {
      pe_x = run.n;
      t0 = run.t0;
      t1 = run.t1;
    } else {
      pe_x = static_cast<int>(min(static_cast<long long>(run.n), cur.P + cur.np - run.base));
      t0 = max(cur.lo, static_cast<int>((max(run.base, cur.P) - cur.P + cur.f) * kPage));
      t1 = static_cast<int>(min((min(run.end, cur.P + cur.np) - cur.P + cur.f) * kPage, static_cast<long long>(cur.L)));
    }
  };
  bounds();
  columns();
  auto finish_piece = [&]() {
    const long long slot = run.fixed ? static_cast<long long>(blockIdx.x) : blockIdx.x + static_cast<long long>(cur.b);
    int4_finish<D, MTOK, COMB>(a, st, slot, sub, h, lane);
    if (!run.fixed && warp == 0 && lane == 0 && blockIdx.y == 0) {
      if (cur.P >= run.base) a.seg_first[cur.b] = static_cast<int>(blockIdx.x);
      if (cur.P + cur.np <= run.end) a.seg_last[cur.b] = static_cast<int>(blockIdx.x);
    }
    st.reset();
    have_q = false;
  };
  // wait for stage k (in `slot`, round rnd); on a timeout (a copy that never completes) raise
  // the flag, let the copies already issued land (bounded), and report failure
  auto wait_stage = [&](int k, int slot, int rnd) -> bool {
    const uint32_t fb = smem_u32(&s_full[slot]);
    if (__builtin_expect(__all_sync(FULL, mbar_try_wait(fb, rnd & 1)), 1)) return true;
    if (__all_sync(FULL, mbar_wait(fb, rnd & 1, p.wait_ns))) return true;
    if (lane == 0) atomicOr(&g_flags_decode_int4, ERR_TIMEOUT);
    for (int i = k; i < k + NS && i < n_stages; ++i)
      mbar_wait(smem_u32(&s_full[i % NS]), (i / NS) & 1, 100000000ull);
    return false;
  };

  int j = 0, sj = 0, rj = 0;  // stage j lives in slot sj = j % NS, round rj = j / NS
  while (j < n_stages) {
    const int x = j * W + sub;
    if (x >= run.n) break;
    if (x >= pe_x) {  // pieces this warp is done with (or has no page of)
      while (run.base + x >= cur.P + cur.np && cur.b < a.B) {
        finish_piece();
        seq_next<MODS>(a, cur);
      }
      if (cur.b >= a.B) break;  // cannot happen: the run lies inside the batch's pages
      bounds();
      columns();
    }
    if (!have_q) {
      float qmul;
      if (q_prefetched != cur.b) asm volatile("griddepcontrol.wait;" ::: "memory");
      load_frag<D>(p, qarea, cur.b, h, lane, qf, qs0, qs1, qmul, q_prefetched == cur.b);
      sm24 = p.sm_log2 * kTwo24 * qmul;
      if constexpr (COMB) {  // columns 4..7 repeat columns 0..3 (lane l + 16 holds column n + 4)
#pragma unroll
        for (int k = 0; k < Gm::KSTEPS; ++k) {
          qf[k][0] = __shfl_sync(FULL, qf[k][0], lane & 15);
          qf[k][1] = __shfl_sync(FULL, qf[k][1], lane & 15);
        }
        const float r0 = __shfl_xor_sync(FULL, qs0, 2), r1 = __shfl_xor_sync(FULL, qs1, 2);
        if ((lane & 3) >= 2) {
          qs0 = r0;
          qs1 = r1;
        }
      }
      q_prefetched = -1;
      if (pe_x < run.n && !run.fixed) {  // the run goes on into another sequence: fetch its query now
        SeqCursor nx = cur;
        seq_next<MODS>(a, nx);
        if (nx.b < a.B) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          fetch_frag<D>(p, qarea, nx.b, h, lane);
          q_prefetched = nx.b;
        }
      }
      have_q = true;
    }
    const int nb = (x + off) * kPage;  // position of the page's row 0 in its sequence
    const int sj1 = sj + 1 == NS ? 0 : sj + 1, rj1 = sj + 1 == NS ? rj + 1 : rj;
    const uint32_t so[2] = {base + sj * Gm::STAGE, base + sj1 * Gm::STAGE};
    // two full pages of the piece inside every column's key range (one query token: the piece)
    const int tpair = MTOK ? min(t1, limf) : t1;
    const bool pair = nb >= (MTOK ? max(t0, lwl) : t0) && nb + (W + 1) * kPage <= tpair && x + W < pe_x;
    if (warp == 0 && ((j * W) >> 5) >= cb) {  // entering a new batch of block ids: load the one two ahead
      cb = ((j * W) >> 5) + 1;
      store_batch(cb + 1);
    }
    if (__builtin_expect(pair, 1)) {
      if (!wait_stage(j, sj, rj) || !wait_stage(j + 1, sj1, rj1)) {
        abort = true;
        break;
      }
      if (warp == 0 && !rest) {  // the slots never used yet
        rest = true;
        for (int k = 2; k < NS && k < n_stages; ++k) issue(k, k);
      }
      int4_pages<D, W, 2, false, MODS, MTOK, COMB>(st, so, lo, qf, qs0, qs1, sm24, lane, nb, t0, t1, lim0, lim1, lw0,
                                             lw1, p, md);
      release(j, sj);
      release(j + 1, sj1);
      j += 2;
      sj = sj1 + 1 == NS ? 0 : sj1 + 1;
      rj = sj1 + 1 == NS ? rj1 + 1 : rj1;
    } else {
      if (!wait_stage(j, sj, rj)) {
        abort = true;
        break;
      }
      if (warp == 0 && !rest) {
        rest = true;
        for (int k = 2; k < NS && k < n_stages; ++k) issue(k, k);
      }
      int4_pages<D, W, 1, true, MODS, MTOK, COMB>(st, so, lo, qf, qs0, qs1, sm24, lane, nb, t0, t1, lim0, lim1, lw0,
                                            lw1, p, md);
      release(j, sj);
      j += 1;
      sj = sj1;
      rj = rj1;
    }
  }
  if (cur.b < a.B) finish_piece();
  if (!run.fixed && !abort) {
    while (cur.P + cur.np < run.end && cur.b < a.B - 1) {  // later pieces of the run without a page of this warp
      seq_next<MODS>(a, cur);
      if (cur.b >= a.B) break;
      finish_piece();
    }
  }
}

constexpr int kStagesInt4 = 4;

template <int D>
size_t int4_smem_bytes() {
  using Gm = Int4Geom<D>;
  return static_cast<size_t>(kStagesInt4) * Gm::STAGE + 8 * Gm::QBYTES + 1024;
}

bool take_flags_decode_int4(cudaStream_t stream, unsigned *host_word) {
  static const unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(host_word, g_flags_decode_int4, sizeof(unsigned), 0,
                                cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return false;
  return cudaMemcpyToSymbolAsync(g_flags_decode_int4, &zero, sizeof(unsigned), 0,
                                 cudaMemcpyHostToDevice, stream) == cudaSuccess;
}

template <int D, int W, int VAR>
static kvq_status launch_int4_w(const Int4Params &p, const SplitPlan &plan, cudaStream_t s) {
  const size_t smem = int4_smem_bytes<D>();
  static size_t attr_done[kMaxDevices] = {};
  if (ensure_dynamic_smem(decode_int4_kernel<D, kStagesInt4, W, VAR>, smem, attr_done) != cudaSuccess)
    return KVQ_ERR_CUDA;
  const dim3 grid(plan.seg_ctas, plan.head_groups);
  // query pre-rotation, then the split kernel as its programmatic dependent
  constexpr bool MTOK = VAR == 1 || VAR == 2;
  const long long warps = static_cast<long long>(p.s.B) * p.s.Hk;
  static size_t rot_done[kMaxDevices] = {};
  if (ensure_dynamic_smem(rotate_q_int4_kernel<D, MTOK>, 8 * Int4Geom<D>::QBYTES, rot_done) != cudaSuccess)
    return KVQ_ERR_CUDA;
  rotate_q_int4_kernel<D, MTOK><<<static_cast<unsigned>((warps + 7) / 8), 256, 8 * Int4Geom<D>::QBYTES, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  if (launch_dependent(decode_int4_kernel<D, kStagesInt4, W, VAR>, grid, dim3(256), s, p, smem) != cudaSuccess)
    return KVQ_ERR_CUDA;
  const long long rows = static_cast<long long>(p.s.B) * p.s.Hq;
  if (launch_dependent(merge_kernel<D>, dim3(static_cast<unsigned>((rows + 7) / 8)), dim3(256), s, p.s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return launch_status();
}

template <int D, int VAR>
static kvq_status launch_int4(const Int4Params &p, const SplitPlan &plan, cudaStream_t s) {
  switch (plan.warps_per_head) {
    case 1: return launch_int4_w<D, 1, VAR>(p, plan, s);
    case 2: return launch_int4_w<D, 2, VAR>(p, plan, s);
    case 4: return launch_int4_w<D, 4, VAR>(p, plan, s);
    case 8: return launch_int4_w<D, 8, VAR>(p, plan, s);
    default: return KVQ_ERR_UNSUPPORTED;
  }
}

}  // namespace kvq

using namespace kvq;


namespace kvq {

// Multi-token decode (unified_attention_int4 with max_seqlen_q > 1): the query tokens of every
// sequence are cut into blocks of up to QB = 8 / G tokens -- the MMA's 8 columns, G heads per
// token -- and each block is a virtual sequence whose keys end at its last token's position + 1.
// vseq[v] = {sequence b (its block-table row), that key end, the block's first q / out row, its
// tokens}; entries past the last block are empty (key end 0). One CTA, sequences 256 at a time.
__global__ void __launch_bounds__(256) build_vseq_kernel(const int32_t *qsl, int q_uniform, const int32_t *seq_lens,
                                                         int B, int QB, int max_blocks, int total_q, int4 *vseq,
                                                         int vmax) {
  __shared__ long long s_scan[8];
  long long running = 0;
  for (int base = 0; base < B; base += 256) {
    const int b = base + threadIdx.x;
    int qb = 0, r0 = 0, L = 0;
    if (b < B) {
      if (qsl != nullptr) {
        r0 = __ldg(qsl + b);
        const int r1 = __ldg(qsl + b + 1);
        qb = r1 - r0;
        if (r0 < 0 || qb < 0 || r1 > total_q) {  // query rows outside q: skipped, flagged
          atomicOr(&g_flags_decode_int4, ERR_SEQLEN);
          qb = 0;
        }
      } else {
        r0 = b * q_uniform;
        qb = q_uniform;
      }
      L = __ldg(seq_lens + b);
      if (L > max_blocks * kPage) {
        atomicOr(&g_flags_decode_int4, ERR_SEQLEN);
        L = max_blocks * kPage;
      }
      L = max(L, 0);
    }
    const long long nv = (qb + QB - 1) / QB;
    long long chunk;
    const long long off = block_scan_256(nv, s_scan, &chunk) + running - nv;
    for (int k = 0; k < nv; ++k) {
      const int i0 = k * QB, nq = min(QB, qb - i0);
      if (off + k < vmax) vseq[off + k] = make_int4(b, max(0, L - qb + i0 + nq), r0 + i0, nq);
    }
    running += chunk;
  }
  for (long long v = running + threadIdx.x; v < vmax; v += 256) vseq[v] = make_int4(0, 0, 0, 0);
}

// Geometry of a decode call: multi-token or not, tokens per block QB, (virtual) sequences.
struct CallGeom {
  bool mtok;
  int QB;
  long long nseq;
};
static bool call_geom(int B, int Hq, int Hk, const kvq_score_mods *mods, CallGeom *g) {
  g->mtok = mods != nullptr && (mods->q_len > 1 || mods->query_start_loc != nullptr);
  g->QB = 1;
  g->nseq = B;
  if (!g->mtok) return true;
  if (Hk < 1 || Hq % Hk != 0 || Hq / Hk > 8) return false;
  g->QB = 8 / (Hq / Hk);
  if (mods->query_start_loc != nullptr) {
    if (mods->total_q < 0) return false;
    g->nseq = static_cast<long long>(B) + (mods->total_q + g->QB - 1) / g->QB;  // sum of ceil(q_b / QB)
  } else {
    g->nseq = static_cast<long long>(B) * ((mods->q_len + g->QB - 1) / g->QB);
  }
  return g->nseq <= 0x7fffffffLL;
}
static size_t mods_workspace_bytes(int B, int Hq, int Hk, int D, int num_splits, const kvq_score_mods *mods,
                                   SplitPlan *plan, CallGeom *g) {
  if (!call_geom(B, Hq, Hk, mods, g)) return 0;
  if (!make_plan(static_cast<int>(g->nseq), Hk, num_splits, plan)) return 0;
  const size_t ws = workspace_bytes(static_cast<int>(g->nseq), g->QB * Hq, D, *plan);
  // multi-token calls: the virtual-sequence list, then the query fragments of every virtual sequence
  return ws + (g->mtok ? round256(static_cast<size_t>(g->nseq) * sizeof(int4)) : 0) +
         qfrag_bytes(static_cast<int>(g->nseq), Hk, D);
}

}  // namespace kvq

extern "C" size_t kvq_decode_int4_mods_workspace_bytes(int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                                       int32_t num_splits, const kvq_score_mods *mods) {
  if (B < 0 || Hq < 1 || Hk < 1 || Hq % Hk || (D != 64 && D != 128) || num_splits < 0) return 0;
  if (mods && (mods->q_len < 0 || (mods->query_start_loc && mods->total_q < 0))) return 0;
  SplitPlan plan;
  CallGeom g;
  return mods_workspace_bytes(B, Hq, Hk, D, num_splits, mods, &plan, &g);
}

extern "C" kvq_status kvq_decode_int4_mods(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                           const float *k_scale, const float *v_scale,
                                           const int32_t *block_table, int32_t max_blocks,
                                           const int32_t *seq_lens, const float *rht_signs,
                                           float softmax_scale, int32_t num_splits, void *workspace,
                                           size_t workspace_bytes, void *out, kvq_dtype out_dtype,
                                           int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                           int32_t block_size, int64_t num_blocks,
                                           const kvq_score_mods *mods, kvq_stream_t stream) {
  if (B < 0 || Hq < 1 || Hk < 1 || max_blocks < 0 || num_splits < 0 || num_blocks < 1)
    return KVQ_ERR_INVALID_ARG;
  if (mods && (mods->sliding_window < 0 || !(mods->softcap >= 0.f) || !(mods->softcap < INFINITY) ||
               (mods->sinks && !aligned(mods->sinks, 4)) ||
               (mods->alibi_slopes && !aligned(mods->alibi_slopes, 4)) || mods->q_len < 0 ||
               (mods->lse_out && !aligned(mods->lse_out, 4)) ||
               (mods->query_start_loc && (!aligned(mods->query_start_loc, 4) || mods->total_q < 0))))
    return KVQ_ERR_INVALID_ARG;
  if (Hq % Hk != 0) return KVQ_ERR_INVALID_ARG;
  if (out_dtype != KVQ_BF16 && out_dtype != KVQ_F16 && out_dtype != KVQ_F32) return KVQ_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (block_size != kPage) return KVQ_ERR_UNSUPPORTED;
  if (Hq / Hk > 8) return KVQ_ERR_UNSUPPORTED;
  if (!(softmax_scale > 0.f) || !(softmax_scale < INFINITY)) return KVQ_ERR_INVALID_ARG;
  SplitPlan plan;
  CallGeom cg;
  if (!call_geom(B, Hq, Hk, mods, &cg) || !make_plan(static_cast<int>(cg.nseq), Hk, num_splits, &plan))
    return KVQ_ERR_UNSUPPORTED;
  if (B == 0 || cg.nseq == 0) return KVQ_OK;
  const size_t need = mods_workspace_bytes(B, Hq, Hk, D, num_splits, mods, &plan, &cg);
  if (need == 0) return KVQ_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !k_scale || !v_scale || !block_table || !seq_lens || !out ||
      !workspace)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_scale, 16) ||
      !aligned(v_scale, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(out, 16) || !aligned(workspace, 16) || (rht_signs && !aligned(rht_signs, 16)))
    return KVQ_ERR_INVALID_ARG;
  if (max_blocks < 1) return KVQ_ERR_INVALID_ARG;
  if (workspace_bytes < need) return KVQ_ERR_WORKSPACE;

  Int4Params p;
  SplitArgs &sa = p.s;
  const int nseq = static_cast<int>(cg.nseq);
  sa.seq_lens = seq_lens;
  sa.max_blocks = max_blocks;
  sa.num_splits = num_splits;
  sa.B = nseq;
  sa.Hq = cg.QB * Hq;  // output rows per (virtual) sequence
  sa.Q = cg.QB;
  sa.Hk = Hk;
  sa.G = Hq / Hk;
  sa.heads_per_cta = plan.heads_per_cta;
  sa.warps_per_head = plan.warps_per_head;
  sa.seg_ctas = plan.seg_ctas;
  sa.slots = plan.slots;
  workspace_carve(workspace, nseq, cg.QB * Hq, D, plan, &sa.part_o, &sa.part_lse, &sa.seg_first, &sa.seg_last);
  int4 *vseq = cg.mtok ? reinterpret_cast<int4 *>(static_cast<uint8_t *>(workspace) +
                                                  kvq::workspace_bytes(nseq, cg.QB * Hq, D, plan))
                       : nullptr;
  p.qfrag = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(workspace) + kvq::workspace_bytes(nseq, cg.QB * Hq, D, plan) +
                                         (cg.mtok ? round256(static_cast<size_t>(nseq) * sizeof(int4)) : 0));
  sa.vseq = vseq;
  sa.signs = rht_signs;
  sa.out = out;
  sa.out_dtype = out_dtype;
  sa.window = mods ? mods->sliding_window : 0;
  sa.sinks = mods ? mods->sinks : nullptr;
  sa.lse_out = mods ? mods->lse_out : nullptr;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  if (!int4_tensor_maps(k_cache, v_cache, k_scale, v_scale, num_blocks, Hk, D, &p.maps)) return KVQ_ERR_CUDA;
  p.block_table = block_table;
  p.bt_rows = B;
  const double sm = rht_signs ? static_cast<double>(softmax_scale) / D : softmax_scale;
  p.sm_log2 = static_cast<float>(sm * 1.4426950408889634);
  p.num_blocks = num_blocks;
  const double cap2 = mods ? static_cast<double>(mods->softcap) * 1.4426950408889634 : 0.0;
  p.softcap2 = static_cast<float>(cap2);
  p.inv_softcap2 = cap2 > 0.0 ? static_cast<float>(1.0 / cap2) : 0.f;
  p.alibi = mods ? mods->alibi_slopes : nullptr;
  p.wait_ns = debug_wait_ns();
  p.withhold = debug_take_withhold();  // one call only
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cg.mtok) {  // the virtual sequences, in stream order before the split kernel
    build_vseq_kernel<<<1, 256, 0, s>>>(mods->query_start_loc, mods->query_start_loc ? 0 : mods->q_len, seq_lens, B,
                                        cg.QB, max_blocks, mods->total_q, vseq, nseq);
    if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  }
  // sinks act in the merge only; window, soft cap and ALiBi need the modifier kernel (which also
  // takes multi-token decode); multi-token decode alone has its own
  // a single-token call with G <= 4 heads per kv head fills the MMA's idle columns with a second page
  const bool scored = p.softcap2 > 0.f || p.alibi != nullptr || sa.window > 0, comb = Hq / Hk <= 4;
  const int var = scored ? (cg.mtok || !comb ? 1 : 4) : cg.mtok ? 2 : (comb ? 3 : 0);
  switch (var) {
    case 0: return D == 128 ? launch_int4<128, 0>(p, plan, s) : launch_int4<64, 0>(p, plan, s);
    case 1: return D == 128 ? launch_int4<128, 1>(p, plan, s) : launch_int4<64, 1>(p, plan, s);
    case 2: return D == 128 ? launch_int4<128, 2>(p, plan, s) : launch_int4<64, 2>(p, plan, s);
    case 4: return D == 128 ? launch_int4<128, 4>(p, plan, s) : launch_int4<64, 4>(p, plan, s);
    default: return D == 128 ? launch_int4<128, 3>(p, plan, s) : launch_int4<64, 3>(p, plan, s);
  }
}

extern "C" kvq_status kvq_decode_int4(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_table, int32_t max_blocks,
                                      const int32_t *seq_lens, const float *rht_signs,
                                      float softmax_scale, int32_t num_splits, void *workspace,
                                      size_t workspace_bytes, void *out, kvq_dtype out_dtype,
                                      int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                      int32_t block_size, int64_t num_blocks, kvq_stream_t stream) {
  return kvq_decode_int4_mods(q, k_cache, v_cache, k_scale, v_scale, block_table, max_blocks, seq_lens,
                              rht_signs, softmax_scale, num_splits, workspace, workspace_bytes, out,
                              out_dtype, B, Hq, Hk, D, block_size, num_blocks, nullptr, stream);
}

// ---------------------------------------------------------------------------------------------
// Allocation-free variant: the same decode with its scratch in a device array of this library.
// ---------------------------------------------------------------------------------------------
namespace kvq {

// Scratch of kvq_decode_int4_noalloc: one array per GPU that loads the library, kept until exit.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

// Device address of the array on the current device, looked up once per device. In host code
// g_noalloc_scratch names a host-side stand-in, never a device address.
static void *noalloc_scratch() {
  static std::mutex mu;
  static void *addr[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace kvq

extern "C" kvq_status kvq_decode_int4_noalloc(const void *q, const uint8_t *k_cache,
                                              const uint8_t *v_cache, const float *k_scale,
                                              const float *v_scale, const int32_t *block_table,
                                              int32_t max_blocks, const int32_t *seq_lens,
                                              const float *rht_signs, float softmax_scale,
                                              int32_t num_splits, void *out, kvq_dtype out_dtype,
                                              int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                              int32_t block_size, int64_t num_blocks,
                                              kvq_stream_t stream) {
  if (B == 0)  // empty work: a successful no-op, as for the workspace entry point
    return kvq_decode_int4(q, k_cache, v_cache, k_scale, v_scale, block_table, max_blocks, seq_lens,
                           rht_signs, softmax_scale, num_splits, nullptr, 0, out, out_dtype, B, Hq, Hk, D,
                           block_size, num_blocks, stream);
  void *scratch = kvq::noalloc_scratch();
  if (scratch == nullptr) return KVQ_ERR_CUDA;
  // The workspace entry point validates everything and rejects a scratch need above the array
  // size with KVQ_ERR_WORKSPACE before launching anything.
  return kvq_decode_int4(q, k_cache, v_cache, k_scale, v_scale, block_table, max_blocks, seq_lens,
                         rht_signs, softmax_scale, num_splits, scratch, KVQ_NOALLOC_SCRATCH_BYTES,
                         out, out_dtype, B, Hq, Hk, D, block_size, num_blocks, stream);
}
