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
// GB300 design. One warp owns one (kv head, run of pages) and streams it through a private
// NSTAGE-deep ring in shared memory filled by TMA: per page, one lane issues four tensor loads
// (this head's 16 K rows and 16 V rows, gathered from the page's [token][head] rows into a
// [token] tile with the 64B/32B swizzle that makes the fragment reads conflict-free, and the
// scale-word boxes) completing on the stage's mbarrier; waits are bounded and report a flag.
// No block-wide barrier is needed. Both contractions run on the tensor
// cores (mma.m16n8k16, fp16 operands, fp32 accumulation) on exact operands: a nibble pair
// masked into an fp16 pair with a zero exponent field IS the pair of fp16 subnormals n * 2^-24
// (low nibble) or n * 2^-20 (high nibble), so one LOP3 turns 2 nibbles into MMA operands
// without any offset; the power of two goes into the per-token scale, and the zero-point is
// applied as the split-dot correction of the pages (sum q n - zp sum q; sum P_v v - sum P_v zp):
//   * S^T[16 tokens x 8 heads] = K[16 x D] . Q^T  (q of a high-nibble dim pre-divided by 16);
//   * O^T[D x 8 heads] += V^T[D x 16 tokens] . P_v^T with P_v = p * scale_v in fp16; the
//     tokens (the K dimension) and the D rows are permuted so that a lane's V bytes become A
//     fragments with one PRMT per pair of m-tiles.
// The G query heads of a kv head share every K/V byte loaded (GQA), padded to the MMA's N = 8.

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
  float sm_log2;  // softmax scale (divided by D when rotating) times log2(e)
  int64_t num_blocks;
};

constexpr uint32_t kLo = 0x000F000Fu;  // low nibbles of bytes 0 and 2 -> fp16 subnormal pair n * 2^-24
constexpr uint32_t kHi = 0x00F000F0u;  // high nibbles -> fp16 subnormal pair n * 2^-20
constexpr float kTwo24 = 16777216.0f;
constexpr float kTwo20 = 1048576.0f;

template <int D>
struct Int4Geom {
  static constexpr int RB = D / 2;        // bytes per token row of one head
  static constexpr int KCH = D / 8;       // K bytes per lane per row
  static constexpr int VCH = D / 16;      // V bytes per lane per token
  static constexpr int TILE = 16 * RB;    // one head's page of one pool (TMA box)
  static constexpr int KVSTAGE = 2 * TILE < 1024 ? 1024 : 2 * TILE;  // K tile, V tile; 1024-aligned
  static constexpr int SCSTAGE = 2 * 16 * 4 * 4;                     // K, V scale boxes (<= 4 heads)
  static constexpr int WPR = D / 32;      // K words per lane per row
  static constexpr int KSTEPS = D / 16;
  static constexpr int MT = D / 16;       // m-tiles of the PV product
  static constexpr int QBYTES = 8 * D * 2 + 64;
};

// Per-warp TMA ring state, carried across the pieces of a CTA: pages issued / consumed so far
// (stage = count % NSTAGE, phase parity = (count / NSTAGE) & 1) and a sticky abort bit.
struct Ring {
  uint8_t *kv;     // NSTAGE x KVSTAGE bytes, 1024-aligned
  uint8_t *sc;     // NSTAGE x SCSTAGE bytes
  uint32_t bars;   // shared address of NSTAGE mbarriers
  uint32_t issued, consumed;
  bool abort;
};

template <int D, int NSTAGE>
__device__ __forceinline__ void int4_piece(const Int4Params &p, Ring &rg, uint8_t *qarea, int b, int h,
                                           int sub, int t0, int t1, long long slot) {
  using Gm = Int4Geom<D>;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.s.G, WPH = p.s.warps_per_head, Hk = p.s.Hk;

  // -------- this warp's pages: first, first + WPH, ... <= last page of the piece
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

  // -------- query: q_rot = bf16(H(q * d1)) for the G heads of kv head h, as fp16 B operands
  {
    constexpr int J = D / 32;
    const __nv_bfloat16 *qb = p.q + (static_cast<long long>(b) * p.s.Hq + static_cast<long long>(h) * G) * D;
    __half *qh = reinterpret_cast<__half *>(qarea);
    float *qsum = reinterpret_cast<float *>(qarea + 8 * D * 2);
    for (int n = G; n < 8; ++n) {  // padded MMA columns
#pragma unroll
      for (int j = 0; j < J; ++j) qh[n * D + lane + 32 * j] = __float2half_rn(0.f);
      if (lane == 0) qsum[n] = 0.f;
    }
    for (int n = 0; n < G; ++n) {
      float x[J];
#pragma unroll
      for (int j = 0; j < J; ++j) x[j] = __bfloat162float(qb[n * D + lane + 32 * j]);
      if (p.s.signs != nullptr) {
#pragma unroll
        for (int j = 0; j < J; ++j) x[j] *= __ldg(p.s.signs + lane + 32 * j);
#pragma unroll
        for (int mask = 1; mask < 32; mask <<= 1) {
#pragma unroll
          for (int j = 0; j < J; ++j) x[j] = butterfly_xor(x[j], lane, mask);
        }
        butterfly_local<J>(x);
#pragma unroll
        for (int j = 0; j < J; ++j) x[j] = bf16_round(x[j]);
      }
      // odd dims meet high nibbles, which enter the MMA 16x larger: pre-divide q by 16 (exact)
      float eff = 0.f;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        const __half v = __float2half_rn((e & 1) ? x[j] * 0.0625f : x[j]);
        qh[n * D + e] = v;
        eff += (e & 1) ? __half2float(v) * 16.f : __half2float(v);
      }
      eff = warp_sum(eff);
      if (lane == 0) qsum[n] = eff * (1.0f / kTwo24);  // sum of the q the products use, in MMA units
    }
  }
  __syncwarp();
  // B fragment of k-step ks = 2m + s: the dims a K word's nibbles occupy after the LOP3 split
  // (word j = WPR * t + m: low nibbles 8j + 2s, 8j + 4 + 2s; high nibbles one dim up)
  uint32_t qf[Gm::KSTEPS][2];
  {
    const __half *qh = reinterpret_cast<const __half *>(qarea) + g * D;
#pragma unroll
    for (int ks = 0; ks < Gm::KSTEPS; ++ks) {
      const int j = Gm::WPR * t + (ks >> 1), s2 = 2 * (ks & 1);
      qf[ks][0] = h2_as_u32(__halves2half2(qh[8 * j + s2], qh[8 * j + 4 + s2]));
      qf[ks][1] = h2_as_u32(__halves2half2(qh[8 * j + 1 + s2], qh[8 * j + 5 + s2]));
    }
  }
  const float *qsum = reinterpret_cast<const float *>(qarea + 8 * D * 2);
  const float qs0 = qsum[2 * t], qs1 = qsum[2 * t + 1];
  const float sm24 = p.sm_log2 * kTwo24;  // the K operands carry a factor 2^-24
  __syncwarp();

  // -------- TMA ring: per page, lane 0 loads this head's 16 K rows and 16 V rows (swizzled
  // boxes) plus the scale-word boxes, all completing on the stage's mbarrier.
  const int SH = p.maps.scale_heads;                 // heads per scale box
  const int hh = SH == 4 ? (h & 3) : h;              // this head's column in the scale box
  const int sc_h0 = SH == 4 ? (h & ~3) : 0;
  constexpr uint32_t kTx = 2 * Gm::TILE;             // + the two scale boxes (below)
  const uint32_t tx = kTx + 2 * 16 * SH * 4;
  auto issue = [&](int k) {
    const int kk = k & 31;
    if (k > 0 && kk == 0) {
      bids_cur = bids_next;
      bids_next = load_bids((k >> 5) + 1);
    }
    const int blk_raw = __shfl_sync(FULL, bids_cur, kk);
    if (k >= n_my) return;
    const bool ok = blk_raw >= 0 && blk_raw < p.num_blocks;
    const int blk = ok ? blk_raw : 0;  // out of range: flagged, page 0 read instead
    const int stg = static_cast<int>(rg.issued % NSTAGE);
    ++rg.issued;
    if (lane == 0) {
      if (!ok) atomicOr(&g_flags_decode_int4, ERR_BLOCK);
      const uint32_t bar = rg.bars + 8 * stg;
      const uint32_t kv = smem_u32(rg.kv + stg * Gm::KVSTAGE), sc = smem_u32(rg.sc + stg * Gm::SCSTAGE);
      fence_proxy_async();
      mbar_arrive_expect_tx(bar, tx);
      tma_load_4d(kv, &p.maps.k, 0, h, 0, blk, bar);
      tma_load_4d(kv + Gm::TILE, &p.maps.v, 0, h, 0, blk, bar);
      if (SH == 4) {
        tma_load_3d(sc, &p.maps.ks, sc_h0, 0, blk, bar);
        tma_load_3d(sc + Gm::SCSTAGE / 2, &p.maps.vs, sc_h0, 0, blk, bar);
      } else {
        tma_load_2d(sc, &p.maps.ks, 0, blk, bar);
        tma_load_2d(sc + Gm::SCSTAGE / 2, &p.maps.vs, 0, blk, bar);
      }
    }
  };
  // wait for the next page; on a timeout (a copy that never completes) raise the flag and abort
  auto wait_next = [&]() -> bool {
    const uint32_t stg = rg.consumed % NSTAGE, par = (rg.consumed / NSTAGE) & 1;
    const bool ok = mbar_wait(rg.bars + 8 * stg, par);
    if (!__all_sync(FULL, ok)) {
      if (lane == 0) atomicOr(&g_flags_decode_int4, ERR_TIMEOUT);
      rg.abort = true;
      return false;
    }
    return true;
  };

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, pz0 = 0.f, pz1 = 0.f;
  float acc[Gm::MT][4];
#pragma unroll
  for (int i = 0; i < Gm::MT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  if (rg.abort) return;
#pragma unroll
  for (int k = 0; k < NSTAGE - 1; ++k) issue(k);

  for (int k = 0; k < n_my; ++k) {
    issue(k + NSTAGE - 1);
    const uint32_t stg = rg.consumed % NSTAGE;
    if (!wait_next()) break;
    ++rg.consumed;
    const uint8_t *kt = rg.kv + stg * Gm::KVSTAGE, *vt = kt + Gm::TILE;
    const uint32_t *sk = reinterpret_cast<const uint32_t *>(rg.sc + stg * Gm::SCSTAGE);
    const uint32_t *sv = sk + Gm::SCSTAGE / 8;
    const int nb = (first + k * WPH) * kPage;  // position of the page's row 0
    const bool ok0 = nb + g >= t0 && nb + g < t1;
    const bool ok1 = nb + g + 8 >= t0 && nb + g + 8 < t1;

    // ---- scores: S = (sum_d q_d n_d - zp sum_d q_d) * scale_k * sm (base 2)
    const uint32_t kw0 = sk[g * SH + hh], kw1 = sk[(g + 8) * SH + hh];
    float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};  // two MMA chains
    {
      uint32_t wa[Gm::WPR], wb[Gm::WPR];
      if constexpr (Gm::WPR == 4) {
        const uint4 a4 = lds128(kt + swz<Gm::RB>(g, 16 * t)), b4 = lds128(kt + swz<Gm::RB>(g + 8, 16 * t));
        wa[0] = a4.x; wa[1] = a4.y; wa[2] = a4.z; wa[3] = a4.w;
        wb[0] = b4.x; wb[1] = b4.y; wb[2] = b4.z; wb[3] = b4.w;
      } else {
        const uint2 a2 = lds64(kt + swz<Gm::RB>(g, 8 * t)), b2 = lds64(kt + swz<Gm::RB>(g + 8, 8 * t));
        wa[0] = a2.x; wa[1] = a2.y;
        wb[0] = b2.x; wb[1] = b2.y;
      }
#pragma unroll
      for (int m = 0; m < Gm::WPR; ++m) {
        const uint32_t xa = wa[m] >> 8, xb = wb[m] >> 8;
        mma_f16_16816(c, wa[m] & kLo, wb[m] & kLo, wa[m] & kHi, wb[m] & kHi, qf[2 * m][0], qf[2 * m][1]);
        mma_f16_16816(c2, xa & kLo, xb & kLo, xa & kHi, xb & kHi, qf[2 * m + 1][0], qf[2 * m + 1][1]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] += c2[i];
    const uint32_t vw0 = sv[g * SH + hh], vw1 = sv[(g + 8) * SH + hh];
    const float ck0 = __uint_as_float(kw0 & ~0xFu) * sm24, ck1 = __uint_as_float(kw1 & ~0xFu) * sm24;
    const float zk0 = static_cast<float>(kw0 & 0xFu), zk1 = static_cast<float>(kw1 & 0xFu);
    const float s00 = ok0 ? (c[0] - zk0 * qs0) * ck0 : -INFINITY;  // token g,   head 2t
    const float s01 = ok0 ? (c[1] - zk0 * qs1) * ck0 : -INFINITY;  // token g,   head 2t+1
    const float s10 = ok1 ? (c[2] - zk1 * qs0) * ck1 : -INFINITY;  // token g+8, head 2t
    const float s11 = ok1 ? (c[3] - zk1 * qs1) * ck1 : -INFINITY;  // token g+8, head 2t+1

    // ---- online softmax (base 2)
    const float mx0 = fmaxf(m0, warp_max_g(fmaxf(s00, s10)));
    const float mx1 = fmaxf(m1, warp_max_g(fmaxf(s01, s11)));
    const float r0 = mx0 == -INFINITY ? 0.f : mx0, r1 = mx1 == -INFINITY ? 0.f : mx1;
    const float al0 = fast_exp2(m0 - r0), al1 = fast_exp2(m1 - r1);
    m0 = mx0;
    m1 = mx1;
    const float p00 = fast_exp2(s00 - r0), p10 = fast_exp2(s10 - r0);
    const float p01 = fast_exp2(s01 - r1), p11 = fast_exp2(s11 - r1);
    l0 = l0 * al0 + (p00 + p10);
    l1 = l1 * al1 + (p01 + p11);

    // ---- P_v = p * scale_v (fp16), and sum P_v * zp_v for the zero-point correction
    const float sv0 = __uint_as_float(vw0 & ~0xFu), sv1 = __uint_as_float(vw1 & ~0xFu);
    const float zv0 = static_cast<float>(vw0 & 0xFu), zv1 = static_cast<float>(vw1 & 0xFu);
    const __half2 X0 = __floats2half2_rn(ok0 ? p00 * sv0 : 0.f, ok1 ? p10 * sv1 : 0.f);
    const __half2 X1 = __floats2half2_rn(ok0 ? p01 * sv0 : 0.f, ok1 ? p11 * sv1 : 0.f);
    const float2 f0 = __half22float2(X0), f1 = __half22float2(X1);
    pz0 = pz0 * al0 + (f0.x * zv0 + f0.y * zv1);
    pz1 = pz1 * al1 + (f1.x * zv0 + f1.y * zv1);
    if (!__all_sync(FULL, al0 == 1.f && al1 == 1.f)) {  // a running max moved: rescale
#pragma unroll
      for (int i = 0; i < Gm::MT; ++i) {
        acc[i][0] *= al0;
        acc[i][1] *= al1;
        acc[i][2] *= al0;
        acc[i][3] *= al1;
      }
    }
    // B fragment of P_v^T: this lane needs head g at tokens 2t, 2t+1 (b01), 2t+8, 2t+9 (b23)
    const int src0 = 8 * t + (g >> 1), src1 = src0 + 4;
    const uint32_t x0 = h2_as_u32(X0), x1 = h2_as_u32(X1);
    const uint32_t y0 = __shfl_sync(FULL, x0, src0), y1 = __shfl_sync(FULL, x1, src0);
    const uint32_t z0 = __shfl_sync(FULL, x0, src1), z1 = __shfl_sync(FULL, x1, src1);
    const uint32_t ya = (g & 1) ? y1 : y0, za = (g & 1) ? z1 : z0;
    const uint32_t b01 = __byte_perm(ya, za, 0x5410), b23 = __byte_perm(ya, za, 0x7632);

    // ---- O^T += V^T . P_v^T
    {
      constexpr int VW = Gm::VCH / 4;  // V words per token per lane (2 or 1)
      uint32_t va[VW], vb[VW], vc[VW], vd[VW];
      if constexpr (VW == 2) {
        const uint2 A = lds64(vt + swz<Gm::RB>(2 * t, 8 * g)), B2 = lds64(vt + swz<Gm::RB>(2 * t + 1, 8 * g));
        const uint2 C = lds64(vt + swz<Gm::RB>(2 * t + 8, 8 * g)), E = lds64(vt + swz<Gm::RB>(2 * t + 9, 8 * g));
        va[0] = A.x; va[1] = A.y; vb[0] = B2.x; vb[1] = B2.y;
        vc[0] = C.x; vc[1] = C.y; vd[0] = E.x; vd[1] = E.y;
      } else {
        va[0] = lds32(vt + swz<Gm::RB>(2 * t, 4 * g));
        vb[0] = lds32(vt + swz<Gm::RB>(2 * t + 1, 4 * g));
        vc[0] = lds32(vt + swz<Gm::RB>(2 * t + 8, 4 * g));
        vd[0] = lds32(vt + swz<Gm::RB>(2 * t + 9, 4 * g));
      }
#pragma unroll
      for (int wi = 0; wi < VW; ++wi) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t sel = hf ? 0x7632u : 0x5410u;
          const uint32_t x = __byte_perm(va[wi], vb[wi], sel), y = __byte_perm(vc[wi], vd[wi], sel);
          const int mt = 4 * wi + 2 * hf;
          mma_f16_16816(acc[mt], x & kLo, x & kHi, y & kLo, y & kHi, b01, b23);
          const uint32_t x8 = x >> 8, y8 = y >> 8;
          mma_f16_16816(acc[mt + 1], x8 & kLo, x8 & kHi, y8 & kLo, y8 & kHi, b01, b23);
        }
      }
    }
    __syncwarp();
  }
  if (rg.abort) {  // let every copy already issued land before the warp moves on or exits
    while (rg.consumed < rg.issued) {
      mbar_wait(rg.bars + 8 * (rg.consumed % NSTAGE), (rg.consumed / NSTAGE) & 1);
      ++rg.consumed;
    }
  }
  __syncwarp();

  // -------- epilogue: undo the subnormal scaling, apply the zero-point term, normalise
  l0 = warp_sum_g(l0);
  l1 = warp_sum_g(l1);
  pz0 = warp_sum_g(pz0);
  pz1 = warp_sum_g(pz1);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  float o0[D / 8], o1[D / 8];
#pragma unroll
  for (int mt = 0; mt < Gm::MT; ++mt) {
    o0[2 * mt] = (acc[mt][0] * kTwo24 - pz0) * inv0;
    o1[2 * mt] = (acc[mt][1] * kTwo24 - pz1) * inv1;
    o0[2 * mt + 1] = (acc[mt][2] * kTwo20 - pz0) * inv0;
    o1[2 * mt + 1] = (acc[mt][3] * kTwo20 - pz1) * inv1;
  }
  const float lse0 = l0 > 0.f ? m0 + log2f(l0) : -INFINITY;
  const float lse1 = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
  store_partial<D>(p.s, slot, sub, h, lane, o0, o1, lse0, lse1);
}

template <int D, int NSTAGE>
__global__ void __launch_bounds__(256, 2) decode_int4_kernel(const __grid_constant__ Int4Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t s_bars[8][NSTAGE];
  // the swizzled TMA tiles need 1024-byte alignment: round the dynamic base up (1 KB of slack)
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  asm volatile("griddepcontrol.launch_dependents;");  // let the merge kernel's launch begin early
  using Gm = Int4Geom<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // dynamic smem: [8 warps][NSTAGE][KVSTAGE] K/V tiles, then [8][NSTAGE][SCSTAGE], then [8][QBYTES]
  Ring rg;
  rg.kv = smem + warp * NSTAGE * Gm::KVSTAGE;
  rg.sc = smem + 8 * NSTAGE * Gm::KVSTAGE + warp * NSTAGE * Gm::SCSTAGE;
  uint8_t *qarea = smem + 8 * NSTAGE * (Gm::KVSTAGE + Gm::SCSTAGE) + warp * Gm::QBYTES;
  rg.bars = smem_u32(&s_bars[warp][0]);
  rg.issued = rg.consumed = 0;
  rg.abort = false;
  if (lane == 0) {
    for (int i = 0; i < NSTAGE; ++i) mbar_init(rg.bars + 8 * i, 1);
    mbar_init_fence();
  }
  __syncwarp();
  const int hl = warp % p.s.heads_per_cta;
  const int sub = warp / p.s.heads_per_cta;
  const int h = blockIdx.y * p.s.heads_per_cta + hl;
  for_each_piece(p.s, &g_flags_decode_int4, [&](int b, int t0, int t1, long long slot) {
    int4_piece<D, NSTAGE>(p, rg, qarea, b, h, sub, t0, t1, slot);
  });
}

constexpr int kStagesInt4 = 4;

template <int D>
size_t int4_smem_bytes() {
  using Gm = Int4Geom<D>;
  return 8 * static_cast<size_t>(kStagesInt4 * (Gm::KVSTAGE + Gm::SCSTAGE) + Gm::QBYTES) + 1024;
}

bool take_flags_decode_int4(cudaStream_t stream, unsigned *host_word) {
  static const unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(host_word, g_flags_decode_int4, sizeof(unsigned), 0,
                                cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return false;
  return cudaMemcpyToSymbolAsync(g_flags_decode_int4, &zero, sizeof(unsigned), 0,
                                 cudaMemcpyHostToDevice, stream) == cudaSuccess;
}

template <int D>
static kvq_status launch_int4(const Int4Params &p, const SplitPlan &plan, cudaStream_t s) {
  const size_t smem = int4_smem_bytes<D>();
  static bool attr_set = false;  // per process; the attribute is per function, not per device
  if (!attr_set) {
    if (cudaFuncSetAttribute(decode_int4_kernel<D, kStagesInt4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return KVQ_ERR_CUDA;
    attr_set = true;
  }
  const dim3 grid(plan.seg_ctas, plan.head_groups);
  decode_int4_kernel<D, kStagesInt4><<<grid, 256, smem, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  const long long rows = static_cast<long long>(p.s.B) * p.s.Hq;
  if (launch_dependent(merge_kernel<D>, dim3(static_cast<unsigned>((rows + 7) / 8)), dim3(256), s, p.s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return launch_status();
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_decode_int4(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_table, int32_t max_blocks,
                                      const int32_t *seq_lens, const float *rht_signs,
                                      float softmax_scale, int32_t num_splits, void *workspace,
                                      size_t workspace_bytes, void *out, kvq_dtype out_dtype,
                                      int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                      int32_t block_size, int64_t num_blocks, kvq_stream_t stream) {
  if (B < 0 || Hq < 1 || Hk < 1 || max_blocks < 0 || num_splits < 0 || num_blocks < 1)
    return KVQ_ERR_INVALID_ARG;
  if (Hq % Hk != 0) return KVQ_ERR_INVALID_ARG;
  if (out_dtype != KVQ_BF16 && out_dtype != KVQ_F16 && out_dtype != KVQ_F32) return KVQ_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (block_size != kPage) return KVQ_ERR_UNSUPPORTED;
  if (Hq / Hk > 8) return KVQ_ERR_UNSUPPORTED;
  if (!(softmax_scale > 0.f) || !(softmax_scale < INFINITY)) return KVQ_ERR_INVALID_ARG;
  SplitPlan plan;
  if (!make_plan(B, Hk, num_splits, &plan)) return KVQ_ERR_UNSUPPORTED;
  if (B == 0) return KVQ_OK;
  if (!q || !k_cache || !v_cache || !k_scale || !v_scale || !block_table || !seq_lens || !out ||
      !workspace)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_scale, 16) ||
      !aligned(v_scale, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(out, 16) || !aligned(workspace, 16) || (rht_signs && !aligned(rht_signs, 16)))
    return KVQ_ERR_INVALID_ARG;
  if (max_blocks < 1) return KVQ_ERR_INVALID_ARG;
  if (workspace_bytes < kvq::workspace_bytes(B, Hq, D, plan)) return KVQ_ERR_WORKSPACE;

  Int4Params p;
  SplitArgs &sa = p.s;
  sa.seq_lens = seq_lens;
  sa.max_blocks = max_blocks;
  sa.num_splits = num_splits;
  sa.B = B;
  sa.Hq = Hq;
  sa.Hk = Hk;
  sa.G = Hq / Hk;
  sa.heads_per_cta = plan.heads_per_cta;
  sa.warps_per_head = plan.warps_per_head;
  sa.slots = plan.slots;
  workspace_carve(workspace, B, Hq, D, plan, &sa.part_o, &sa.part_lse, &sa.seg_first, &sa.seg_last);
  sa.signs = rht_signs;
  sa.out = out;
  sa.out_dtype = out_dtype;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  if (!int4_tensor_maps(k_cache, v_cache, k_scale, v_scale, num_blocks, Hk, D, &p.maps)) return KVQ_ERR_CUDA;
  p.block_table = block_table;
  const double sm = rht_signs ? static_cast<double>(softmax_scale) / D : softmax_scale;
  p.sm_log2 = static_cast<float>(sm * 1.4426950408889634);
  p.num_blocks = num_blocks;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return D == 128 ? launch_int4<128>(p, plan, s) : launch_int4<64>(p, plan, s);
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
  void *scratch = kvq::noalloc_scratch();
  if (scratch == nullptr) return KVQ_ERR_CUDA;
  // The workspace entry point validates everything and rejects a scratch need above the array
  // size with KVQ_ERR_WORKSPACE before launching anything.
  return kvq_decode_int4(q, k_cache, v_cache, k_scale, v_scale, block_table, max_blocks, seq_lens,
                         rht_signs, softmax_scale, num_splits, scratch, KVQ_NOALLOC_SCRATCH_BYTES,
                         out, out_dtype, B, Hq, Hk, D, block_size, num_blocks, stream);
}
