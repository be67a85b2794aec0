// kvq_decode_tq: split-KV paged decode attention over the TurboQuant combined K+V slot with
// FP8 (E4M3FN) keys and 4-bit or 3-bit uniform values.
//
// Follows triton_turboquant_decode.py, _tq_decode_stage1 with KEY_FP8 = 1: per token the key is
// the E4M3 decode of the slot's first D bytes and score = ATTN_SCALE * sum_d q_d k_d; values are
// idx * scale + zero with scale and zero fp16 words after the value bytes (4-bit: dimension d in
// byte d / 2, high nibble for odd d; 3-bit: LSB-first stream); an online softmax accumulates
// acc / l and lse per split, and the splits are merged by log-sum-exp (decode_common.cuh).
//
// GB300 design: one warp per kv head and run of pages (the split of decode_common.cuh), each warp
// with its own ring of page tiles brought by the tensor-memory accelerator: one 4-D box per
// (page, kv head) lands the 16 slots' used bytes as [token][row] rows (no per-lane copies), and an
// mbarrier per ring slot says when it has landed; mma.m16n8k16 for both contractions, separate
// merge kernel. Keys go to fp16 with the hardware E4M3x2 -> f16x2 conversion (exact); q (fp32,
// shifted by a power of two into the fp16 range, decode_common.cuh) is split into fp16 hi + lo
// parts, two MMAs per k-step, so the score keeps ~22 bits; the lanes build their q fragments from
// global memory directly. Value indices enter as exact fp16 subnormals (the index bits masked into
// a zero-exponent fp16: idx * 2^-24, or idx * 2^-20 for a high nibble) weighted by
// P_v = 2^(S - m) * scale in fp16 against a per-column softmax reference m that keeps P_v inside
// fp16 (decode_common.cuh); the power of two is undone in the epilogue and sum_n p_n * zero_n is
// added in fp32.

#include "decode_common.cuh"
#include "kvq_host.h"

namespace kvq {

__device__ unsigned g_flags_decode_tq = 0;

struct TqParams {
  SplitArgs s;
  CUtensorMap map;  // the slot pool as {slot_bytes, 16, Hk, num_blocks}, box {row bytes, 16, 1, 1}
  const float *q;
  const int32_t *block_table;
  float sc_log2;  // attn_scale * log2(e)
  int64_t num_blocks;
  unsigned long long wait_ns;  // limit of every bounded wait on a ring slot
  int32_t withhold;            // error-path tests only: warp 0 of CTA (0, 0) never issues its ring tile `withhold`
};

constexpr uint32_t kLoTq = 0x000F000Fu;  // low nibbles -> fp16 subnormals idx * 2^-24
constexpr uint32_t kHiTq = 0x00F000F0u;  // high nibbles -> idx * 2^-20

template <int D, int VBITS>
struct TqGeom {
  static constexpr int KCH = D / 4;             // K bytes per lane per row
  static constexpr int KCHUNKS = KCH / 16;      // 16-byte reads per row
  static constexpr int VDB = (D * VBITS + 7) / 8;
  static constexpr int RB = (D + VDB + 4 + 15) / 16 * 16;  // staged bytes of a slot: key, values, scale, zero
  static constexpr int TILE = kPage * RB;       // one (page, kv head) tile: 16 rows
  static constexpr int VCH = D / 16;            // 4-bit values: bytes per lane per token
  static constexpr int KSTEPS = D / 16;
  static constexpr int MT = D / 16;
};

__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two_bytes) {
  const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_bytes), __NV_E4M3);
  return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
}

// Per-warp ring state carried from piece to piece: tiles issued so far (ring slot and mbarrier
// phase of tile K are K % NSTAGE and (K / NSTAGE) & 1), and whether a wait ran out.
struct TqRing {
  const uint8_t *ring_p;  // the warp's first ring slot
  uint32_t ring;  // its shared-window address
  uint32_t bar;   // shared address of its first mbarrier (8 bytes each)
  uint32_t used;
  bool failed;
};

// PACKQ (G <= 4): the q hi parts of the G heads fill MMA columns 0..3 and the lo parts columns
// 4..7, so one MMA per k-step yields both halves of every score (added across lanes t, t ^ 2);
// otherwise hi and lo take one MMA each.
template <int D, int VBITS, int NSTAGE, bool PACKQ>
__device__ __forceinline__ void tq_piece(const TqParams &p, TqRing &rg, int b, int h, int sub, int t0, int t1,
                                         long long slot) {
  using Gm = TqGeom<D, VBITS>;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.s.G, WPH = p.s.warps_per_head;

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
      if (!ok) atomicOr(&g_flags_decode_tq, ERR_BLOCK);
      const uint32_t sl = (K0 + k) % NSTAGE;
      const uint32_t bar = rg.bar + 8 * sl;
      fence_proxy_async();  // earlier reads of the slot come before the copy that refills it
      mbar_arrive_expect_tx(bar, Gm::TILE);
      tma_load_4d(rg.ring + sl * Gm::TILE, &p.map, 0, 0, h, ok ? blk : 0, bar);
    }
  };
#pragma unroll
  for (int k = 0; k < NSTAGE - 1; ++k) issue(k);

  // -------- q -> fp16 hi / lo B fragments, straight from global memory: lane (g, t) holds column
  // g (head g, or PACKQ: head g % 4, its hi part for g < 4 and its lo part for g >= 4) at the
  // dims 32 t .. 32 t + 31 (D = 128) its K reads cover, k-step ks taking dims KCH t + 4 ks .. + 3
  float sc2;  // score scale of the piece: attn_scale * log2 e * 2^k
  uint32_t qhi[Gm::KSTEPS][2], qlo[PACKQ ? 1 : Gm::KSTEPS][2];
  {
    const int head = PACKQ ? (g & 3) : g;
    const bool live = head < G;
    const float4 *src = reinterpret_cast<const float4 *>(
        p.q + (static_cast<long long>(b) * p.s.Hq + static_cast<long long>(h) * G + (live ? head : 0)) * D + t * Gm::KCH);
    float qv[Gm::KCH];
#pragma unroll
    for (int j = 0; j < Gm::KCH / 4; ++j) {
      const float4 v = live ? __ldg(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      qv[4 * j] = v.x;
      qv[4 * j + 1] = v.y;
      qv[4 * j + 2] = v.z;
      qv[4 * j + 3] = v.w;
    }
    float qmax = 0.f;
#pragma unroll
    for (int j = 0; j < Gm::KCH; ++j) qmax = fmaxf(qmax, fabsf(qv[j]));
    const int qk = query_shift(warp_max(qmax), 0, &g_flags_decode_tq);
    const float qdiv = pow2i(-qk);
    sc2 = p.sc_log2 * pow2i(qk);
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

  // 3-bit: the lane's D/8 indices per token start at bit 3 * (D/8) * g of the value bytes
  constexpr int kV3Bytes = 3 * D / 64;  // bytes per lane (6 at D = 128, 3 at D = 64)
  const int v3_off = D + kV3Bytes * g;
  const int v3_al = v3_off & ~3;

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float pz0 = 0.f, pz1 = 0.f;
  float acc[Gm::MT][4];
#pragma unroll
  for (int i = 0; i < Gm::MT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  int k = 0;
  for (; k < n_my; ++k) {
    issue(k + NSTAGE - 1);
    {
      const uint32_t K = K0 + k;
      const uint32_t bar = rg.bar + 8 * (K % NSTAGE), par = (K / NSTAGE) & 1;
      if (!__all_sync(FULL, mbar_try_wait(bar, par)) && !__all_sync(FULL, mbar_wait(bar, par, p.wait_ns))) {
        if (lane == 0) atomicOr(&g_flags_decode_tq, ERR_TIMEOUT);
        rg.failed = true;
        break;
      }
    }
    const uint8_t *st = rg.ring_p + ((K0 + k) % NSTAGE) * Gm::TILE;
    const int nb = (first + k * WPH) * kPage;
    const bool ok0 = nb + g >= t0 && nb + g < t1;
    const bool ok1 = nb + g + 8 >= t0 && nb + g + 8 < t1;
    const uint8_t *row0 = st + g * Gm::RB, *row1 = st + (g + 8) * Gm::RB;

    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ch = 0; ch < Gm::KCHUNKS; ++ch) {
      const uint4 ra = lds128(row0 + t * Gm::KCH + 16 * ch);
      const uint4 rb = lds128(row1 + t * Gm::KCH + 16 * ch);
      const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ks = 4 * ch + i;
        const uint32_t a0 = e4m3x2_to_h2(wa[i] & 0xffffu), a2 = e4m3x2_to_h2(wa[i] >> 16);
        const uint32_t a1 = e4m3x2_to_h2(wb[i] & 0xffffu), a3 = e4m3x2_to_h2(wb[i] >> 16);
        if constexpr (PACKQ) {
          mma_f16_16816(c, a0, a1, a2, a3, qhi[ks][0], qhi[ks][1]);
        } else {
          mma_f16_16816(c, a0, a1, a2, a3, qhi[ks][0], qhi[ks][1]);
          mma_f16_16816(c, a0, a1, a2, a3, qlo[ks][0], qlo[ks][1]);
        }
      }
    }
    if constexpr (PACKQ) {
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] += __shfl_xor_sync(FULL, c[i], 2);  // hi (t < 2) + lo (t >= 2)
    }
    const uint32_t sz0 = lds32(row0 + D + Gm::VDB), sz1 = lds32(row1 + D + Gm::VDB);
    const float s00 = ok0 ? c[0] * sc2 : -INFINITY;
    const float s01 = ok0 ? c[1] * sc2 : -INFINITY;
    const float s10 = ok1 ? c[2] * sc2 : -INFINITY;
    const float s11 = ok1 ? c[3] * sc2 : -INFINITY;
    const float2 szf0 = __half22float2(u32_as_h2(sz0)), szf1 = __half22float2(u32_as_h2(sz1));  // (scale, zero)

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
      const float n0 = tr0 ? ref_new(b0, ms0, x0, &g_flags_decode_tq) : m0;
      const float n1 = tr1 ? ref_new(b1, ms1, x1, &g_flags_decode_tq) : m1;
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
      if (fmaxf(fmaxf(w00, w10), fmaxf(w01, w11)) > kWeightHi) atomicOr(&g_flags_decode_tq, ERR_RANGE);
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

    if constexpr (VBITS == 4) {
      constexpr int VW = Gm::VCH / 4;
      uint32_t va[VW], vb[VW], vc[VW], vd[VW];
      const uint8_t *vr = st + D + g * Gm::VCH;  // tokens 2t, 2t + 1, 2t + 8, 2t + 9: the lane's dims 16 g ..
      if constexpr (VW == 2) {
        const uint2 A = lds64(vr + (2 * t) * Gm::RB), B2 = lds64(vr + (2 * t + 1) * Gm::RB);
        const uint2 C = lds64(vr + (2 * t + 8) * Gm::RB), E = lds64(vr + (2 * t + 9) * Gm::RB);
        va[0] = A.x; va[1] = A.y; vb[0] = B2.x; vb[1] = B2.y;
        vc[0] = C.x; vc[1] = C.y; vd[0] = E.x; vd[1] = E.y;
      } else {
        va[0] = lds32(vr + (2 * t) * Gm::RB);
        vb[0] = lds32(vr + (2 * t + 1) * Gm::RB);
        vc[0] = lds32(vr + (2 * t + 8) * Gm::RB);
        vd[0] = lds32(vr + (2 * t + 9) * Gm::RB);
      }
#pragma unroll
      for (int wi = 0; wi < VW; ++wi) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t sel = hf ? 0x7632u : 0x5410u;
          const uint32_t x = __byte_perm(va[wi], vb[wi], sel), y = __byte_perm(vc[wi], vd[wi], sel);
          const int mt = 4 * wi + 2 * hf;
          mma_f16_16816(acc[mt], x & kLoTq, x & kHiTq, y & kLoTq, y & kHiTq, b01, b23);
          const uint32_t x8 = x >> 8, y8 = y >> 8;
          mma_f16_16816(acc[mt + 1], x8 & kLoTq, x8 & kHiTq, y8 & kLoTq, y8 & kHiTq, b01, b23);
        }
      }
    } else {
      // 3-bit: the lane's D/8 indices per token, LSB first, starting (v3_off - v3_al) bytes in
      const int sh = 8 * (v3_off - v3_al);
      unsigned long long w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // tokens 2t, 2t + 1, 2t + 8, 2t + 9
        const uint8_t *r = st + (2 * t + (i & 1) + 8 * (i >> 1)) * Gm::RB + v3_al;
        w[i] = ((static_cast<unsigned long long>(lds32(r + 4)) << 32) | lds32(r)) >> sh;
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
    const float s0 = VBITS == 4 ? 16777216.f : v3_scale(mt, 0), s1 = VBITS == 4 ? 1048576.f : v3_scale(mt, 1);
    o0[2 * mt] = (acc[mt][0] * s0 + pz0) * inv0;
    o1[2 * mt] = (acc[mt][1] * s0 + pz1) * inv1;
    o0[2 * mt + 1] = (acc[mt][2] * s1 + pz0) * inv0;
    o1[2 * mt + 1] = (acc[mt][3] * s1 + pz1) * inv1;
  }
  const float lse0 = l0 > 0.f ? m0 + log2f(l0) : -INFINITY;
  const float lse1 = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
  store_partial<D>(p.s, slot, sub, h, lane, o0, o1, lse0, lse1);
}

extern __shared__ __align__(128) uint8_t kvq_tq_dsmem[];

template <int D, int VBITS, int NSTAGE, bool PACKQ>
__global__ void __launch_bounds__(256, 2) decode_tq_kernel(const __grid_constant__ TqParams p) {
  using Gm = TqGeom<D, VBITS>;
  __shared__ __align__(8) uint64_t s_bar[8][NSTAGE];
  asm volatile("griddepcontrol.launch_dependents;");  // let the merge kernel's launch begin early
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // ring slots start at the first 128-byte aligned offset of the dynamic buffer
  const uint32_t dbase = smem_u32(kvq_tq_dsmem);
  const uint32_t off = ((128u - (dbase & 127u)) & 127u) + warp * NSTAGE * Gm::TILE;
  TqRing rg;
  rg.ring_p = kvq_tq_dsmem + off;
  rg.ring = dbase + off;
  rg.bar = smem_u32(&s_bar[warp][0]);
  rg.used = 0;
  rg.failed = false;
  if (lane == 0) {
    for (int i = 0; i < NSTAGE; ++i) mbar_init(rg.bar + 8 * i, 1);
    mbar_init_fence();
  }
  __syncwarp();
  const int hl = warp % p.s.heads_per_cta;
  const int sub = warp / p.s.heads_per_cta;
  const int h = blockIdx.y * p.s.heads_per_cta + hl;
  for_each_piece(p.s, &g_flags_decode_tq, [&](int b, int t0, int t1, long long slot) {
    if (!rg.failed) tq_piece<D, VBITS, NSTAGE, PACKQ>(p, rg, b, h, sub, t0, t1, slot);
  });
}

constexpr int kStagesTq = 4;

template <int D, int VBITS>
constexpr size_t tq_smem_bytes() {
  return 8 * static_cast<size_t>(kStagesTq) * TqGeom<D, VBITS>::TILE + 128;
}

bool take_flags_decode_tq(cudaStream_t stream, unsigned *host_word) {
  static const unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(host_word, g_flags_decode_tq, sizeof(unsigned), 0,
                                cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return false;
  return cudaMemcpyToSymbolAsync(g_flags_decode_tq, &zero, sizeof(unsigned), 0,
                                 cudaMemcpyHostToDevice, stream) == cudaSuccess;
}

template <int D, int VBITS, bool PACKQ>
static kvq_status launch_tq(TqParams &p, const SplitPlan &plan, const uint8_t *cache, int slot_bytes, int Hk,
                            cudaStream_t s) {
  using Gm = TqGeom<D, VBITS>;
  if (!tq_tensor_map(cache, p.num_blocks, Hk, slot_bytes, Gm::RB, &p.map)) return KVQ_ERR_CUDA;
  const size_t smem = tq_smem_bytes<D, VBITS>();
  static size_t attr_done[kMaxDevices] = {};
  if (ensure_dynamic_smem(decode_tq_kernel<D, VBITS, kStagesTq, PACKQ>, smem, attr_done) != cudaSuccess)
    return KVQ_ERR_CUDA;
  const dim3 grid(plan.seg_ctas, plan.head_groups);
  decode_tq_kernel<D, VBITS, kStagesTq, PACKQ><<<grid, 256, smem, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  const long long rows = static_cast<long long>(p.s.B) * p.s.Hq;
  if (launch_dependent(merge_kernel<D>, dim3(static_cast<unsigned>((rows + 7) / 8)), dim3(256), s, p.s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return launch_status();
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_decode_tq_lse(const float *q, const uint8_t *kv_cache, int32_t slot_bytes,
                                        int32_t value_bits, const int32_t *block_table,
                                        int32_t max_blocks, const int32_t *seq_lens, float attn_scale,
                                        int32_t num_splits, void *workspace, size_t workspace_bytes,
                                        float *out, float *lse_out, int32_t B, int32_t Hq, int32_t Hk,
                                        int32_t D, int32_t block_size, int64_t num_blocks,
                                        kvq_stream_t stream) {
  if (B < 0 || Hq < 1 || Hk < 1 || max_blocks < 0 || num_splits < 0 || num_blocks < 1)
    return KVQ_ERR_INVALID_ARG;
  if (Hq % Hk != 0) return KVQ_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (value_bits != 3 && value_bits != 4) return KVQ_ERR_UNSUPPORTED;
  if (block_size != kPage || Hq / Hk > 8) return KVQ_ERR_UNSUPPORTED;
  const int vdb = (D * value_bits + 7) / 8;
  if (slot_bytes % 16 != 0 || slot_bytes < D + vdb + 4) return KVQ_ERR_INVALID_ARG;
  if (!(attn_scale > 0.f) || !(attn_scale < INFINITY)) return KVQ_ERR_INVALID_ARG;
  SplitPlan plan;
  if (!make_plan(B, Hk, num_splits, &plan)) return KVQ_ERR_UNSUPPORTED;
  if (B == 0) return KVQ_OK;
  if (!q || !kv_cache || !block_table || !seq_lens || !out || !workspace) return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4) || !aligned(out, 16) || !aligned(workspace, 16) || !aligned(lse_out, 4))
    return KVQ_ERR_INVALID_ARG;
  if (max_blocks < 1) return KVQ_ERR_INVALID_ARG;
  if (workspace_bytes < kvq::workspace_bytes(B, Hq, D, plan)) return KVQ_ERR_WORKSPACE;

  TqParams p;
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
  workspace_carve(workspace, B, Hq, D, plan, &sa.part_o, &sa.part_lse, &sa.seg_first, &sa.seg_last);
  sa.signs = nullptr;
  sa.window = 0;
  sa.sinks = nullptr;
  sa.vseq = nullptr;
  sa.lse_out = lse_out;
  sa.out = out;
  sa.out_dtype = KVQ_F32;
  p.q = q;
  p.block_table = block_table;
  p.wait_ns = debug_wait_ns();
  p.withhold = debug_take_withhold();  // one call only
  p.sc_log2 = static_cast<float>(static_cast<double>(attn_scale) * 1.4426950408889634);
  p.num_blocks = num_blocks;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // packed q columns whenever G <= 4 (4-bit values on the 64 x 4096 workload: 94.1 vs 97.4 us per
  // call, measured on GB300)
  const bool packq = sa.G <= 4;
  if (D == 128) {
    if (value_bits == 4) return packq ? launch_tq<128, 4, true>(p, plan, kv_cache, slot_bytes, Hk, s) : launch_tq<128, 4, false>(p, plan, kv_cache, slot_bytes, Hk, s);
    return packq ? launch_tq<128, 3, true>(p, plan, kv_cache, slot_bytes, Hk, s) : launch_tq<128, 3, false>(p, plan, kv_cache, slot_bytes, Hk, s);
  }
  if (value_bits == 4) return packq ? launch_tq<64, 4, true>(p, plan, kv_cache, slot_bytes, Hk, s) : launch_tq<64, 4, false>(p, plan, kv_cache, slot_bytes, Hk, s);
  return packq ? launch_tq<64, 3, true>(p, plan, kv_cache, slot_bytes, Hk, s) : launch_tq<64, 3, false>(p, plan, kv_cache, slot_bytes, Hk, s);
}

extern "C" kvq_status kvq_decode_tq(const float *q, const uint8_t *kv_cache, int32_t slot_bytes,
                                    int32_t value_bits, const int32_t *block_table,
                                    int32_t max_blocks, const int32_t *seq_lens, float attn_scale,
                                    int32_t num_splits, void *workspace, size_t workspace_bytes,
                                    float *out, int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                    int32_t block_size, int64_t num_blocks, kvq_stream_t stream) {
  return kvq_decode_tq_lse(q, kv_cache, slot_bytes, value_bits, block_table, max_blocks, seq_lens, attn_scale,
                           num_splits, workspace, workspace_bytes, out, nullptr, B, Hq, Hk, D, block_size,
                           num_blocks, stream);
}
