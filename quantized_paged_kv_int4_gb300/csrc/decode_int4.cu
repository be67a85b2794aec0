// kvq_decode_int4: split-KV paged decode attention over the INT4 per-(token, head) cache.
//
// Follows int4_per_token_head.py, unified_attention_int4 and _attn_packed in its decode (3D,
// segment) mode: q is rotated like the cache (bf16(H(q * d1))), the softmax scale is divided by
// D, every page of the block table is walked, nibbles are used as plain integers with the
// zero-point applied through the split-dot correction
//     S = (sum_d q_d n_d - zp * sum_d q_d) * scale_k * sm,
// values enter the P.V product as P_v = p * scale_v with the correction - sum(P_v * zp_v), and
// the per-split results are merged by log-sum-exp and rotated back (decode_common.cuh).
//
// GB300 design. One warp owns one (kv head, run of pages) and streams it through a private
// NSTAGE-deep cp.async ring in shared memory: each lane copies exactly the bytes its MMA
// fragments need (16 B of each of two K rows, 8 B of four V rows, one scale word), so the ring
// needs no layout transform and no block-wide barrier. Both contractions run on the tensor
// cores with exact operands:
//   * S^T[16 tokens x 8 heads] = K[16 x D] . Q^T  (mma.m16n8k16, fp16): nibble n enters as the
//     fp16 value 1024 + n (low nibble) or 1024 + 16 n (high nibble, with the matching q
//     element pre-divided by 16), built with one LOP3 per pair; the 1024 offset is folded
//     into a per-head bias;
//   * O^T[D x 8 heads] += V^T[D x 16 tokens] . P_v^T with P_v in fp16 and the same nibble
//     trick; the K dimension (tokens) and the D rows are permuted so that a lane's V bytes
//     become A fragments with one PRMT.
// The G query heads of a kv head share every K/V byte loaded (GQA), padded to the MMA's N = 8.

#include "decode_common.cuh"
#include "kvq_host.h"

namespace kvq {

__device__ unsigned g_flags_decode_int4 = 0;

struct Int4Params {
  SplitArgs s;
  const __nv_bfloat16 *q;
  const uint8_t *k_cache, *v_cache;
  const uint32_t *k_scale, *v_scale;
  const int32_t *block_table;
  const float *signs;
  float sm_log2;  // softmax scale (divided by D when rotating) times log2(e)
  int64_t num_blocks;
};

constexpr uint32_t kMagic = 0x64006400u;  // fp16 pair (1024, 1024)

template <int D>
struct Int4Geom {
  static constexpr int KCH = D / 8;    // K bytes per lane per row
  static constexpr int VCH = D / 16;   // V bytes per lane per token
  static constexpr int KB = 64 * KCH;  // K bytes per stage (2 rows x 32 lanes)
  static constexpr int VB = 128 * VCH; // V bytes per stage (4 tokens x 32 lanes)
  static constexpr int STAGE = KB + VB + 128;
  static constexpr int WPR = D / 32;   // K words per lane per row
  static constexpr int KSTEPS = D / 16;
  static constexpr int MT = D / 16;    // m-tiles of the PV product
  static constexpr int QBYTES = 8 * D * 2 + 64;
};

template <int D, int NSTAGE>
__device__ __forceinline__ void int4_piece(const Int4Params &p, uint8_t *ring, uint8_t *qarea,
                                           int b, int h, int sub, int t0, int t1, long long slot) {
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

  // -------- query: q_rot = bf16(H(q * d1)) for the G heads of kv head h; fp16 B operands
  {
    constexpr int J = D / 32;
    const __nv_bfloat16 *qb = p.q + (static_cast<long long>(b) * p.s.Hq + static_cast<long long>(h) * G) * D;
    __half *qh = reinterpret_cast<__half *>(qarea);
    float *qsum = reinterpret_cast<float *>(qarea + 8 * D * 2);
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      float x[J];
#pragma unroll
      for (int j = 0; j < J; ++j) x[j] = n < G ? __bfloat162float(qb[n * D + lane + 32 * j]) : 0.f;
      if (p.signs != nullptr && n < G) {
#pragma unroll
        for (int j = 0; j < J; ++j) x[j] *= __ldg(p.signs + lane + 32 * j);
#pragma unroll
        for (int mask = 1; mask < 32; mask <<= 1) {
#pragma unroll
          for (int j = 0; j < J; ++j) x[j] = butterfly_xor(x[j], lane, mask);
        }
        butterfly_local<J>(x);
#pragma unroll
        for (int j = 0; j < J; ++j) x[j] = bf16_round(x[j]);
      }
      float raw = 0.f, eff = 0.f;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        const __half v = __float2half_rn((e & 1) ? x[j] * 0.0625f : x[j]);
        qh[n * D + e] = v;
        const float f = __half2float(v);
        raw += f;
        eff += (e & 1) ? f * 16.f : f;
      }
      raw = warp_sum(raw);
      eff = warp_sum(eff);
      if (lane == 0) {
        qsum[n] = eff;             // sum of the q values the products use (zero-point term)
        qsum[8 + n] = 1024.f * raw;  // the fp16 offset of the nibble encoding
      }
    }
  }
  __syncwarp();
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
  const float bias0 = qsum[8 + 2 * t], bias1 = qsum[8 + 2 * t + 1];
  __syncwarp();

  // -------- cp.async ring
  const uint32_t ring_s = smem_u32(ring);
  const long long row_stride = static_cast<long long>(Hk) * (D / 2);  // bytes between token rows
  auto issue = [&](int k) {
    const int kk = k & 31;
    if (k > 0 && kk == 0) {
      bids_cur = bids_next;
      bids_next = load_bids((k >> 5) + 1);
    }
    const int blk = __shfl_sync(FULL, bids_cur, kk);
    const bool in = k < n_my;
    const bool ok = in && blk >= 0 && blk < p.num_blocks;
    if (in && !ok && lane == 0) atomicOr(&g_flags_decode_int4, ERR_BLOCK);
    const uint32_t st = ring_s + (k % NSTAGE) * Gm::STAGE;
    const long long row0 = static_cast<long long>(ok ? blk : 0) * kPage * Hk + h;  // token 0 row
    const uint8_t *kb = p.k_cache + row0 * (D / 2);
    cp_async<Gm::KCH>(st + lane * Gm::KCH, kb + g * row_stride + t * Gm::KCH, ok);
    cp_async<Gm::KCH>(st + (32 + lane) * Gm::KCH, kb + (g + 8) * row_stride + t * Gm::KCH, ok);
    const uint8_t *vb = p.v_cache + row0 * (D / 2);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tok = 2 * t + (i & 1) + 8 * (i >> 1);
      cp_async<Gm::VCH>(st + Gm::KB + (i * 32 + lane) * Gm::VCH, vb + tok * row_stride + g * Gm::VCH, ok);
    }
    const uint32_t *sp = (lane < 16 ? p.k_scale : p.v_scale) + row0 + static_cast<long long>(lane & 15) * Hk;
    cp_async<4>(st + Gm::KB + Gm::VB + lane * 4, sp, ok);
    cp_async_commit();
  };

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float pz0 = 0.f, pz1 = 0.f, ps0 = 0.f, ps1 = 0.f;
  float acc[Gm::MT][4];
#pragma unroll
  for (int i = 0; i < Gm::MT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

#pragma unroll
  for (int k = 0; k < NSTAGE - 1; ++k) issue(k);

  for (int k = 0; k < n_my; ++k) {
    issue(k + NSTAGE - 1);
    cp_async_wait<NSTAGE - 1>();
    __syncwarp();
    const uint32_t st = ring_s + (k % NSTAGE) * Gm::STAGE;
    const int nb = (first + k * WPH) * kPage;  // position of the page's row 0
    const bool ok0 = nb + g >= t0 && nb + g < t1;
    const bool ok1 = nb + g + 8 >= t0 && nb + g + 8 < t1;

    // ---- scores
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    {
      uint32_t wa[Gm::WPR], wb[Gm::WPR];
      if constexpr (Gm::WPR == 4) {
        const uint4 a4 = lds128(st + lane * 16), b4 = lds128(st + (32 + lane) * 16);
        wa[0] = a4.x; wa[1] = a4.y; wa[2] = a4.z; wa[3] = a4.w;
        wb[0] = b4.x; wb[1] = b4.y; wb[2] = b4.z; wb[3] = b4.w;
      } else {
        const uint2 a2 = lds64(st + lane * 8), b2 = lds64(st + (32 + lane) * 8);
        wa[0] = a2.x; wa[1] = a2.y;
        wb[0] = b2.x; wb[1] = b2.y;
      }
#pragma unroll
      for (int m = 0; m < Gm::WPR; ++m) {
        const uint32_t xa = wa[m] >> 8, xb = wb[m] >> 8;
        mma_f16_16816(c, and_or(wa[m], 0x000F000Fu, kMagic), and_or(wb[m], 0x000F000Fu, kMagic),
                      and_or(wa[m], 0x00F000F0u, kMagic), and_or(wb[m], 0x00F000F0u, kMagic),
                      qf[2 * m][0], qf[2 * m][1]);
        mma_f16_16816(c, and_or(xa, 0x000F000Fu, kMagic), and_or(xb, 0x000F000Fu, kMagic),
                      and_or(xa, 0x00F000F0u, kMagic), and_or(xb, 0x00F000F0u, kMagic),
                      qf[2 * m + 1][0], qf[2 * m + 1][1]);
      }
    }
    const uint32_t sb = st + Gm::KB + Gm::VB;
    const uint32_t kw0 = lds32(sb + g * 4), kw1 = lds32(sb + (g + 8) * 4);
    const uint32_t vw0 = lds32(sb + (16 + g) * 4), vw1 = lds32(sb + (24 + g) * 4);
    const float ck0 = __uint_as_float(kw0 & ~0xFu) * p.sm_log2;
    const float ck1 = __uint_as_float(kw1 & ~0xFu) * p.sm_log2;
    const float zk0 = static_cast<float>(kw0 & 0xFu), zk1 = static_cast<float>(kw1 & 0xFu);
    float s00 = ok0 ? (c[0] - bias0 - zk0 * qs0) * ck0 : -INFINITY;  // token g,   head 2t
    float s01 = ok0 ? (c[1] - bias1 - zk0 * qs1) * ck0 : -INFINITY;  // token g,   head 2t+1
    float s10 = ok1 ? (c[2] - bias0 - zk1 * qs0) * ck1 : -INFINITY;  // token g+8, head 2t
    float s11 = ok1 ? (c[3] - bias1 - zk1 * qs1) * ck1 : -INFINITY;  // token g+8, head 2t+1

    // ---- online softmax (base 2)
    const float mx0 = fmaxf(m0, warp_max_g(fmaxf(s00, s10)));
    const float mx1 = fmaxf(m1, warp_max_g(fmaxf(s01, s11)));
    const float r0 = mx0 == -INFINITY ? 0.f : mx0, r1 = mx1 == -INFINITY ? 0.f : mx1;
    const float al0 = exp2f(m0 - r0), al1 = exp2f(m1 - r1);
    m0 = mx0;
    m1 = mx1;
    const float p00 = exp2f(s00 - r0), p10 = exp2f(s10 - r0);
    const float p01 = exp2f(s01 - r1), p11 = exp2f(s11 - r1);
    l0 = l0 * al0 + (p00 + p10);
    l1 = l1 * al1 + (p01 + p11);

    // ---- P_v = p * scale_v (fp16), its sums for the offset and zero-point corrections
    const float sv0 = __uint_as_float(vw0 & ~0xFu), sv1 = __uint_as_float(vw1 & ~0xFu);
    const float zv0 = static_cast<float>(vw0 & 0xFu), zv1 = static_cast<float>(vw1 & 0xFu);
    const __half2 X0 = __floats2half2_rn(ok0 ? p00 * sv0 : 0.f, ok1 ? p10 * sv1 : 0.f);
    const __half2 X1 = __floats2half2_rn(ok0 ? p01 * sv0 : 0.f, ok1 ? p11 * sv1 : 0.f);
    const float2 f0 = __half22float2(X0), f1 = __half22float2(X1);
    ps0 = ps0 * al0 + (f0.x + f0.y);
    ps1 = ps1 * al1 + (f1.x + f1.y);
    pz0 = pz0 * al0 + (f0.x * zv0 + f0.y * zv1);
    pz1 = pz1 * al1 + (f1.x * zv0 + f1.y * zv1);
#pragma unroll
    for (int i = 0; i < Gm::MT; ++i) {
      acc[i][0] *= al0;
      acc[i][1] *= al1;
      acc[i][2] *= al0;
      acc[i][3] *= al1;
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
        const uint2 A = lds64(st + Gm::KB + lane * 8), B2 = lds64(st + Gm::KB + (32 + lane) * 8);
        const uint2 C = lds64(st + Gm::KB + (64 + lane) * 8), E = lds64(st + Gm::KB + (96 + lane) * 8);
        va[0] = A.x; va[1] = A.y; vb[0] = B2.x; vb[1] = B2.y;
        vc[0] = C.x; vc[1] = C.y; vd[0] = E.x; vd[1] = E.y;
      } else {
        va[0] = lds32(st + Gm::KB + lane * 4);
        vb[0] = lds32(st + Gm::KB + (32 + lane) * 4);
        vc[0] = lds32(st + Gm::KB + (64 + lane) * 4);
        vd[0] = lds32(st + Gm::KB + (96 + lane) * 4);
      }
#pragma unroll
      for (int wi = 0; wi < VW; ++wi) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t sel = hf ? 0x7632u : 0x5410u;
          const uint32_t x = __byte_perm(va[wi], vb[wi], sel), y = __byte_perm(vc[wi], vd[wi], sel);
          const int mt = 4 * wi + 2 * hf;
          mma_f16_16816(acc[mt], and_or(x, 0x000F000Fu, kMagic), and_or(x, 0x00F000F0u, kMagic),
                        and_or(y, 0x000F000Fu, kMagic), and_or(y, 0x00F000F0u, kMagic), b01, b23);
          const uint32_t x8 = x >> 8, y8 = y >> 8;
          mma_f16_16816(acc[mt + 1], and_or(x8, 0x000F000Fu, kMagic), and_or(x8, 0x00F000F0u, kMagic),
                        and_or(y8, 0x000F000Fu, kMagic), and_or(y8, 0x00F000F0u, kMagic), b01, b23);
        }
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  __syncwarp();

  // -------- epilogue: finish the corrections, normalise, store the partial
  l0 = warp_sum_g(l0);
  l1 = warp_sum_g(l1);
  ps0 = warp_sum_g(ps0);
  ps1 = warp_sum_g(ps1);
  pz0 = warp_sum_g(pz0);
  pz1 = warp_sum_g(pz1);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const float off0 = 1024.f * ps0, off1 = 1024.f * ps1;
  float o0[D / 8], o1[D / 8];
#pragma unroll
  for (int mt = 0; mt < Gm::MT; ++mt) {
    o0[2 * mt] = (acc[mt][0] - off0 - pz0) * inv0;
    o1[2 * mt] = (acc[mt][1] - off1 - pz1) * inv1;
    o0[2 * mt + 1] = ((acc[mt][2] - off0) * 0.0625f - pz0) * inv0;
    o1[2 * mt + 1] = ((acc[mt][3] - off1) * 0.0625f - pz1) * inv1;
  }
  const float lse0 = l0 > 0.f ? m0 + log2f(l0) : -INFINITY;
  const float lse1 = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
  store_partial<D>(p.s, slot, sub, h, lane, o0, o1, lse0, lse1);
}

template <int D, int NSTAGE>
__global__ void __launch_bounds__(256, 2) decode_int4_kernel(const Int4Params p) {
  extern __shared__ __align__(16) uint8_t smem[];
  using Gm = Int4Geom<D>;
  const int warp = threadIdx.x >> 5;
  uint8_t *ring = smem + warp * (NSTAGE * Gm::STAGE + Gm::QBYTES);
  uint8_t *qarea = ring + NSTAGE * Gm::STAGE;
  const int hl = warp % p.s.heads_per_cta;
  const int sub = warp / p.s.heads_per_cta;
  const int h = blockIdx.y * p.s.heads_per_cta + hl;
  for_each_piece(p.s, &g_flags_decode_int4, [&](int b, int t0, int t1, long long slot) {
    int4_piece<D, NSTAGE>(p, ring, qarea, b, h, sub, t0, t1, slot);
  });
}

constexpr int kStagesInt4 = 4;

template <int D>
size_t int4_smem_bytes() {
  return 8 * static_cast<size_t>(kStagesInt4 * Int4Geom<D>::STAGE + Int4Geom<D>::QBYTES);
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
static kvq_status launch_int4(const Int4Params &p, const SplitPlan &plan, const MergeArgs &m,
                              cudaStream_t s) {
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
  merge_kernel<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(m);
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
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_scale, 4) ||
      !aligned(v_scale, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(out, 16) || !aligned(workspace, 16) || (rht_signs && !aligned(rht_signs, 16)))
    return KVQ_ERR_INVALID_ARG;
  if (max_blocks < 1) return KVQ_ERR_INVALID_ARG;
  const size_t need = kvq::workspace_bytes(B, Hq, D, plan);
  if (workspace_bytes < need) return KVQ_ERR_WORKSPACE;

  SplitArgs sa;
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
  const long long prows = plan.slots * plan.warps_per_head * Hq;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  sa.part_o = reinterpret_cast<float *>(ws);
  size_t off = ((prows * D * sizeof(float)) + 255) / 256 * 256;
  sa.part_lse = reinterpret_cast<float *>(ws + off);
  off += ((prows * sizeof(float)) + 255) / 256 * 256;
  sa.seg_first = reinterpret_cast<int32_t *>(ws + off);
  off += ((B * sizeof(int32_t)) + 255) / 256 * 256;
  sa.seg_last = reinterpret_cast<int32_t *>(ws + off);

  Int4Params p;
  p.s = sa;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = reinterpret_cast<const uint32_t *>(k_scale);
  p.v_scale = reinterpret_cast<const uint32_t *>(v_scale);
  p.block_table = block_table;
  p.signs = rht_signs;
  const double sm = rht_signs ? static_cast<double>(softmax_scale) / D : softmax_scale;
  p.sm_log2 = static_cast<float>(sm * 1.4426950408889634);
  p.num_blocks = num_blocks;

  MergeArgs m;
  m.s = sa;
  m.signs = rht_signs;
  m.out = out;
  m.out_dtype = out_dtype;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return D == 128 ? launch_int4<128>(p, plan, m, s) : launch_int4<64>(p, plan, m, s);
}
