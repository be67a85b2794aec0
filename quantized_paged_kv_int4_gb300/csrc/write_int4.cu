// kvq_write_int4: random-sign Hadamard rotation + asymmetric INT4 quantization + page scatter.
//
// Follows int4_per_token_head.py, reshape_and_cache_int4 (single_rht of K and V, cast back to
// bf16) and _reshape_cache_int4_kernel (per (token, head) min/max, scale, zero-point hidden in the
// scale word's low mantissa bits, nibble packing, slot_mapping scatter). The rotation is fused:
// the rotated vector never goes to memory.
//
// Mapping: one thread per (token, kv head) vector (write_int4_kernel below): the rotation keeps
// the pages' stage order h = 1, 2, ..., D/2 on packed fp32 pairs inside the thread. Writes of up
// to 8192 (token, head) pairs -- a decode step's new tokens -- take write_int4_lanes_kernel
// instead (eight lanes per vector, the same stage order and bytes, shorter per-vector latency).
// Quantization avoids float<->int conversions: for u = x * inv + zp (two roundings, as the pages),
// clamp(rha(u), 0, 15) == trunc(clamp(u + 0.5, 0, 15.5)) (u + 0.5 rounded as the pages' rha does;
// for u < 0 both give 0), and trunc of a value in [0, 15.5] is the low bits of (value + 2^23)
// added with round-toward-zero.

#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {

__device__ unsigned g_flags_write = 0;

struct WriteParams {
  const __nv_bfloat16 *key, *value;
  int64_t k_stride_t, k_stride_h, v_stride_t, v_stride_h;
  uint8_t *k_cache, *v_cache;
  uint32_t *k_scale, *v_scale;
  const int64_t *slot_mapping;
  const float *signs;
  int32_t T, Hk, block_size;
  int64_t num_blocks;
  uint32_t pairs;               // T * Hk (< 2^31)
  uint32_t hk_magic, hk_shift;  // pair / Hk == (umulhi(pair, hk_magic) + pair) >> hk_shift
};

// Bits of the code clamp(rha(u), 0, 15) for the fp32 value u the pages round, as 0x49000000 | code.
// w = fl(u + 0.5) scaled by 2^-4 is one fused multiply-add (u * 2^-4 is exact, so its single
// rounding is that of u + 0.5), saturated to [0, 1] (NaN -> 0); adding 2^19 toward zero leaves
// trunc(16 w) in the low bits (the ulp at 2^19 is 2^-4), and an integer min caps it at 15. Equal to
// trunc(clamp(fl(u + 0.5), 0, 15.5)), which is clamp(rha(u), 0, 15) for every u.
__device__ __forceinline__ uint32_t code_bits(float u) {
  const float w = __saturatef(__fmaf_rn(u, 0.0625f, 0.03125f));
  return min(__float_as_uint(__fadd_rz(w, 524288.0f)), 0x4900000Fu);
}

// Eight code words (element 2i in the low nibble of byte i) -> one packed word. lo + (hi << 4)
// puts a finished byte in bits 0..7 (the constant upper bits land above it); byte_perm gathers.
__device__ __forceinline__ uint32_t pack_codes(const uint32_t (&c)[8]) {
  const uint32_t b0 = c[0] + (c[1] << 4), b1 = c[2] + (c[3] << 4);
  const uint32_t b2 = c[4] + (c[5] << 4), b3 = c[6] + (c[7] << 4);
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) {
  __nv_bfloat162 r;
  memcpy(&r, &w, 4);
  return r;
}

__device__ __forceinline__ uint32_t bf2_bits(float lo, float hi) {
  const __nv_bfloat162 r = __float22bfloat162_rn(make_float2(lo, hi));
  uint32_t w;
  memcpy(&w, &r, 4);
  return w;
}

// The packed fp32 pair helpers (add2 / sub2, kvq_device.cuh) round each component exactly like
// the scalar op. Only packed adds and subtracts are used: a packed multiply feeding a packed add
// can be fused into a multiply-add by the assembler, which would drop the intermediate rounding.

// One thread per (token, kv head) vector of K or V: the whole D-element rotation, the min / max,
// the three divisions and the packing run in the thread, so nothing is repeated across lanes and
// no butterfly stage crosses lanes. A warp takes 16 (token, head) pairs per tile (lane 2i: K of
// pair i, lane 2i + 1: V); it copies the tile's 32 rows into shared memory with coalesced 16-byte
// cp.async (one tile ahead, two buffers per warp) and each lane then reads its own row (row
// stride D * 2 + 16 bytes: the 8 lanes of a quarter-warp read distinct banks).
// Packed fp32 pairs hold elements (k, k + D/2): the stages h = 1 .. D/4 run on pairs
// (add.rn / sub.rn .f32x2, each component rounded like the scalar op), the last stage h = D/2
// inside each pair -- the pages' stage order for every element.
template <int D>
struct WriteGeom {
  static constexpr int RB = D * 2;           // bytes of one bf16 row
  static constexpr int STRIDE = RB + 16;     // padded row in shared memory
  static constexpr int CHUNKS = RB / 16;     // 16-byte chunks per row
  static constexpr int ROWS_PER_COPY = 32 / CHUNKS;
  static constexpr int BUF = 32 * STRIDE;    // one warp buffer
  static constexpr int WARPS = 4;
  static constexpr int SMEM = WARPS * 2 * BUF + D / 2 * 4;  // two buffers per warp, the sign masks
  static constexpr int H = D / 2;            // packed pairs per row
};

template <int D, bool ROT>
__global__ void __launch_bounds__(128, 3) write_int4_kernel(const WriteParams p, long long tiles) {
  using G = WriteGeom<D>;
  constexpr int H = G::H, NW = D / 2;  // packed pairs, bf16 words per row
  extern __shared__ __align__(16) uint8_t wsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *bufs = wsm + warp * 2 * G::BUF;
  uint32_t *smask = reinterpret_cast<uint32_t *>(wsm + G::WARPS * 2 * G::BUF);
  if constexpr (ROT) {  // x * d1 with d1 = +-1 is an exact sign flip: XOR masks of the bf16 words
    for (int i = threadIdx.x; i < NW; i += blockDim.x) {
      const float s0 = __ldg(p.signs + 2 * i), s1 = __ldg(p.signs + 2 * i + 1);
      smask[i] = ((__float_as_uint(s0) >> 16) & 0x8000u) | (__float_as_uint(s1) & 0x80000000u);
    }
  }
  __syncthreads();

  // this lane's row of tile `tile`: pair index, token, head, source row, destination slot
  struct Row {
    const __nv_bfloat16 *src;
    long long slot;
    int h;
    bool live;
  };
  auto row_of = [&](long long tile) {
    Row r;
    const uint32_t pair = static_cast<uint32_t>(tile) * 16u + (lane >> 1);
    r.live = pair < p.pairs;
    const uint32_t t = (__umulhi(pair, p.hk_magic) + pair) >> p.hk_shift;
    const int tt = r.live ? static_cast<int>(t) : 0;
    r.h = r.live ? static_cast<int>(pair - t * static_cast<uint32_t>(p.Hk)) : 0;
    r.src = (lane & 1) ? p.value + tt * p.v_stride_t + r.h * p.v_stride_h
                       : p.key + tt * p.k_stride_t + r.h * p.k_stride_h;
    r.slot = r.live ? __ldg(p.slot_mapping + tt) : -1;
    return r;
  };
  // copy the tile's 32 rows into buffer b: copy i moves rows i * R .. i * R + R - 1 (R = 32 /
  // CHUNKS), CHUNKS lanes per row, 16 bytes each; a row's source address comes from its lane
  auto issue = [&](const Row &me, int b) {
    const uint32_t dst = smem_u32(bufs + b * G::BUF);
    const int sub = lane / G::CHUNKS, col = lane % G::CHUNKS;
#pragma unroll
    for (int i = 0; i < G::CHUNKS; ++i) {
      const int row = i * G::ROWS_PER_COPY + sub;
      const unsigned long long a = __shfl_sync(FULL, reinterpret_cast<unsigned long long>(me.src), row);
      const bool ok = __shfl_sync(FULL, static_cast<int>(me.live), row) != 0;
      cp_async<16>(dst + row * G::STRIDE + col * 16, reinterpret_cast<const uint8_t *>(a) + col * 16, ok);
    }
    cp_async_commit();
  };

  long long tile = static_cast<long long>(blockIdx.x) * G::WARPS + warp;
  const long long step = static_cast<long long>(gridDim.x) * G::WARPS;
  Row cur = row_of(tile < tiles ? tile : 0);
  if (tile < tiles) issue(cur, 0);
  int b = 0;
  for (; tile < tiles; tile += step) {
    const long long nt = tile + step;
    Row nxt = cur;
    if (nt < tiles) {
      nxt = row_of(nt);
      issue(nxt, b ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    const uint8_t *rp = bufs + b * G::BUF + lane * G::STRIDE;
    uint32_t w[NW];
#pragma unroll
    for (int i = 0; i < NW / 4; ++i) {
      const uint4 v = lds128(rp + 16 * i);
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
    __syncwarp();  // every lane has its row: the buffer may be refilled by the next issue

    uint32_t wb[NW];  // the vector as bf16 pairs after the rotation and its bf16 cast
    if constexpr (ROT) {
#pragma unroll
      for (int i = 0; i < NW; ++i) w[i] ^= smask[i];
      unsigned long long P[H];  // P[k] = (x[k], x[k + H])
#pragma unroll
      for (int k = 0; k < H; ++k) {
        const uint32_t a = w[k >> 1], c = w[(k + H) >> 1];
        P[k] = f2pack(__uint_as_float((k & 1) ? (a & 0xffff0000u) : (a << 16)),
                      __uint_as_float((k & 1) ? (c & 0xffff0000u) : (c << 16)));
      }
#pragma unroll
      for (int h = 1; h < H; h <<= 1) {
#pragma unroll
        for (int k = 0; k < H; ++k) {
          if (!(k & h)) {
            const unsigned long long s = add2(P[k], P[k + h]), d = sub2(P[k], P[k + h]);
            P[k] = s;
            P[k + h] = d;
          }
        }
      }
      float x[D];
#pragma unroll
      for (int k = 0; k < H; ++k) {  // the last stage, h = D/2, inside each pair
        float lo, hi;
        f2unpack(P[k], lo, hi);
        x[k] = __fadd_rn(lo, hi);
        x[k + H] = __fsub_rn(lo, hi);
      }
#pragma unroll
      for (int i = 0; i < NW; ++i) wb[i] = bf2_bits(x[2 * i], x[2 * i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < NW; ++i) wb[i] = w[i];
    }

    // min / max over the vector (bf16 pairs: exact, so any order gives the same result: eight
    // independent chains, then a tree), scale, zero-point and inverse per vector
    __nv_bfloat162 mnc[8], mxc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) mnc[c] = mxc[c] = as_bf2(wb[c]);
#pragma unroll
    for (int i = 8; i < NW; ++i) {
      mnc[i & 7] = __hmin2(mnc[i & 7], as_bf2(wb[i]));
      mxc[i & 7] = __hmax2(mxc[i & 7], as_bf2(wb[i]));
    }
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1) {
#pragma unroll
      for (int c = 0; c < w; ++c) {
        mnc[c] = __hmin2(mnc[c], mnc[c + w]);
        mxc[c] = __hmax2(mxc[c], mxc[c + w]);
      }
    }
    const __nv_bfloat162 mn2 = mnc[0], mx2 = mxc[0];
    const float mn = fminf(__low2float(mn2), __high2float(mn2));
    const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
    const float scale = fmaxf(__fdiv_rn(__fsub_rn(mx, mn), 15.0f), 1e-6f);
    const uint32_t zpi = code_bits(__fdiv_rn(-mn, scale)) & 0xFu;
    const float zp = static_cast<float>(zpi);
    const float inv = __fdiv_rn(1.0f, scale);

    bool valid = cur.live;
    if (valid && cur.slot >= p.num_blocks * p.block_size) {
      if (!(lane & 1)) atomicOr(&g_flags_write, ERR_SLOT);
      valid = false;
    }
    valid = valid && cur.slot >= 0;  // padding tokens store nothing
    if (valid) {
      uint32_t packed[D / 8];
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        uint32_t c[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // u = x * inv + zp with both roundings (scalar _rn: never fused)
          const uint32_t v = wb[4 * i + k];
          c[2 * k] = code_bits(__fadd_rn(__fmul_rn(__uint_as_float(v << 16), inv), zp));
          c[2 * k + 1] = code_bits(__fadd_rn(__fmul_rn(__uint_as_float(v & 0xffff0000u), inv), zp));
        }
        packed[i] = pack_codes(c);
      }
      // [num_blocks][block_size][Hk] flattened: (slot / bs * bs + slot % bs) * Hk + h
      const long long row = cur.slot * p.Hk + cur.h;
      uint8_t *dst = ((lane & 1) ? p.v_cache : p.k_cache) + row * (D / 2);
#pragma unroll
      for (int i = 0; i < D / 32; ++i)
        reinterpret_cast<uint4 *>(dst)[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
      ((lane & 1) ? p.v_scale : p.k_scale)[row] = (__float_as_uint(scale) & 0xFFFFFFF0u) | zpi;
    }
    cur = nxt;
    b ^= 1;
  }
}

// ---- eight lanes per vector (write_int4_lanes_kernel): the shorter path for small writes ------
// A decode step writes B new tokens, a few hundred vectors: one thread per vector would leave
// every thread a whole rotation in sequence. Here lane l8 of a vector's eight holds elements
// 16 l8 .. 16 l8 + 15 (D = 128): the stages h = 1 .. 8 run inside the lane, h = 16, 32, 64 on a
// per-warp shared-memory transpose (rows r, r ^ 1, 2, 4 of the 8 x 16 view) -- the same stage order,
// so the bytes are the same; min / max finish across the 8 lanes with shuffles.
template <int D>
struct LaneGeom {
  static constexpr int E = D / 8;          // elements per lane (one row of the 8 x E vector view)
  static constexpr int CPL = E / 8;        // columns per lane in the transposed view
  static constexpr int ROW = E + 4;        // padded row (words): conflict-free row and column access
  static constexpr int VEC = 8 * ROW + 16; // padded vector: the 4 vectors of a warp in two bank halves
};

// One lane's share of a (token, head) vector: E bf16 values as E/2 words (element 2i low).
template <int D>
struct LaneUnit {
  uint32_t w[D / 16];
  long long slot;
  int t, h;
  bool in_range;
};

// Tile = 16 (token, kv head) pairs; warp w takes pairs 2w, 2w + 1, lanes 8v .. 8v + 7 vector v
// (K of pair 0, V of pair 0, K of pair 1, V of pair 1).
template <int D>
__device__ __forceinline__ void load_lane_unit(const WriteParams &p, long long tile, int warp, int v, int l8,
                                          LaneUnit<D> &u) {
  constexpr int E = D / 8;
  const uint32_t pair = static_cast<uint32_t>(tile) * 16u + warp * 2 + (v >> 1);
  u.in_range = pair < p.pairs;
  const uint32_t t = (__umulhi(pair, p.hk_magic) + pair) >> p.hk_shift;
  u.t = u.in_range ? static_cast<int>(t) : 0;
  u.h = u.in_range ? static_cast<int>(pair - t * static_cast<uint32_t>(p.Hk)) : 0;
  u.slot = u.in_range ? __ldg(p.slot_mapping + u.t) : -1;
  const __nv_bfloat16 *src = ((v & 1) ? p.value + u.t * p.v_stride_t + u.h * p.v_stride_h
                                      : p.key + u.t * p.k_stride_t + u.h * p.k_stride_h) + l8 * E;
#pragma unroll
  for (int i = 0; i < E / 8; ++i) {
    // loaded whatever the slot says (a skipped token's row is read but not stored), so the load
    // does not wait for slot_mapping
    const uint4 raw = u.in_range ? __ldg(reinterpret_cast<const uint4 *>(src) + i) : make_uint4(0, 0, 0, 0);
    u.w[4 * i] = raw.x;
    u.w[4 * i + 1] = raw.y;
    u.w[4 * i + 2] = raw.z;
    u.w[4 * i + 3] = raw.w;
  }
}

template <int D, bool ROT>
__global__ void __launch_bounds__(256, 4) write_int4_lanes_kernel(const WriteParams p, long long tiles) {
  using Wg = LaneGeom<D>;
  constexpr int E = Wg::E, CPL = Wg::CPL, NW = E / 2;
  __shared__ __align__(16) float s_buf[8][4 * Wg::VEC];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v = lane >> 3, l8 = lane & 7;
  const bool is_v = v & 1;
  float *buf = &s_buf[warp][v * Wg::VEC];

  // x * d1 with d1 = +-1 is an exact sign flip: XOR the bf16 sign bits of the lane's words
  uint32_t sgn[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) sgn[i] = 0;
  if constexpr (ROT) {
    const float4 *sg = reinterpret_cast<const float4 *>(p.signs + l8 * E);
#pragma unroll
    for (int i = 0; i < E / 4; ++i) {
      const float4 sv = __ldg(sg + i);
      sgn[2 * i] = ((__float_as_uint(sv.x) >> 16) & 0x8000u) | (__float_as_uint(sv.y) & 0x80000000u);
      sgn[2 * i + 1] = ((__float_as_uint(sv.z) >> 16) & 0x8000u) | (__float_as_uint(sv.w) & 0x80000000u);
    }
  }

  LaneUnit<D> cur;
  long long tile = blockIdx.x;
  if (tile < tiles) load_lane_unit<D>(p, tile, warp, v, l8, cur);
  for (; tile < tiles; tile += gridDim.x) {
    LaneUnit<D> nxt;
    const long long nt = tile + gridDim.x;
    if (nt < tiles) load_lane_unit<D>(p, nt, warp, v, l8, nxt);

    bool valid = cur.in_range;
    if (valid && cur.slot >= p.num_blocks * p.block_size) {
      if (l8 == 0 && !is_v) atomicOr(&g_flags_write, ERR_SLOT);
      valid = false;
    }
    valid = valid && cur.slot >= 0;  // padding tokens store nothing

    uint32_t wb[NW];  // the vector as bf16 pairs after the rotation and its bf16 cast
    if constexpr (ROT) {
      float x[E];
#pragma unroll
      for (int i = 0; i < NW; ++i) {
        const uint32_t w = cur.w[i] ^ sgn[i];
        x[2 * i] = __uint_as_float(w << 16);
        x[2 * i + 1] = __uint_as_float(w & 0xffff0000u);
      }
      butterfly_local2<E>(x);  // h = 1 .. E/2 inside the lane's row
      // stages h = E, 2E, 4E pair rows r and r ^ 1, 2, 4: transpose, butterfly over rows, back
      __syncwarp();  // the previous tile's reads of buf are done
#pragma unroll
      for (int i = 0; i < E / 4; ++i)
        *reinterpret_cast<float4 *>(buf + l8 * Wg::ROW + 4 * i) = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
      __syncwarp();
      float c[CPL][8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if constexpr (CPL == 2) {
          const float2 f = *reinterpret_cast<const float2 *>(buf + r * Wg::ROW + 2 * l8);
          c[0][r] = f.x;
          c[1][r] = f.y;
        } else {
          c[0][r] = buf[r * Wg::ROW + l8];
        }
      }
      if constexpr (CPL == 2) {
        butterfly_cols2(c);
      } else {
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc) butterfly_local<8>(c[cc]);
      }
      __syncwarp();
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if constexpr (CPL == 2)
          *reinterpret_cast<float2 *>(buf + r * Wg::ROW + 2 * l8) = make_float2(c[0][r], c[1][r]);
        else
          buf[r * Wg::ROW + l8] = c[0][r];
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < E / 4; ++i) {
        const float4 f = *reinterpret_cast<const float4 *>(buf + l8 * Wg::ROW + 4 * i);
        wb[2 * i] = bf2_bits(f.x, f.y);
        wb[2 * i + 1] = bf2_bits(f.z, f.w);
      }
    } else {
#pragma unroll
      for (int i = 0; i < NW; ++i) wb[i] = cur.w[i];
    }

    // min / max over the vector: bf16 pairs in the lane (exact), then fp32 across the 8 lanes
    __nv_bfloat162 mn2 = as_bf2(wb[0]), mx2 = mn2;
#pragma unroll
    for (int i = 1; i < NW; ++i) {
      mn2 = __hmin2(mn2, as_bf2(wb[i]));
      mx2 = __hmax2(mx2, as_bf2(wb[i]));
    }
    float mn = fminf(__low2float(mn2), __high2float(mn2));
    float mx = fmaxf(__low2float(mx2), __high2float(mx2));
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(FULL, mn, m));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, m));
    }
    const float scale = fmaxf(__fdiv_rn(__fsub_rn(mx, mn), 15.0f), 1e-6f);
    const uint32_t zpi = code_bits(__fdiv_rn(-mn, scale)) & 0xFu;
    const float zp = static_cast<float>(zpi);
    const float inv = __fdiv_rn(1.0f, scale);

    uint32_t packed[E / 8];
#pragma unroll
    for (int i = 0; i < E / 8; ++i) {
      uint32_t c[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w = wb[4 * i + k];
        c[2 * k] = code_bits(__fadd_rn(__fmul_rn(__uint_as_float(w << 16), inv), zp));
        c[2 * k + 1] = code_bits(__fadd_rn(__fmul_rn(__uint_as_float(w & 0xffff0000u), inv), zp));
      }
      packed[i] = pack_codes(c);
    }
    if (valid) {
      // [num_blocks][block_size][Hk] flattened: (slot / bs * bs + slot % bs) * Hk + h
      const long long row = cur.slot * p.Hk + cur.h;
      uint8_t *dst = (is_v ? p.v_cache : p.k_cache) + row * (D / 2) + l8 * (E / 2);
      if constexpr (E == 16)
        *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
      else
        *reinterpret_cast<uint32_t *>(dst) = packed[0];
      if (l8 == 0) (is_v ? p.v_scale : p.k_scale)[row] = (__float_as_uint(scale) & 0xFFFFFFF0u) | zpi;
    }
    if (nt < tiles) cur = nxt;
  }
}

// (token, head) pairs up to which a write takes the eight-lanes-per-vector kernel: measured on
// GB300 (Hk 8, D 128), the two kernels break even at 1024 tokens (8.2 us); at 32 tokens the lane
// form takes 5.8 us against 6.9, at 4096 tokens 14.3 against 11.9
constexpr uint32_t kLanesMaxPairs = 8192;

template <int D, bool ROT>
kvq_status launch_write(const WriteParams &p, long long tiles, cudaStream_t s) {
  using G = WriteGeom<D>;
  static size_t attr_done[kMaxDevices] = {};
  if (ensure_dynamic_smem(write_int4_kernel<D, ROT>, G::SMEM, attr_done) != cudaSuccess) return KVQ_ERR_CUDA;
  static int per_sm = 0;  // resident CTAs per SM, from the occupancy calculator
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, write_int4_kernel<D, ROT>, 128, G::SMEM) != cudaSuccess ||
        n < 1)
      n = 1;
    per_sm = n;
  }
  const long long cap = static_cast<long long>(sm_count() > 0 ? sm_count() : 1) * per_sm;
  if (p.pairs <= kLanesMaxPairs) {  // small write: eight lanes per vector, one 16-pair tile per CTA
    const long long cap8 = static_cast<long long>(sm_count() > 0 ? sm_count() : 1) * 4;
    write_int4_lanes_kernel<D, ROT><<<static_cast<unsigned>(tiles < cap8 ? tiles : cap8), 256, 0, s>>>(p, tiles);
    return launch_status();
  }
  const long long ctas = (tiles + G::WARPS - 1) / G::WARPS;
  write_int4_kernel<D, ROT><<<static_cast<unsigned>(ctas < cap ? ctas : cap), 128, G::SMEM, s>>>(p, tiles);
  return launch_status();
}

bool take_flags_write(cudaStream_t stream, unsigned *host_word) {
  static const unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(host_word, g_flags_write, sizeof(unsigned), 0,
                                cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return false;
  return cudaMemcpyToSymbolAsync(g_flags_write, &zero, sizeof(unsigned), 0,
                                 cudaMemcpyHostToDevice, stream) == cudaSuccess;
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_write_int4(const void *key, const void *value, int64_t k_stride_t,
                                     int64_t k_stride_h, int64_t v_stride_t, int64_t v_stride_h,
                                     uint8_t *k_cache, uint8_t *v_cache, float *k_scale,
                                     float *v_scale, const int64_t *slot_mapping,
                                     const float *rht_signs, int32_t T, int32_t Hk, int32_t D,
                                     int32_t block_size, int64_t num_blocks,
                                     kvq_stream_t stream) {
  if (T < 0 || Hk < 1 || block_size < 1 || num_blocks < 1) return KVQ_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (T == 0) return KVQ_OK;
  if (!key || !value || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping)
    return KVQ_ERR_INVALID_ARG;
  const int vec = 8;  // elements per 16-byte vector load
  if (!aligned(key, vec * 2) || !aligned(value, vec * 2) || k_stride_t % vec || k_stride_h % vec ||
      v_stride_t % vec || v_stride_h % vec || k_stride_t < 0 || k_stride_h < 0 ||
      v_stride_t < 0 || v_stride_h < 0)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_scale, 4) ||
      !aligned(v_scale, 4) || !aligned(slot_mapping, 8) || (rht_signs && !aligned(rht_signs, 16)))
    return KVQ_ERR_INVALID_ARG;

  WriteParams p;
  p.key = static_cast<const __nv_bfloat16 *>(key);
  p.value = static_cast<const __nv_bfloat16 *>(value);
  p.k_stride_t = k_stride_t;
  p.k_stride_h = k_stride_h;
  p.v_stride_t = v_stride_t;
  p.v_stride_h = v_stride_h;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = reinterpret_cast<uint32_t *>(k_scale);
  p.v_scale = reinterpret_cast<uint32_t *>(v_scale);
  p.slot_mapping = slot_mapping;
  p.signs = rht_signs;
  p.T = T;
  p.Hk = Hk;
  p.block_size = block_size;
  p.num_blocks = num_blocks;

  const long long pairs = static_cast<long long>(T) * Hk;
  if (pairs >= (1LL << 31)) return KVQ_ERR_UNSUPPORTED;
  p.pairs = static_cast<uint32_t>(pairs);
  // division by the invariant Hk (Granlund and Montgomery, "Division by invariant integers using
  // multiplication", round-up variant): l = ceil(log2 Hk), m = floor(2^32 (2^l - Hk) / Hk) + 1;
  // exact for every pair < 2^31, where umulhi(pair, m) + pair stays below 2^32
  uint32_t l = 0;
  while ((1LL << l) < Hk) ++l;
  p.hk_shift = l;
  p.hk_magic = static_cast<uint32_t>((((1ULL << 32) * ((1ULL << l) - static_cast<uint64_t>(Hk))) / Hk) + 1);
  const long long tiles = (pairs + 15) / 16;  // 16 (token, head) pairs per warp tile
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 128)
    return rht_signs ? launch_write<128, true>(p, tiles, s) : launch_write<128, false>(p, tiles, s);
  return rht_signs ? launch_write<64, true>(p, tiles, s) : launch_write<64, false>(p, tiles, s);
}
