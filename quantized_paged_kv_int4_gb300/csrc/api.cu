// libkvq host glue: status strings, split planning and workspace sizing, device-flag readout.

#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "kvq_host.h"

namespace kvq {

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

bool make_plan(int B, int Hk, int num_splits, SplitPlan *plan) {
  if (B < 0 || Hk < 1 || num_splits < 0) return false;
  int hpc;
  if (Hk <= 8) {
    if (Hk & (Hk - 1)) return false;  // 1, 2, 4 or 8
    hpc = Hk;
  } else {
    if (Hk % 8) return false;
    hpc = 8;
  }
  plan->heads_per_cta = hpc;
  plan->head_groups = Hk / hpc;
  plan->warps_per_head = 8 / hpc;
  if (num_splits > 0) {
    const long long ctas = static_cast<long long>(B) * num_splits;
    if (ctas > 0x7fffffffLL) return false;
    plan->seg_ctas = static_cast<int>(ctas);
    plan->slots = ctas;
  } else {
    const int sms = sm_count();
    if (sms <= 0) return false;
    // two resident CTAs per SM across all head groups
    plan->seg_ctas = (2 * sms + plan->head_groups - 1) / plan->head_groups;
    plan->slots = static_cast<long long>(plan->seg_ctas) + B;
  }
  return true;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool int4_tensor_maps(const void *k_cache, const void *v_cache, const void *k_scale, const void *v_scale,
                      long long num_blocks, int Hk, int D, Int4Maps *maps) {
  struct Entry {
    const void *kc, *vc, *ks, *vs;
    long long nb;
    int hk, d;
    Int4Maps maps;
  };
  static std::mutex mu;
  static Entry cache[16];
  static int n_cached = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cached; ++i) {
    const Entry &e = cache[i];
    if (e.kc == k_cache && e.vc == v_cache && e.ks == k_scale && e.vs == v_scale && e.nb == num_blocks &&
        e.hk == Hk && e.d == D) {
      *maps = e.maps;
      return true;
    }
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
  if (enc == nullptr) return false;
  Int4Maps m;
  std::memset(&m, 0, sizeof(m));
  const int hpb = Hk < 8 ? Hk : 8;  // heads per box: one CTA's kv heads
  const cuuint64_t rb = static_cast<cuuint64_t>(D / 2);
  // dims {row bytes, token, head, page}: the token stride (Hk rows) is larger than the head
  // stride, so a box lands in shared memory as [head][token][row]
  const cuuint64_t kv_dim[4] = {rb, 16, static_cast<cuuint64_t>(Hk), static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t kv_stride[3] = {rb * Hk, rb, rb * Hk * 16};
  const cuuint32_t kv_box[4] = {static_cast<cuuint32_t>(rb), 16, static_cast<cuuint32_t>(hpb), 1};
  const cuuint32_t ones[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  for (int i = 0; i < 2; ++i) {
    if (enc(i ? &m.v : &m.k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(i ? v_cache : k_cache), kv_dim,
            kv_stride, kv_box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  for (int i = 0; i < 2; ++i) {
    CUtensorMap *dst = i ? &m.vs : &m.ks;
    void *base = const_cast<void *>(i ? v_scale : k_scale);
    CUresult r;
    if (Hk > 8) {  // Hk a multiple of 8: a [16][8] box of words at the CTA's first head
      const cuuint64_t dim[3] = {static_cast<cuuint64_t>(Hk), 16, static_cast<cuuint64_t>(num_blocks)};
      const cuuint64_t stride[2] = {4ull * Hk, 64ull * Hk};
      const cuuint32_t box[3] = {8, 16, 1};
      r = enc(dst, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, base, dim, stride, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {  // the page's whole [16][Hk] block of words
      const cuuint64_t dim[2] = {16ull * Hk, static_cast<cuuint64_t>(num_blocks)};
      const cuuint64_t stride[1] = {64ull * Hk};
      const cuuint32_t box[2] = {static_cast<cuuint32_t>(16 * Hk), 1};
      r = enc(dst, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, base, dim, stride, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return false;
  }
  m.heads_per_box = hpb;
  Entry &e = cache[next];
  e.kc = k_cache;
  e.vc = v_cache;
  e.ks = k_scale;
  e.vs = v_scale;
  e.nb = num_blocks;
  e.hk = Hk;
  e.d = D;
  e.maps = m;
  next = (next + 1) % 16;
  if (n_cached < 16) ++n_cached;
  *maps = m;
  return true;
}

bool tq_tensor_map(const void *cache, long long num_blocks, int Hk, int slot_bytes, int row_bytes, CUtensorMap *map) {
  struct Entry {
    const void *c;
    long long nb;
    int hk, sb, rb;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry entries[16];
  static int n_cached = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cached; ++i) {
    const Entry &e = entries[i];
    if (e.c == cache && e.nb == num_blocks && e.hk == Hk && e.sb == slot_bytes && e.rb == row_bytes) {
      *map = e.map;
      return true;
    }
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
  if (enc == nullptr) return false;
  const cuuint64_t sb = static_cast<cuuint64_t>(slot_bytes);
  const cuuint64_t dim[4] = {sb, 16, static_cast<cuuint64_t>(Hk), static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t stride[3] = {sb * Hk, sb, sb * Hk * 16};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(row_bytes), 16, 1, 1};
  const cuuint32_t ones[4] = {1, 1, 1, 1};
  CUtensorMap m;
  if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(cache), dim, stride, box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry &e = entries[next];
  e.c = cache;
  e.nb = num_blocks;
  e.hk = Hk;
  e.sb = slot_bytes;
  e.rb = row_bytes;
  e.map = m;
  next = (next + 1) % 16;
  if (n_cached < 16) ++n_cached;
  *map = m;
  return true;
}

size_t workspace_bytes(int B, int Hq, int D, const SplitPlan &plan) {
  const size_t rows = static_cast<size_t>(plan.slots) * plan.warps_per_head * Hq;
  return round256(rows * D * sizeof(float)) + round256(rows * sizeof(float)) +
         2 * round256(static_cast<size_t>(B) * sizeof(int32_t));
}

void workspace_carve(void *workspace, int B, int Hq, int D, const SplitPlan &plan, float **part_o,
                     float **part_lse, int32_t **seg_first, int32_t **seg_last) {
  const size_t rows = static_cast<size_t>(plan.slots) * plan.warps_per_head * Hq;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  *part_o = reinterpret_cast<float *>(ws);
  ws += round256(rows * D * sizeof(float));
  *part_lse = reinterpret_cast<float *>(ws);
  ws += round256(rows * sizeof(float));
  *seg_first = reinterpret_cast<int32_t *>(ws);
  ws += round256(static_cast<size_t>(B) * sizeof(int32_t));
  *seg_last = reinterpret_cast<int32_t *>(ws);
}

// kvq_copy_async: a grid-stride loop of 16-byte copies.
__global__ void __launch_bounds__(256) copy16_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src,
                                                     long long n) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = src[i];
}

// The address a kernel uses for p: device (or managed) memory as it is, pinned host memory by its
// mapped device address; false for anything else (pageable host memory, an unknown pointer).
static bool device_view(const void *p, const void **view) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the error the query left
    return false;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *view = p;
    return true;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) {
    *view = a.devicePointer;
    return true;
  }
  return false;
}

static std::atomic<unsigned long long> g_wait_ns{2000000000ull};
static std::atomic<int> g_withhold{-1};
unsigned long long debug_wait_ns() { return g_wait_ns.load(); }
int debug_take_withhold() { return g_withhold.exchange(-1); }

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_debug_set_wait(uint64_t wait_limit_ns, int32_t withhold_stage) {
  if (withhold_stage < -1) return KVQ_ERR_INVALID_ARG;
  kvq::g_wait_ns.store(wait_limit_ns == 0 ? 2000000000ull : wait_limit_ns);
  kvq::g_withhold.store(withhold_stage);
  return KVQ_OK;
}

extern "C" kvq_status kvq_copy_async(void *dst, const void *src, size_t bytes, kvq_stream_t stream) {
  if (bytes == 0) return KVQ_OK;
  if (dst == nullptr || src == nullptr || bytes % 16 != 0 || !aligned(dst, 16) || !aligned(src, 16))
    return KVQ_ERR_INVALID_ARG;
  const void *d = nullptr, *s = nullptr;
  if (!device_view(dst, &d) || !device_view(src, &s)) return KVQ_ERR_INVALID_ARG;
  const uintptr_t a = reinterpret_cast<uintptr_t>(d), b = reinterpret_cast<uintptr_t>(s);
  if (a < b + bytes && b < a + bytes) return KVQ_ERR_INVALID_ARG;
  const long long n = static_cast<long long>(bytes / 16);
  const long long cap = static_cast<long long>(sm_count() > 0 ? sm_count() : 1) * 8;
  const long long grid = (n + 255) / 256 < cap ? (n + 255) / 256 : cap;
  copy16_kernel<<<static_cast<unsigned>(grid), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4 *>(const_cast<void *>(d)), static_cast<const uint4 *>(s), n);
  return launch_status();
}

extern "C" const char *kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARG: return "KVQ_ERR_INVALID_ARG: invalid pointer, size, stride or alignment";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED: shape outside the compiled set";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE: workspace too small";
    case KVQ_ERR_OUT_OF_RANGE: return "KVQ_ERR_OUT_OF_RANGE: device-side index check failed";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA: CUDA runtime error";
  }
  return "KVQ_ERR_UNKNOWN";
}

extern "C" int32_t kvq_abi_version(void) { return 5; }

extern "C" size_t kvq_decode_workspace_bytes(int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                             int32_t num_splits) {
  if (B < 0 || Hq < 1 || Hk < 1 || Hq % Hk || (D != 64 && D != 128)) return 0;
  SplitPlan plan;
  if (!make_plan(B, Hk, num_splits, &plan)) return 0;
  return workspace_bytes(B, Hq, D, plan) + qfrag_bytes(B, Hk, D);  // the INT4 call's query fragments
}

extern "C" kvq_status kvq_device_error(kvq_stream_t stream, uint32_t *flags) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned words[5] = {0, 0, 0, 0, 0};
  if (!take_flags_write(s, &words[0]) || !take_flags_decode_int4(s, &words[1]) ||
      !take_flags_decode_tq(s, &words[2]) || !take_flags_decode_tq_mse(s, &words[3]) ||
      !take_flags_kpool(s, &words[4]))
    return KVQ_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ERR_CUDA;
  const uint32_t all = words[0] | words[1] | words[2] | words[3] | words[4];
  if (flags) *flags = all;
  return all ? KVQ_ERR_OUT_OF_RANGE : KVQ_OK;
}
