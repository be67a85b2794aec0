// Host-side helpers shared by the libkvq translation units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Status of the launch just enqueued.
inline kvq_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// SM count of the current device (cached per device).
int sm_count();

// Read-and-clear of each translation unit's device flag word (enqueued on `stream`, then the
// caller synchronizes). Each returns false when the CUDA calls failed.
bool take_flags_write(cudaStream_t stream, unsigned *host_word);
bool take_flags_decode_int4(cudaStream_t stream, unsigned *host_word);
bool take_flags_decode_tq(cudaStream_t stream, unsigned *host_word);
bool take_flags_decode_tq_mse(cudaStream_t stream, unsigned *host_word);
bool take_flags_kpool(cudaStream_t stream, unsigned *host_word);

// Error-path test settings (kvq_debug_set_wait): the limit of the decode kernels' bounded waits on
// page copies, and the ring stage whose copies the next decode call withholds (taken by that call:
// -1 afterwards).
unsigned long long debug_wait_ns();
int debug_take_withhold();

// Split-partition geometry shared by workspace sizing and the launches.
struct SplitPlan {
  int heads_per_cta;   // kv heads one CTA covers (<= 8)
  int head_groups;     // Hk / heads_per_cta
  int warps_per_head;  // 8 / heads_per_cta
  int seg_ctas;        // CTAs along the sequence axis (grid.x)
  long long slots;     // partial-result slots (before the warps_per_head factor)
};
bool make_plan(int B, int Hk, int num_splits, SplitPlan *plan);
// Workspace: partial outputs [slots * warps_per_head, Hq, D] fp32, their log-sum-exps
// [slots * warps_per_head, Hq] fp32, then seg_first / seg_last [B] int32 (each region 256-byte
// aligned). Needs no initialisation.
size_t workspace_bytes(int B, int Hq, int D, const SplitPlan &plan);
inline size_t round256(size_t n) { return (n + 255) / 256 * 256; }
// Single-token INT4 decode: the rotated query's MMA fragments, (2 D/16 + 3) words per lane of one
// warp per (sequence, kv head), after the split workspace.
inline size_t qfrag_bytes(int B, int Hk, int D) {
  return round256(static_cast<size_t>(B) * Hk * (2 * (D / 16) + 3) * 32 * sizeof(uint32_t));
}
void workspace_carve(void *workspace, int B, int Hq, int D, const SplitPlan &plan, float **part_o,
                     float **part_lse, int32_t **seg_first, int32_t **seg_last);

// TMA descriptors of one INT4 cache (K, V pools and their scale words), see int4_tensor_maps.
struct Int4Maps {
  CUtensorMap k, v, ks, vs;
  int heads_per_box;  // kv heads one box covers: min(Hk, 8)
};
// Encode (or fetch from a small cache) the tensor maps of the pools, with HB = min(Hk, 8):
//   K / V  [num_blocks][16][Hk][D/2] bytes viewed as dims {D/2, 16, Hk, num_blocks} (token
//          stride Hk * D/2, head stride D/2); box {D/2, 16, HB, 1} = HB heads' 16 token rows
//          of one page, stored [head][token][row] with the 64B (D = 128) or 32B (D = 64) swizzle;
//   scales [num_blocks][16][Hk] words: Hk <= 8: dims {16 * Hk, num_blocks}, box {16 * Hk, 1}
//          (the page's whole block); Hk > 8: dims {Hk, 16, num_blocks}, box {8, 16, 1}.
// Returns false if the driver entry point is unavailable or an encode fails.
bool int4_tensor_maps(const void *k_cache, const void *v_cache, const void *k_scale, const void *v_scale,
                      long long num_blocks, int Hk, int D, Int4Maps *maps);
// The TurboQuant combined-slot pool [num_blocks][16][Hk][slot_bytes] viewed as dims
// {slot_bytes, 16, Hk, num_blocks} (token stride Hk * slot_bytes, head stride slot_bytes); box
// {row_bytes, 16, 1, 1} = the first row_bytes of the 16 slots of one (page, head), stored
// [token][row_bytes] without swizzle. slot_bytes and row_bytes multiples of 16, row_bytes <= 256
// and <= slot_bytes. Cached like int4_tensor_maps; false if the driver entry point is unavailable
// or the encode fails.
bool tq_tensor_map(const void *cache, long long num_blocks, int Hk, int slot_bytes, int row_bytes, CUtensorMap *map);

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device. The attribute
// lives with the function in each device's context, so it is set once per (instantiation,
// device): `done[dev]` holds the largest size set there so far (devices past kMaxDevices set it
// on every call).
constexpr int kMaxDevices = 64;
template <typename Kernel>
cudaError_t ensure_dynamic_smem(Kernel *kernel, size_t bytes, size_t (&done)[kMaxDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && done[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess && cached) done[dev] = bytes;
  return e;
}

// Launch `kernel` as a programmatic dependent of the kernel just enqueued on s (it may start once
// that kernel has executed griddepcontrol.launch_dependents, and must execute griddepcontrol.wait
// before reading anything that kernel writes).
template <typename Args>
cudaError_t launch_dependent(void (*kernel)(Args), dim3 grid, dim3 block, cudaStream_t s, const Args &a,
                             size_t dynamic_smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = dynamic_smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace kvq
