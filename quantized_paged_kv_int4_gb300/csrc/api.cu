// libkvq host glue: status strings, split planning and workspace sizing, device-flag readout.

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

static size_t round256(size_t n) { return (n + 255) / 256 * 256; }

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

}  // namespace kvq

using namespace kvq;

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

extern "C" int32_t kvq_abi_version(void) { return 1; }

extern "C" size_t kvq_decode_workspace_bytes(int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                             int32_t num_splits) {
  if (B < 0 || Hq < 1 || Hk < 1 || Hq % Hk || (D != 64 && D != 128)) return 0;
  SplitPlan plan;
  if (!make_plan(B, Hk, num_splits, &plan)) return 0;
  return workspace_bytes(B, Hq, D, plan);
}

extern "C" kvq_status kvq_device_error(kvq_stream_t stream, uint32_t *flags) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned words[3] = {0, 0, 0};
  if (!take_flags_write(s, &words[0]) || !take_flags_decode_int4(s, &words[1]) ||
      !take_flags_decode_tq(s, &words[2]))
    return KVQ_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ERR_CUDA;
  const uint32_t all = words[0] | words[1] | words[2];
  if (flags) *flags = all;
  return all ? KVQ_ERR_OUT_OF_RANGE : KVQ_OK;
}
