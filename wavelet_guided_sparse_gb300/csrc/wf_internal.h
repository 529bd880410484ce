// Host-side interface between the C-ABI layer (wf_api.cu) and the kernel
// launchers (wf_dwt.cu, wf_score.cu, wf_filter.cu, wf_attn.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include <atomic>
#include <stdint.h>

#include "wavefilter.h"

namespace wf {

// Validated sizes handed to the launchers.
struct LaunchDims {
  int64_t units;  // batch * heads
  int n_prompt;
  int n_gen;
  int head_dim;
  int levels;
  int dtype;
};

// Plan of the recursive filter (cluster size, per-CTA capacity, where the
// token logits live); a pure function of the sizes.
struct FilterPlan {
  int cluster;       // CTAs per unit
  int spans_cap;     // max coarse survivors per CTA
  int rows_cap;      // spans_cap << levels
  int sorted_cap;    // power of two >= k_L (bitonic sort width)
  bool t_in_smem;    // token logits in shared memory (else workspace)
  size_t smem_bytes; // dynamic shared memory per CTA
  size_t t_bytes;    // workspace bytes for token logits (0 if in smem)
};

struct ScorePlan {
  int cluster;
  int per_cta;
  size_t smem_bytes;
};

struct AttnPlan {
  int cluster;
  int tile_keys;
  int n_tiles;
  size_t smem_bytes;
};

bool plan_filter(const LaunchDims& ld, const int32_t* k, FilterPlan* plan);
bool plan_score(const LaunchDims& ld, ScorePlan* plan);
bool plan_attn(const LaunchDims& ld, int budget, AttnPlan* plan);

cudaError_t launch_dwt_lowpass(const LaunchDims& ld, const void* kp, float* out, int levels,
                               cudaStream_t stream);
cudaError_t launch_score_topk(const LaunchDims& ld, const ScorePlan& plan, const void* q,
                              const float* al, int k_l, int32_t* idx_l, float* scores,
                              int32_t* status, cudaStream_t stream);
cudaError_t launch_recursive_filter(const LaunchDims& ld, const FilterPlan& plan, const void* q,
                                    const void* kp, const int32_t* idx_l, const int32_t* k,
                                    int32_t* idx, float* t_ws, int32_t* status,
                                    cudaStream_t stream);
cudaError_t launch_sparse_attn(const LaunchDims& ld, const AttnPlan& plan, const void* q,
                               const void* kp, const void* vp, const void* kg, const void* vg,
                               const int32_t* idx, int budget, float* o, float* lse,
                               int32_t* status, cudaStream_t stream);

// Dynamic shared memory the planners allow per CTA (the sm_103a opt-in limit
// is 227 KB; a little is left for static shared memory).
constexpr size_t kMaxSmem = 225 * 1024;

// Records the last CUDA error of this thread for wf_last_error_string().
void note_cuda_error(cudaError_t e);

// Raises a kernel's dynamic shared-memory limit to the device's opt-in
// maximum minus the kernel's static shared memory, once per device.
template <auto Kern>
inline cudaError_t ensure_max_smem() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, Kern);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           optin - static_cast<int>(fa.sharedSizeBytes));
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace wf
