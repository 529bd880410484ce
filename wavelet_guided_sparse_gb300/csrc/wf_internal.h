// Host-side interface between the C-ABI layer (wf_api.cu) and the kernel
// launchers (wf_dwt.cu: step 1; wf_path.cu: steps 2-5; wf_cache.cu: the
// cache writes of eqs. (2) and (4)).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "wavefilter.h"

namespace wf {

// Validated sizes handed to the launchers.
struct LaunchDims {
  int64_t units;  // batch * heads
  int batch;
  int n_prompt;
  int n_gen;
  int head_dim;
  int levels;
  int dtype;
};

// Phases of the fused path kernel (wf_path.cu).
enum : int { kPhaseScore = 1, kPhaseFilter = 2, kPhaseAttend = 4, kPhaseAll = 7 };
// Request bit for plan_path with kPhaseAll: compute A_L inside the path
// kernel (step 1 fused into the scoring) where the plan allows it.
enum : int { kPhaseFuseDwt = 8 };
// Request bit for plan_path with kPhaseAll or kPhaseScore when the caller
// passes a cached fp32 A_L: stage its rows by tensor copies where the plan
// allows it.
enum : int { kPhaseCachedAl = 16 };

// Launch plan of the path kernel; a pure function of the sizes and the
// device's SM count.
struct PathPlan {
  int mode;          // kPhase* bit set (without kPhaseFuseDwt)
  int fuse_dwt;      // 1: the path kernel computes A_L itself (no separate DWT launch)
  int al_stage;      // 1: cached A_L rows staged by bulk copies (PathArgs::al)
  int al_ring;       // their ring depth (64-row stages)
  int cluster;       // CTAs per unit
  int per_cta_p;     // score: coarse positions per CTA
  int rows_cap;      // filter: token rows per CTA (capacity)
  int sorted_cap;    // filter: power of two >= k_L
  int keys_cap;      // candidates per CTA (capacity)
  int gather_all;    // Top-K variant
  int klist_cap;     // attend: key slots per CTA (capacity)
  int tile_keys;     // attend: keys per staged tile
  int f_stages;      // filter: cp.async ring depth
  int a_stages;      // attend: cp.async ring depth
  bool t_in_smem;    // token logits in shared memory (else workspace)
  int filter_fast;   // 0: general filter; 1: token logits resident in tensor
                     // memory; 2: token logits recomputed per pass (no spill)
  int f_nb;          // fast filter: tensor-memory accumulator slots
  size_t smem_bytes; // dynamic shared memory per CTA
  size_t t_bytes;    // workspace bytes for token logits (0 if in shared memory)
};

// Row pitch (floats) of the coarse logits [U, P, pitch]: G rounded up to a
// multiple of four, so that every row starts on a 16-byte boundary.
inline int coarse_logit_pitch(int G) { return (G + 3) & ~3; }

// Pointers of one path launch (device memory unless noted).
struct PathArgs {
  const void *q, *kp, *vp, *kg, *vg;
  const float* zl;   // score phase without the fused stream: coarse logits
                     // [U, P, coarse_logit_pitch(G)], log2 domain (Q·A_L·log2e/√d)
  const float* al;   // or, instead: an fp32 A_L [U, P, d] whose logits the score
                     // phase forms itself
  const int32_t* idx_l_in;
  const int32_t* idx_in;
  int32_t* idx_l_out;
  float* scores_out;
  int32_t* idx_out;
  float* o;
  float* lse;
  int32_t* status;
  float* t_ws;
  const int32_t* k;  // host, levels + 1 entries (filter phase), else null
  int k_l;
  int budget;
};

int device_sm_count();
bool plan_path(const LaunchDims& ld, int mode, const int32_t* k, int k_l, int budget,
               int sm_count, PathPlan* plan);

// Streams Kp once and writes its level-`levels` Haar approximation as fp32
// to `out` [U, N_p/2^levels, d]; if zl != nullptr (levels = ld.levels), then
// also the coarse logits of every row against the unit's queries `q` to zl
// [U, P, coarse_logit_pitch(G)] in the log2 domain.
cudaError_t launch_dwt_lowpass(const LaunchDims& ld, const void* kp, float* out, const void* q,
                               float* zl, int levels, int32_t* status, cudaStream_t stream);

cudaError_t launch_path(const LaunchDims& ld, const PathPlan& plan, const PathArgs& args,
                        cudaStream_t stream);

// Cache initialisation (eq. (2)) from token-major K/V [batch, N_p + G,
// heads, d] into Kp/Vp/Kg/Vg, with fp32 A_L of the prompt keys if `al` is
// set; and the generation-row update (eq. (4)) from [batch, G, heads, d].
cudaError_t launch_cache_init(const LaunchDims& ld, const void* k, const void* v, void* kp,
                              void* vp, void* kg, void* vg, float* al, cudaStream_t stream);
cudaError_t launch_cache_update(const LaunchDims& ld, const void* k, const void* v, void* kg,
                                void* vg, cudaStream_t stream);
// Eq. (4) over `rows` positions per sequence (pos [batch, rows], prompt or
// generation) from token-major K/V [batch, rows, heads, d]; A_L (nullable)
// re-formed at the touched coarse positions; bad positions flagged in
// *status (nullable).
cudaError_t launch_cache_scatter(const LaunchDims& ld, const void* k, const void* v,
                                 const int32_t* pos, int rows, void* kp, void* vp, void* kg,
                                 void* vg, float* al, int32_t* status, cudaStream_t stream);

// Longer orthonormal bases (wf_basis.cu).  Filter taps (fp32 copy of the
// caller's low-pass) and the launch arguments of the level-by-level filter.
struct BasisTaps {
  float g[16];
  int n;
};
struct BasisFilterParams {
  const void* q;
  const void* kp;
  const float* a_all;                      // levels 1..L, level-major fp32 blocks
  int64_t level_off[WF_MAX_LEVELS + 1];    // element offset of level j's block
  int32_t* cand;                           // [2][units][cap]: candidates, survivors
  uint32_t* keys;                          // [units][cap] scores as ordered bits
  float* z;                                // [units][cap][G] logits (log2 domain)
  int32_t* idx;                            // out: [units][k_0] selected tokens
  int64_t units, cap;
  int n_prompt, n_gen, levels;
  int32_t k[WF_MAX_LEVELS + 1];
  float qscale;                            // log2(e) / sqrt(d)
};
// Extremal-phase Daubechies low-pass with n_moments vanishing moments (host;
// 2 n_moments doubles, highest power of the filter polynomial first).
int daubechies_lowpass(int n_moments, double* out);
cudaError_t launch_basis_pyramid(const LaunchDims& ld, const void* kp, float* a_all,
                                 const BasisTaps& taps, cudaStream_t stream);
cudaError_t launch_basis_filter(const LaunchDims& ld, const BasisFilterParams& p,
                                cudaStream_t stream);
// Level-L coarse logits of a longer basis in one pass over the tokens: the
// L periodic levels composed into one filter w of w_len taps (see
// basis_cascade), z_L[c][q] = zscale Σ_m w[m] Q_q·Kp[(2^L c + m) mod N_p],
// written to zl [U, P, gz] (bf16 inputs).
constexpr int kMaxCascade = 2048;
struct BasisCoarseParams {
  const void* q;
  const void* kp;
  float* zl;
  int n_prompt, n_gen, levels, w_len, gz;
  float zscale;
  float w[kMaxCascade];
};
// The composed filter of `levels` periodic levels of the low-pass g (taps
// doubles, computed in double, stored as fp32 in w); returns its length
// (levels·... = (2^levels - 1)(taps - 1) + 1), or -1 if above kMaxCascade.
int basis_cascade(const double* g, int taps, int levels, float* w);
int basis_cascade_len(int taps, int levels);
cudaError_t launch_basis_coarse(const LaunchDims& ld, const BasisCoarseParams& p,
                                cudaStream_t stream);

// Dynamic shared memory the planners allow per CTA (the sm_103a opt-in limit
// is 227 KB; a little is left for static shared memory).
constexpr size_t kMaxSmem = 225 * 1024;

// Poll limit armed by wf_debug_inject_wait_timeout for the next kernel
// launch that streams through mbarrier-counted copies (0: none); reading it
// disarms it.
uint32_t consume_wait_injection();

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
