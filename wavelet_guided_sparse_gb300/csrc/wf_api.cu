// C ABI of the WaveFilter KV-filtering path: argument validation, workspace
// layout and the step driver.  Kernels live in wf_dwt.cu (step 1),
// wf_path.cu (steps 2-5, one cluster kernel whose phases the entry points
// select) and wf_cache.cu (the cache writes of eqs. (2) and (4)).
//
// Every entry point validates on the host first and enqueues nothing on a
// validation error.  Nothing here allocates device memory or synchronises,
// except wf_read_device_status(), which is documented as synchronising.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <algorithm>
#include <cmath>
#include <cstring>
#include <atomic>

#include "wavefilter.h"
#include "wf_internal.h"

#include <cuda_bf16.h>

namespace {

using wf::LaunchDims;

constexpr size_t kAlign = 256;
constexpr size_t kHeaderBytes = 256;  // status word + padding

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_bytes(int dtype) { return dtype == WF_BF16 ? 2 : 4; }

int check_dims(const wf_dims* d, LaunchDims* ld) {
  if (d == nullptr) return WF_ERR_NULL;
  if (d->dtype != WF_BF16 && d->dtype != WF_F32) return WF_ERR_UNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 128) return WF_ERR_UNSUPPORTED;
  if (d->batch < 1 || d->heads < 1 || d->n_prompt < 1 || d->n_gen < 1) return WF_ERR_SHAPE;
  if (d->levels < 1 || d->levels > WF_MAX_LEVELS) return WF_ERR_SHAPE;
  if (d->n_gen > WF_MAX_GEN) return WF_ERR_UNSUPPORTED;
  if (d->n_prompt % (1 << d->levels) != 0) return WF_ERR_SHAPE;
  const int64_t units = static_cast<int64_t>(d->batch) * d->heads;
  if (units > 65535) return WF_ERR_UNSUPPORTED;  // one grid row per unit
  ld->units = units;
  ld->batch = d->batch;
  ld->n_prompt = d->n_prompt;
  ld->n_gen = d->n_gen;
  ld->head_dim = d->head_dim;
  ld->levels = d->levels;
  ld->dtype = d->dtype;
  return WF_OK;
}

// Per-level survivor counts: 1 <= k_L <= N_p/2^L, 1 <= k_j <= 2 k_{j+1}.
int check_k(const LaunchDims& ld, const int32_t* k) {
  if (k == nullptr) return WF_ERR_NULL;
  const int P = ld.n_prompt >> ld.levels;
  if (k[ld.levels] < 1 || k[ld.levels] > P) return WF_ERR_SHAPE;
  for (int j = ld.levels - 1; j >= 0; --j)
    if (k[j] < 1 || static_cast<int64_t>(k[j]) > 2 * static_cast<int64_t>(k[j + 1]))
      return WF_ERR_SHAPE;
  return WF_OK;
}

// Workspace layout shared by every entry point: [status header | coarse
// logits | A_L | S_L | S | t].
struct Layout {
  size_t zl, al, idx_l, idx, t, total;
};

Layout layout(const LaunchDims& ld, const int32_t* k, const wf::PathPlan* fp) {
  Layout L;
  size_t o = kHeaderBytes;
  const size_t rows = static_cast<size_t>(ld.units) * (ld.n_prompt >> ld.levels);
  L.zl = o;  // coarse logits [U, P, coarse_logit_pitch(G)] fp32
  o = align_up(o + sizeof(float) * rows * wf::coarse_logit_pitch(ld.n_gen));
  L.al = o;  // fp32 A_L [U, P, d] of a separate streaming launch
  o = align_up(o + sizeof(float) * rows * ld.head_dim);
  L.idx_l = o;
  o = align_up(o + sizeof(int32_t) * ld.units * (k ? k[ld.levels] : 0));
  L.idx = o;
  o = align_up(o + sizeof(int32_t) * ld.units * (k ? k[0] : 0));
  L.t = o;
  o = align_up(o + (fp ? fp->t_bytes : 0));
  L.total = o;
  return L;
}

int32_t* status_word(void* ws) { return static_cast<int32_t*>(ws); }

// The plan of wf_step: one launch where the path kernel fuses step 1;
// otherwise two.  The second launch then forms the coarse logits itself from
// the A_L the stream wrote (*from_al: every CTA's A_L rows staged in shared
// memory, the cached-A_L path), or, where that staging does not fit, reads
// the logits the stream formed in its epilogue.
bool step_plan(const LaunchDims& ld, const int32_t* k, wf::PathPlan* plan, bool* from_al) {
  *from_al = false;
  const int sms = wf::device_sm_count();
  if (!wf::plan_path(ld, wf::kPhaseAll | wf::kPhaseFuseDwt, k, k[ld.levels], k[0], sms, plan))
    return false;
  if (plan->fuse_dwt) return true;
  wf::PathPlan c;
  if (wf::plan_path(ld, wf::kPhaseAll | wf::kPhaseCachedAl, k, k[ld.levels], k[0], sms, &c) &&
      c.al_stage) {
    *plan = c;
    *from_al = true;
  }
  return true;
}

// The longer-basis step takes the Haar path kernel with precomputed coarse
// logits when every level between L and 0 keeps all children (then only the
// level-L logits depend on the basis), the inputs are bf16, and the composed
// level-L filter is short enough; returns the plan of that route.
bool basis_coarse_route(const LaunchDims& ld, int32_t taps, const int32_t* k, wf::PathPlan* plan) {
  if (ld.dtype != WF_BF16 || ld.n_gen > 64 || wf::basis_cascade_len(taps, ld.levels) < 0)
    return false;
  for (int j = 1; j < ld.levels; ++j)
    if (k[j] != 2 * k[j + 1]) return false;
  return wf::plan_path(ld, wf::kPhaseAll, k, k[ld.levels], k[0], wf::device_sm_count(), plan);
}

// Filter taps of a longer basis: 2..16 taps, an even count.
int check_taps(const double* g, int32_t taps, wf::BasisTaps* t) {
  if (g == nullptr) return WF_ERR_NULL;
  if (taps < 2 || taps > 16 || taps % 2 != 0) return WF_ERR_UNSUPPORTED;
  t->n = taps;
  for (int i = 0; i < 16; ++i) t->g[i] = i < taps ? static_cast<float>(g[i]) : 0.f;
  return WF_OK;
}

// Workspace of the longer-basis step: [status header | A_1..A_L | candidates
// and survivors | keys | logits | selected tokens].
struct BasisLayout {
  size_t a_all, cand, keys, z, idx, total;
  int64_t cap;
};

BasisLayout basis_layout(const LaunchDims& ld, const int32_t* k) {
  BasisLayout L;
  int64_t cap = ld.n_prompt >> ld.levels;
  for (int j = 0; j < ld.levels; ++j) cap = std::max<int64_t>(cap, 2 * int64_t{k[j + 1]});
  L.cap = cap;
  size_t levels_el = 0;
  for (int j = 1; j <= ld.levels; ++j)
    levels_el += static_cast<size_t>(ld.units) * (ld.n_prompt >> j) * ld.head_dim;
  size_t o = kHeaderBytes;
  L.a_all = o;
  o = align_up(o + sizeof(float) * levels_el);
  L.cand = o;
  o = align_up(o + sizeof(int32_t) * 2 * ld.units * cap);
  L.keys = o;
  o = align_up(o + sizeof(uint32_t) * ld.units * cap);
  L.z = o;
  o = align_up(o + sizeof(float) * ld.units * cap * ld.n_gen);
  L.idx = o;
  o = align_up(o + sizeof(int32_t) * ld.units * k[0]);
  L.total = o;
  return L;
}

thread_local char g_last_error[256] = "no error";

// Poll limit of the next injected wait timeout (wf_debug_inject_wait_timeout).
std::atomic<uint32_t> g_wait_injection{0};

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return WF_OK;
  wf::note_cuda_error(e);
  return WF_ERR_CUDA;
}

}  // namespace

namespace wf {
uint32_t consume_wait_injection() { return g_wait_injection.exchange(0u); }

void note_cuda_error(cudaError_t e) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
}
}  // namespace wf

extern "C" {

const char* wf_last_error_string(void) { return g_last_error; }

const char* wf_status_string(int status) {
  switch (status) {
    case WF_OK: return "ok";
    case WF_ERR_NULL: return "a required pointer is NULL";
    case WF_ERR_SHAPE: return "inconsistent sizes or per-level k";
    case WF_ERR_UNSUPPORTED: return "unsupported head_dim, dtype, n_gen or size";
    case WF_ERR_WORKSPACE: return "workspace too small";
    case WF_ERR_CUDA: return "CUDA launch or query failed";
    case WF_ERR_DEVICE_CHECK: return "device-side check failed";
    case WF_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    default: return "unknown status";
  }
}

int wf_default_k_per_level(int32_t n_prompt, int32_t levels, int32_t budget, int32_t* k_out) {
  if (k_out == nullptr) return WF_ERR_NULL;
  if (levels < 1 || levels > WF_MAX_LEVELS || budget < 1 || n_prompt < 1) return WF_ERR_SHAPE;
  if (n_prompt % (1 << levels) != 0) return WF_ERR_SHAPE;
  const int64_t top = n_prompt >> levels;
  int64_t kl = (2 * static_cast<int64_t>(budget) + (1 << levels) - 1) >> levels;
  if (kl > top) kl = top;
  if (kl < 1) kl = 1;
  k_out[levels] = static_cast<int32_t>(kl);
  for (int j = levels - 1; j >= 1; --j) {
    const int64_t a = kl << (levels - j), b = n_prompt >> j;
    k_out[j] = static_cast<int32_t>(a < b ? a : b);
  }
  k_out[0] = budget;
  if (budget > 2 * static_cast<int64_t>(k_out[1 < levels ? 1 : levels])) return WF_ERR_SHAPE;
  return WF_OK;
}

int wf_workspace_bytes(const wf_dims* dims, const int32_t* k_per_level, size_t* bytes) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (bytes == nullptr) return WF_ERR_NULL;
  st = check_k(ld, k_per_level);
  if (st != WF_OK) return st;
  const int sms = wf::device_sm_count();
  wf::PathPlan all, step, filt;
  bool from_al = false;
  if (!wf::plan_path(ld, wf::kPhaseAll | wf::kPhaseFuseDwt, k_per_level, k_per_level[ld.levels],
                     k_per_level[0], sms, &all) ||
      !step_plan(ld, k_per_level, &step, &from_al) ||
      !wf::plan_path(ld, wf::kPhaseFilter, k_per_level, k_per_level[ld.levels], k_per_level[0],
                     sms, &filt))
    return WF_ERR_UNSUPPORTED;
  const size_t t = std::max(all.t_bytes, std::max(step.t_bytes, filt.t_bytes));
  const wf::PathPlan& big = all.t_bytes == t ? all : (step.t_bytes == t ? step : filt);
  *bytes = layout(ld, k_per_level, &big).total;
  return WF_OK;
}

int wf_step_launch_count(const wf_dims* dims, const int32_t* k_per_level, int32_t* launches) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (launches == nullptr) return WF_ERR_NULL;
  st = check_k(ld, k_per_level);
  if (st != WF_OK) return st;
  wf::PathPlan plan;
  if (!wf::plan_path(ld, wf::kPhaseAll | wf::kPhaseFuseDwt, k_per_level, k_per_level[ld.levels],
                     k_per_level[0], wf::device_sm_count(), &plan))
    return WF_ERR_UNSUPPORTED;
  *launches = plan.fuse_dwt ? 1 : 2;
  return WF_OK;
}

int wf_step_plan(const wf_dims* dims, const int32_t* k_per_level, wf_plan* out) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (out == nullptr) return WF_ERR_NULL;
  st = check_k(ld, k_per_level);
  if (st != WF_OK) return st;
  wf::PathPlan plan;
  bool from_al = false;
  if (!step_plan(ld, k_per_level, &plan, &from_al)) return WF_ERR_UNSUPPORTED;
  out->launches = plan.fuse_dwt ? 1 : 2;
  out->cluster = plan.cluster;
  out->final_gather = plan.gather_all;
  out->token_logits = plan.filter_fast == 1   ? WF_LOGITS_TENSOR_MEMORY
                      : plan.filter_fast == 2 ? WF_LOGITS_RECOMPUTED
                      : plan.t_in_smem        ? WF_LOGITS_SHARED
                                              : WF_LOGITS_WORKSPACE;
  out->smem_bytes = static_cast<int32_t>(plan.smem_bytes);
  out->filter_stages = plan.f_stages;
  out->attend_stages = plan.a_stages;
  out->stream_is_dwt_lowpass = from_al ? 1 : 0;
  out->al_stages = from_al && plan.al_stage ? plan.al_ring : 0;
  return WF_OK;
}

int wf_debug_inject_wait_timeout(int32_t polls) {
  if (polls < 0) return WF_ERR_SHAPE;
  g_wait_injection.store(static_cast<uint32_t>(polls));
  return WF_OK;
}

int wf_clear_device_status(void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr) return WF_ERR_NULL;
  if (workspace_bytes < kHeaderBytes) return WF_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(int32_t),
                                     static_cast<cudaStream_t>(stream)));
}

int wf_read_device_status(const void* workspace, size_t workspace_bytes, void* stream,
                          int32_t* status_out) {
  if (workspace == nullptr || status_out == nullptr) return WF_ERR_NULL;
  if (workspace_bytes < kHeaderBytes) return WF_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return WF_ERR_CUDA;
  *status_out = v;
  return WF_OK;
}

int wf_dwt_lowpass(const wf_dims* dims, const void* Kp, float* AL, float* A_all, void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (Kp == nullptr || AL == nullptr) return WF_ERR_NULL;
  if (!aligned16(Kp) || !aligned16(AL) || (A_all && !aligned16(A_all))) return WF_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = wf::launch_dwt_lowpass(ld, Kp, AL, nullptr, nullptr, ld.levels, nullptr, s);
  if (e == cudaSuccess && A_all != nullptr) {
    // Test aid: every level j = 1..L, each from its own pass over Kp.
    size_t off = 0;
    for (int j = 1; j <= ld.levels && e == cudaSuccess; ++j) {
      e = wf::launch_dwt_lowpass(ld, Kp, A_all + off, nullptr, nullptr, j, nullptr, s);
      off += static_cast<size_t>(ld.units) * (ld.n_prompt >> j) * ld.head_dim;
    }
  }
  return cuda_status(e);
}

int wf_cache_init(const wf_dims* dims, const void* K, const void* V, void* Kp, void* Vp,
                  void* Kg, void* Vg, float* AL, void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (K == nullptr || V == nullptr || Kp == nullptr || Vp == nullptr || Kg == nullptr ||
      Vg == nullptr)
    return WF_ERR_NULL;
  if (!aligned16(K) || !aligned16(V) || !aligned16(Kp) || !aligned16(Vp) || !aligned16(Kg) ||
      !aligned16(Vg) || (AL && !aligned16(AL)))
    return WF_ERR_ALIGNMENT;
  return cuda_status(wf::launch_cache_init(ld, K, V, Kp, Vp, Kg, Vg, AL,
                                           static_cast<cudaStream_t>(stream)));
}

int wf_cache_update(const wf_dims* dims, const void* K, const void* V, void* Kg, void* Vg,
                    void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (K == nullptr || V == nullptr || Kg == nullptr || Vg == nullptr) return WF_ERR_NULL;
  if (!aligned16(K) || !aligned16(V) || !aligned16(Kg) || !aligned16(Vg)) return WF_ERR_ALIGNMENT;
  return cuda_status(
      wf::launch_cache_update(ld, K, V, Kg, Vg, static_cast<cudaStream_t>(stream)));
}

int wf_cache_scatter(const wf_dims* dims, const void* K, const void* V,
                     const int32_t* positions, int32_t n_rows, void* Kp, void* Vp, void* Kg,
                     void* Vg, float* AL, void* workspace, size_t workspace_bytes,
                     void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (n_rows < 0) return WF_ERR_SHAPE;
  if (n_rows == 0) return WF_OK;
  if (K == nullptr || V == nullptr || positions == nullptr || Kp == nullptr || Vp == nullptr ||
      Kg == nullptr || Vg == nullptr)
    return WF_ERR_NULL;
  if (!aligned16(K) || !aligned16(V) || !aligned16(Kp) || !aligned16(Vp) || !aligned16(Kg) ||
      !aligned16(Vg) || (AL && !aligned16(AL)) || (workspace && !aligned16(workspace)) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u) != 0)
    return WF_ERR_ALIGNMENT;
  if (workspace != nullptr && workspace_bytes < kHeaderBytes) return WF_ERR_WORKSPACE;
  return cuda_status(wf::launch_cache_scatter(
      ld, K, V, positions, n_rows, Kp, Vp, Kg, Vg, AL,
      workspace ? status_word(workspace) : nullptr, static_cast<cudaStream_t>(stream)));
}

int wf_score_topk(const wf_dims* dims, const void* Q, const float* AL, int32_t k_L,
                  int32_t* idx_L, float* scores_L, void* workspace, size_t workspace_bytes,
                  void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (Q == nullptr || AL == nullptr || idx_L == nullptr || workspace == nullptr)
    return WF_ERR_NULL;
  if (!aligned16(Q) || !aligned16(AL) || !aligned16(idx_L) || !aligned16(workspace) ||
      (scores_L && !aligned16(scores_L)))
    return WF_ERR_ALIGNMENT;
  if (k_L < 1 || k_L > (ld.n_prompt >> ld.levels)) return WF_ERR_SHAPE;
  const Layout L = layout(ld, nullptr, nullptr);
  if (workspace_bytes < L.total) return WF_ERR_WORKSPACE;
  wf::PathPlan plan;
  if (!wf::plan_path(ld, wf::kPhaseScore | wf::kPhaseCachedAl, nullptr, k_L, 0,
                     wf::device_sm_count(), &plan))
    return WF_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  wf::PathArgs a = {};
  a.q = Q;
  a.al = AL;  // the score phase forms the coarse logits itself
  a.idx_l_out = idx_L;
  a.scores_out = scores_L;
  a.status = status_word(workspace);
  a.k_l = k_L;
  return cuda_status(wf::launch_path(ld, plan, a, s));
}

int wf_recursive_filter(const wf_dims* dims, const void* Q, const void* Kp, const int32_t* idx_L,
                        const int32_t* k_per_level, int32_t* idx, void* workspace,
                        size_t workspace_bytes, void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (Q == nullptr || Kp == nullptr || idx_L == nullptr || idx == nullptr ||
      workspace == nullptr)
    return WF_ERR_NULL;
  if (!aligned16(Q) || !aligned16(Kp) || !aligned16(idx_L) || !aligned16(idx) ||
      !aligned16(workspace))
    return WF_ERR_ALIGNMENT;
  st = check_k(ld, k_per_level);
  if (st != WF_OK) return st;
  wf::PathPlan plan;
  if (!wf::plan_path(ld, wf::kPhaseFilter, k_per_level, k_per_level[ld.levels], k_per_level[0],
                     wf::device_sm_count(), &plan))
    return WF_ERR_UNSUPPORTED;
  const Layout L = layout(ld, k_per_level, &plan);
  if (workspace_bytes < L.total) return WF_ERR_WORKSPACE;
  wf::PathArgs a = {};
  a.q = Q;
  a.kp = Kp;
  a.idx_l_in = idx_L;
  a.idx_out = idx;
  a.status = status_word(workspace);
  a.t_ws = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.t);
  a.k = k_per_level;
  a.k_l = k_per_level[ld.levels];
  a.budget = k_per_level[0];
  return cuda_status(wf::launch_path(ld, plan, a, static_cast<cudaStream_t>(stream)));
}

int wf_sparse_gather_attn(const wf_dims* dims, const void* Q, const void* Kp, const void* Vp,
                          const void* Kg, const void* Vg, const int32_t* idx, int32_t budget,
                          float* O, float* lse, void* workspace, size_t workspace_bytes,
                          void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (Q == nullptr || Kp == nullptr || Vp == nullptr || Kg == nullptr || Vg == nullptr ||
      O == nullptr || workspace == nullptr || (budget > 0 && idx == nullptr))
    return WF_ERR_NULL;
  if (!aligned16(Q) || !aligned16(Kp) || !aligned16(Vp) || !aligned16(Kg) || !aligned16(Vg) ||
      !aligned16(O) || !aligned16(workspace) || (idx && !aligned16(idx)) ||
      (lse && !aligned16(lse)))
    return WF_ERR_ALIGNMENT;
  if (budget < 0) return WF_ERR_SHAPE;
  if (workspace_bytes < kHeaderBytes) return WF_ERR_WORKSPACE;
  wf::PathPlan plan;
  if (!wf::plan_path(ld, wf::kPhaseAttend, nullptr, 0, budget, wf::device_sm_count(), &plan))
    return WF_ERR_UNSUPPORTED;
  wf::PathArgs a = {};
  a.q = Q;
  a.kp = Kp;
  a.vp = Vp;
  a.kg = Kg;
  a.vg = Vg;
  a.idx_in = idx;
  a.o = O;
  a.lse = lse;
  a.status = status_word(workspace);
  a.budget = budget;
  return cuda_status(wf::launch_path(ld, plan, a, static_cast<cudaStream_t>(stream)));
}

int wf_step(const wf_dims* dims, const void* Q, const void* Kp, const void* Vp, const void* Kg,
            const void* Vg, const int32_t* k_per_level, float* O, float* lse, int32_t* idx_out,
            void* workspace, size_t workspace_bytes, void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (Q == nullptr || Kp == nullptr || Vp == nullptr || Kg == nullptr || Vg == nullptr ||
      O == nullptr || workspace == nullptr)
    return WF_ERR_NULL;
  if (!aligned16(Q) || !aligned16(Kp) || !aligned16(Vp) || !aligned16(Kg) || !aligned16(Vg) ||
      !aligned16(O) || !aligned16(workspace) || (lse && !aligned16(lse)) ||
      (idx_out && !aligned16(idx_out)))
    return WF_ERR_ALIGNMENT;
  st = check_k(ld, k_per_level);
  if (st != WF_OK) return st;
  const int budget = k_per_level[0];
  wf::PathPlan plan;
  bool from_al = false;
  if (!step_plan(ld, k_per_level, &plan, &from_al)) return WF_ERR_UNSUPPORTED;
  const Layout L = layout(ld, k_per_level, &plan);
  if (workspace_bytes < L.total) return WF_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  float* zl = reinterpret_cast<float*>(ws + L.zl);
  float* al = reinterpret_cast<float*>(ws + L.al);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Step 1 runs inside the path kernel when the plan fuses it; otherwise a
  // separate streaming launch writes A_L (and, when the path kernel does not
  // form them itself, each coarse position's logits against the queries).
  if (!plan.fuse_dwt) {
    const cudaError_t e = wf::launch_dwt_lowpass(ld, Kp, al, from_al ? nullptr : Q,
                                                 from_al ? nullptr : zl, ld.levels,
                                                 status_word(workspace), s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  wf::PathArgs a = {};
  a.q = Q;
  a.kp = Kp;
  a.vp = Vp;
  a.kg = Kg;
  a.vg = Vg;
  a.zl = plan.fuse_dwt || from_al ? nullptr : zl;
  a.al = from_al ? al : nullptr;
  a.idx_out = idx_out;
  a.o = O;
  a.lse = lse;
  a.status = status_word(workspace);
  a.t_ws = reinterpret_cast<float*>(ws + L.t);
  a.k = k_per_level;
  a.k_l = k_per_level[ld.levels];
  a.budget = budget;
  return cuda_status(wf::launch_path(ld, plan, a, s));
}

int wf_step_cached_al(const wf_dims* dims, const void* Q, const void* Kp, const void* Vp,
                      const void* Kg, const void* Vg, const float* AL,
                      const int32_t* k_per_level, float* O, float* lse, int32_t* idx_out,
                      void* workspace, size_t workspace_bytes, void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (Q == nullptr || Kp == nullptr || Vp == nullptr || Kg == nullptr || Vg == nullptr ||
      AL == nullptr || O == nullptr || workspace == nullptr)
    return WF_ERR_NULL;
  if (!aligned16(Q) || !aligned16(Kp) || !aligned16(Vp) || !aligned16(Kg) || !aligned16(Vg) ||
      !aligned16(AL) || !aligned16(O) || !aligned16(workspace) || (lse && !aligned16(lse)) ||
      (idx_out && !aligned16(idx_out)))
    return WF_ERR_ALIGNMENT;
  st = check_k(ld, k_per_level);
  if (st != WF_OK) return st;
  const int budget = k_per_level[0];
  wf::PathPlan plan;
  if (!wf::plan_path(ld, wf::kPhaseAll | wf::kPhaseCachedAl, k_per_level, k_per_level[ld.levels], budget,
                     wf::device_sm_count(), &plan))
    return WF_ERR_UNSUPPORTED;
  const Layout L = layout(ld, k_per_level, &plan);
  if (workspace_bytes < L.total) return WF_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  wf::PathArgs a = {};
  a.q = Q;
  a.kp = Kp;
  a.vp = Vp;
  a.kg = Kg;
  a.vg = Vg;
  a.al = AL;  // one launch: the score phase forms the coarse logits from the cached A_L
  a.idx_out = idx_out;
  a.o = O;
  a.lse = lse;
  a.status = status_word(workspace);
  a.t_ws = reinterpret_cast<float*>(ws + L.t);
  a.k = k_per_level;
  a.k_l = k_per_level[ld.levels];
  a.budget = budget;
  return cuda_status(wf::launch_path(ld, plan, a, s));
}

int wf_decode_step_host(const wf_dims* dims, const void* h_Q, const void* h_K, const void* h_V,
                        const int32_t* k_per_level, float* h_O, void* d_Q, void* d_K,
                        void* d_V, const void* Kp, const void* Vp, void* Kg, void* Vg,
                        const float* AL, float* d_O, void* workspace, size_t workspace_bytes,
                        void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (h_Q == nullptr || h_K == nullptr || h_V == nullptr || h_O == nullptr ||
      d_Q == nullptr || d_K == nullptr || d_V == nullptr || Kp == nullptr || Vp == nullptr ||
      Kg == nullptr || Vg == nullptr || AL == nullptr || d_O == nullptr || workspace == nullptr)
    return WF_ERR_NULL;
  if (!aligned16(d_Q) || !aligned16(d_K) || !aligned16(d_V) || !aligned16(Kp) ||
      !aligned16(Vp) || !aligned16(Kg) || !aligned16(Vg) || !aligned16(AL) || !aligned16(d_O) ||
      !aligned16(workspace))
    return WF_ERR_ALIGNMENT;
  st = check_k(ld, k_per_level);
  if (st != WF_OK) return st;
  // Everything the cached step checks, before any copy is enqueued.
  wf::PathPlan plan;
  if (!wf::plan_path(ld, wf::kPhaseAll, k_per_level, k_per_level[ld.levels], k_per_level[0],
                     wf::device_sm_count(), &plan))
    return WF_ERR_UNSUPPORTED;
  if (workspace_bytes < layout(ld, k_per_level, &plan).total) return WF_ERR_WORKSPACE;
  const size_t gen_bytes =
      static_cast<size_t>(ld.units) * ld.n_gen * ld.head_dim * elem_bytes(ld.dtype);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Q, K and V laid out back to back on both sides travel as one copy.
  const auto at = [gen_bytes](const void* p, int i) {
    return static_cast<const char*>(p) + i * gen_bytes;
  };
  const bool packed = h_K == at(h_Q, 1) && h_V == at(h_Q, 2) && d_K == at(d_Q, 1) &&
                      d_V == at(d_Q, 2);
  cudaError_t ce;
  if (packed) {
    ce = cudaMemcpyAsync(d_Q, h_Q, 3 * gen_bytes, cudaMemcpyHostToDevice, s);
  } else {
    ce = cudaMemcpyAsync(d_Q, h_Q, gen_bytes, cudaMemcpyHostToDevice, s);
    if (ce == cudaSuccess) ce = cudaMemcpyAsync(d_K, h_K, gen_bytes, cudaMemcpyHostToDevice, s);
    if (ce == cudaSuccess) ce = cudaMemcpyAsync(d_V, h_V, gen_bytes, cudaMemcpyHostToDevice, s);
  }
  if (ce == cudaSuccess) ce = wf::launch_cache_update(ld, d_K, d_V, Kg, Vg, s);
  if (ce != cudaSuccess) return cuda_status(ce);
  st = wf_step_cached_al(dims, d_Q, Kp, Vp, Kg, Vg, AL, k_per_level, d_O, nullptr, nullptr,
                         workspace, workspace_bytes, stream);
  if (st != WF_OK) return st;
  return cuda_status(cudaMemcpyAsync(h_O, d_O, sizeof(float) * ld.units * ld.n_gen * ld.head_dim,
                                     cudaMemcpyDeviceToHost, s));
}

int wf_daubechies_lowpass(int32_t n_moments, double* taps_out) {
  if (taps_out == nullptr) return WF_ERR_NULL;
  if (n_moments < 1 || n_moments > 8) return WF_ERR_UNSUPPORTED;
  wf::daubechies_lowpass(n_moments, taps_out);
  return WF_OK;
}

int wf_basis_workspace_bytes(const wf_dims* dims, int32_t taps, const int32_t* k_per_level,
                             size_t* bytes) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (bytes == nullptr) return WF_ERR_NULL;
  if (taps < 2 || taps > 16 || taps % 2 != 0) return WF_ERR_UNSUPPORTED;
  st = check_k(ld, k_per_level);
  if (st != WF_OK) return st;
  wf::PathPlan plan;
  *bytes = basis_coarse_route(ld, taps, k_per_level, &plan) ? layout(ld, k_per_level, &plan).total
                                                            : basis_layout(ld, k_per_level).total;
  return WF_OK;
}

int wf_dwt_lowpass_basis(const wf_dims* dims, const double* lowpass, int32_t taps,
                         const void* Kp, float* A_all, void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  wf::BasisTaps t;
  st = check_taps(lowpass, taps, &t);
  if (st != WF_OK) return st;
  if (Kp == nullptr || A_all == nullptr) return WF_ERR_NULL;
  if (!aligned16(Kp) || !aligned16(A_all)) return WF_ERR_ALIGNMENT;
  return cuda_status(
      wf::launch_basis_pyramid(ld, Kp, A_all, t, static_cast<cudaStream_t>(stream)));
}

int wf_step_basis(const wf_dims* dims, const double* lowpass, int32_t taps, const void* Q,
                  const void* Kp, const void* Vp, const void* Kg, const void* Vg,
                  const int32_t* k_per_level, float* O, float* lse, int32_t* idx_out,
                  void* workspace, size_t workspace_bytes, void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  wf::BasisTaps t;
  st = check_taps(lowpass, taps, &t);
  if (st != WF_OK) return st;
  if (Q == nullptr || Kp == nullptr || Vp == nullptr || Kg == nullptr || Vg == nullptr ||
      O == nullptr || workspace == nullptr)
    return WF_ERR_NULL;
  if (!aligned16(Q) || !aligned16(Kp) || !aligned16(Vp) || !aligned16(Kg) || !aligned16(Vg) ||
      !aligned16(O) || !aligned16(workspace) || (lse && !aligned16(lse)) ||
      (idx_out && !aligned16(idx_out)))
    return WF_ERR_ALIGNMENT;
  st = check_k(ld, k_per_level);
  if (st != WF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    wf::PathPlan plan;
    if (basis_coarse_route(ld, taps, k_per_level, &plan)) {
      // Two launches: the basis's level-L logits, then steps 2-5 of the path
      // kernel on them (the tokens under the coarse survivors are scored on
      // their own keys, independent of the basis).
      const Layout L = layout(ld, k_per_level, &plan);
      if (workspace_bytes < L.total) return WF_ERR_WORKSPACE;
      char* ws = static_cast<char*>(workspace);
      float* zl = reinterpret_cast<float*>(ws + L.zl);
      static thread_local wf::BasisCoarseParams cp;  // 16 KB of filter taps: off the stack
      cp.q = Q;
      cp.kp = Kp;
      cp.zl = zl;
      cp.n_prompt = ld.n_prompt;
      cp.n_gen = ld.n_gen;
      cp.levels = ld.levels;
      cp.gz = wf::coarse_logit_pitch(ld.n_gen);
      cp.zscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(ld.head_dim)));
      cp.w_len = wf::basis_cascade(lowpass, taps, ld.levels, cp.w);
      if (cp.w_len < 1) return WF_ERR_UNSUPPORTED;
      cudaError_t ce = wf::launch_basis_coarse(ld, cp, s);
      if (ce != cudaSuccess) return cuda_status(ce);
      wf::PathArgs a = {};
      a.q = Q;
      a.kp = Kp;
      a.vp = Vp;
      a.kg = Kg;
      a.vg = Vg;
      a.zl = zl;
      a.idx_out = idx_out;
      a.o = O;
      a.lse = lse;
      a.status = status_word(workspace);
      a.t_ws = reinterpret_cast<float*>(ws + L.t);
      a.k = k_per_level;
      a.k_l = k_per_level[ld.levels];
      a.budget = k_per_level[0];
      return cuda_status(wf::launch_path(ld, plan, a, s));
    }
  }
  const BasisLayout L = basis_layout(ld, k_per_level);
  if (workspace_bytes < L.total) return WF_ERR_WORKSPACE;
  wf::PathPlan plan;  // steps 4-5 must be plannable before anything is enqueued
  if (!wf::plan_path(ld, wf::kPhaseAttend, nullptr, 0, k_per_level[0], wf::device_sm_count(),
                     &plan))
    return WF_ERR_UNSUPPORTED;
  char* ws = static_cast<char*>(workspace);
  float* a_all = reinterpret_cast<float*>(ws + L.a_all);
  cudaError_t ce = wf::launch_basis_pyramid(ld, Kp, a_all, t, s);
  if (ce != cudaSuccess) return cuda_status(ce);
  wf::BasisFilterParams p = {};
  p.q = Q;
  p.kp = Kp;
  p.a_all = a_all;
  int64_t off = 0;
  for (int j = 1; j <= ld.levels; ++j) {
    p.level_off[j] = off;
    off += ld.units * static_cast<int64_t>(ld.n_prompt >> j) * ld.head_dim;
  }
  p.cand = reinterpret_cast<int32_t*>(ws + L.cand);
  p.keys = reinterpret_cast<uint32_t*>(ws + L.keys);
  p.z = reinterpret_cast<float*>(ws + L.z);
  int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(ws + L.idx);
  p.idx = idx;
  p.units = ld.units;
  p.cap = L.cap;
  p.n_prompt = ld.n_prompt;
  p.n_gen = ld.n_gen;
  p.levels = ld.levels;
  for (int j = 0; j <= ld.levels; ++j) p.k[j] = k_per_level[j];
  p.qscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(ld.head_dim)));
  ce = wf::launch_basis_filter(ld, p, s);
  if (ce != cudaSuccess) return cuda_status(ce);
  return wf_sparse_gather_attn(dims, Q, Kp, Vp, Kg, Vg, idx, k_per_level[0], O, lse, workspace,
                               workspace_bytes, stream);
}

int wf_step_host(const wf_dims* dims, const void* h_Q, const void* h_Kp, const void* h_Vp,
                 const void* h_Kg, const void* h_Vg, const int32_t* k_per_level, float* h_O,
                 float* h_lse, void* d_Q, void* d_Kp, void* d_Vp, void* d_Kg, void* d_Vg,
                 float* d_O, float* d_lse, void* workspace, size_t workspace_bytes,
                 void* stream) {
  LaunchDims ld;
  int st = check_dims(dims, &ld);
  if (st != WF_OK) return st;
  if (h_Q == nullptr || h_Kp == nullptr || h_Vp == nullptr || h_Kg == nullptr ||
      h_Vg == nullptr || h_O == nullptr || d_Q == nullptr || d_Kp == nullptr ||
      d_Vp == nullptr || d_Kg == nullptr || d_Vg == nullptr || d_O == nullptr)
    return WF_ERR_NULL;
  st = check_k(ld, k_per_level);
  if (st != WF_OK) return st;
  const size_t e = elem_bytes(ld.dtype);
  const size_t gen_bytes = static_cast<size_t>(ld.units) * ld.n_gen * ld.head_dim * e;
  const size_t prompt_bytes = static_cast<size_t>(ld.units) * ld.n_prompt * ld.head_dim * e;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Validate the device side before any copy is enqueued.
  size_t need = 0;
  st = wf_workspace_bytes(dims, k_per_level, &need);
  if (st != WF_OK) return st;
  if (workspace == nullptr) return WF_ERR_NULL;
  if (workspace_bytes < need) return WF_ERR_WORKSPACE;
  cudaError_t ce = cudaMemcpyAsync(d_Q, h_Q, gen_bytes, cudaMemcpyHostToDevice, s);
  if (ce == cudaSuccess) ce = cudaMemcpyAsync(d_Kp, h_Kp, prompt_bytes, cudaMemcpyHostToDevice, s);
  if (ce == cudaSuccess) ce = cudaMemcpyAsync(d_Vp, h_Vp, prompt_bytes, cudaMemcpyHostToDevice, s);
  if (ce == cudaSuccess) ce = cudaMemcpyAsync(d_Kg, h_Kg, gen_bytes, cudaMemcpyHostToDevice, s);
  if (ce == cudaSuccess) ce = cudaMemcpyAsync(d_Vg, h_Vg, gen_bytes, cudaMemcpyHostToDevice, s);
  if (ce != cudaSuccess) return WF_ERR_CUDA;
  const bool want_lse = h_lse != nullptr && d_lse != nullptr;
  st = wf_step(dims, d_Q, d_Kp, d_Vp, d_Kg, d_Vg, k_per_level, d_O, want_lse ? d_lse : nullptr,
               nullptr, workspace, workspace_bytes, stream);
  if (st != WF_OK) return st;
  const size_t o_bytes = sizeof(float) * ld.units * ld.n_gen * ld.head_dim;
  ce = cudaMemcpyAsync(h_O, d_O, o_bytes, cudaMemcpyDeviceToHost, s);
  if (ce == cudaSuccess && want_lse)
    ce = cudaMemcpyAsync(h_lse, d_lse, sizeof(float) * ld.units * ld.n_gen,
                         cudaMemcpyDeviceToHost, s);
  return cuda_status(ce);
}

}  // extern "C"
