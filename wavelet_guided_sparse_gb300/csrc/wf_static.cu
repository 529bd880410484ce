// wf_step_static_scratch: the whole path without a caller-provided workspace.
//
// The scratch that wf_step normally takes from the caller's workspace (the
// status word, the level-L approximation A_L and, for the largest budgets,
// spilled token logits) lives here in one file-scope device array instead,
// so the call needs no device allocation at all.  This serves callers that
// cannot allocate device memory: plugin or enqueue interfaces of inference
// engines that forbid allocation inside the call, and latency-critical
// loops where cudaMalloc's implicit device synchronisation is unacceptable.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "wavefilter.h"
#include "wf_internal.h"

namespace {

// The array is allocated on every device that loads this library and stays
// there until the process exits.
constexpr size_t kStaticScratchBytes = static_cast<size_t>(WF_STATIC_SCRATCH_BYTES);
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch, looked up once per device.  In host
// code the array's name only stands in for the symbol; it is not a device
// address, so it is never passed to a kernel directly.
std::atomic<void*> g_scratch_addr[64];

int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return WF_ERR_CUDA;
  }
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      wf::note_cuda_error(e == cudaSuccess ? cudaErrorInvalidSymbol : e);
      return WF_ERR_CUDA;
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return WF_OK;
}

}  // namespace

extern "C" int wf_step_static_scratch(const wf_dims* dims, const void* Q, const void* Kp,
                                      const void* Vp, const void* Kg, const void* Vg,
                                      const int32_t* k_per_level, float* O, float* lse,
                                      int32_t* idx_out, void* stream) {
  size_t need = 0;
  const int st = wf_workspace_bytes(dims, k_per_level, &need);
  if (st != WF_OK) return st;
  if (need > kStaticScratchBytes) return WF_ERR_WORKSPACE;  // beyond the fixed limit
  void* scratch = nullptr;
  const int sa = scratch_address(&scratch);
  if (sa != WF_OK) return sa;
  // The array keeps the previous call's contents: the status word must start
  // at zero.  (A memset is not an allocation.)
  const cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(int32_t),
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    wf::note_cuda_error(e);
    return WF_ERR_CUDA;
  }
  return wf_step(dims, Q, Kp, Vp, Kg, Vg, k_per_level, O, lse, idx_out, scratch,
                 kStaticScratchBytes, stream);
}
