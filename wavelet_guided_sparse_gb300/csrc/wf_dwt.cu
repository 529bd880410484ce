// Step 1: multi-level orthonormal Haar low-pass along the token axis.
//
// WaveFilter (arXiv 2606.00724) §2.2 eq. (5) iterated into the pyramid of
// §2.2 and applied to the cached prompt keys in §3.1.  With g = [1/√2, 1/√2]
// on pairs (2n, 2n+1) the level-L approximation is a scaled span sum:
//   A_L[p] = 2^(-L/2) · Σ_{n in [p·2^L, (p+1)·2^L)} Kp[n].
//
// Design (HBM-bound, one read of Kp): every thread owns one 16-byte column
// chunk of one span (8 bf16 or 4 fp32 channels) and walks the span's 2^L
// rows with up to 16 independent 16-byte loads in flight, accumulating in
// fp32 registers.  Adjacent lanes own adjacent chunks of the same row, so a
// warp instruction reads whole 256-byte rows (d = 128, bf16).  Spans are
// contiguous in memory, so a unit's Kp is streamed front to back exactly once.
#include <cmath>

#include "wf_common.cuh"
#include "wf_internal.h"

namespace wf {

// UNROLL (even, >= 2) rows per group; 2^levels must be a multiple of UNROLL.
template <typename T, int D, int UNROLL>
__global__ void __launch_bounds__(kThreads) dwt_lowpass_kernel(const T* __restrict__ kp,
                                                               float* __restrict__ out,
                                                               int64_t n_spans, int levels,
                                                               float scale) {
  constexpr int V = Elem<T>::kPer16B;  // channels per 16-byte chunk
  constexpr int C = D / V;             // chunks per row
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t span = item / C;
  const int chunk = static_cast<int>(item % C);
  if (span >= n_spans) return;
  const int rows = 1 << levels;
  const T* src = kp + (span << levels) * D + chunk * V;
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
#pragma unroll 1
  for (int r0 = 0; r0 < rows; r0 += UNROLL) {
    uint4 raw[UNROLL];
#pragma unroll
    for (int i = 0; i < UNROLL; ++i) raw[i] = ldg16_stream(src + static_cast<int64_t>(r0 + i) * D);
    // The arithmetic below consumes these (ordered) pass-through values, so
    // all UNROLL loads are issued before the first add waits on memory.
#pragma unroll
    for (int i = 0; i < UNROLL; ++i)
      asm volatile("" : "+r"(raw[i].x), "+r"(raw[i].y), "+r"(raw[i].z), "+r"(raw[i].w));
    // Pairwise within the group keeps the fp32 error of long spans small.
#pragma unroll
    for (int i = 0; i < UNROLL; i += 2) {
      float a[V], b[V];
      widen16(raw[i], static_cast<const T*>(nullptr), a);
      widen16(raw[i + 1], static_cast<const T*>(nullptr), b);
#pragma unroll
      for (int v = 0; v < V; ++v) acc[v] += a[v] + b[v];
    }
  }
  float4* dst = reinterpret_cast<float4*>(out + span * D + chunk * V);
#pragma unroll
  for (int v = 0; v < V; v += 4)
    dst[v / 4] = make_float4(acc[v] * scale, acc[v + 1] * scale, acc[v + 2] * scale,
                             acc[v + 3] * scale);
}

template <typename T, int D>
static cudaError_t launch_dwt_typed(const void* kp, float* out, int64_t units, int n_prompt,
                                    int levels, cudaStream_t stream) {
  constexpr int C = D / Elem<T>::kPer16B;
  const int64_t n_spans = units * (n_prompt >> levels);
  const int64_t items = n_spans * C;
  const int64_t blocks = (items + kThreads - 1) / kThreads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const float scale = static_cast<float>(std::pow(2.0, -0.5 * levels));  // 2^(-L/2)
  const T* k = static_cast<const T*>(kp);
  const dim3 grid(static_cast<unsigned>(blocks));
  switch (levels) {
    case 1: dwt_lowpass_kernel<T, D, 2><<<grid, kThreads, 0, stream>>>(k, out, n_spans, levels, scale); break;
    case 2: dwt_lowpass_kernel<T, D, 4><<<grid, kThreads, 0, stream>>>(k, out, n_spans, levels, scale); break;
    case 3: dwt_lowpass_kernel<T, D, 8><<<grid, kThreads, 0, stream>>>(k, out, n_spans, levels, scale); break;
    default: dwt_lowpass_kernel<T, D, 16><<<grid, kThreads, 0, stream>>>(k, out, n_spans, levels, scale); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_dwt_lowpass(const LaunchDims& ld, const void* kp, float* out, int levels,
                               cudaStream_t stream) {
  const int64_t units = ld.units;
  if (ld.dtype == WF_BF16) {
    if (ld.head_dim == 128)
      return launch_dwt_typed<__nv_bfloat16, 128>(kp, out, units, ld.n_prompt, levels, stream);
    return launch_dwt_typed<__nv_bfloat16, 64>(kp, out, units, ld.n_prompt, levels, stream);
  }
  if (ld.head_dim == 128)
    return launch_dwt_typed<float, 128>(kp, out, units, ld.n_prompt, levels, stream);
  return launch_dwt_typed<float, 64>(kp, out, units, ld.n_prompt, levels, stream);
}

}  // namespace wf
