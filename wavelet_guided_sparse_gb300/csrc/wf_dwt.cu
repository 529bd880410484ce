// Step 1: multi-level orthonormal Haar low-pass along the token axis.
//
// WaveFilter (arXiv 2606.00724) §2.2 eq. (5) iterated into the pyramid of
// §2.2 and applied to the cached prompt keys in §3.1.  With g = [1/√2, 1/√2]
// on pairs (2n, 2n+1) the level-L approximation is a scaled span sum:
//   A_L[p] = 2^(-L/2) · Σ_{n in [p·2^L, (p+1)·2^L)} Kp[n].
//
// Design (HBM-bound, one read of Kp): spans of consecutive units are
// contiguous in memory, so the whole input is one byte stream.  A persistent
// grid of one CTA per SM splits the spans evenly; each CTA streams its
// contiguous byte range through a ring of three 64 KB shared-memory stages
// filled by single bulk copies (TMA engine, mbarrier completion), so 128-192
// KB per SM are in flight independent of register pressure.  Threads reduce
// the staged rows in fp32: for spans of up to 16 rows one thread owns one
// (span, 16-byte column chunk) pair; longer spans are summed in 16-row blocks
// whose partials are combined in a fixed order, with a running sum carried
// across stages for spans longer than a stage; finished rows are stored as
// fp32 A_L.  For the step, the CTA then turns its rows into coarse logits
// Q·A_L/√d against their units' queries (the first quantity step 2 scores)
// while they are still in L2.
#include <algorithm>
#include <cmath>

#include "wf_common.cuh"
#include "wf_internal.h"
#include "wf_mma.cuh"

namespace wf {

namespace {

constexpr int kStageBytes = 64 * 1024;
constexpr int kStages = 3;

template <typename T, int D>
struct DwtSmem {
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(T));
  static constexpr int kRows = kStageBytes / kRowBytes;  // rows per stage
  static constexpr int V = Elem<T>::kPer16B;
  static constexpr int C = D / V;                        // 16-byte chunks per row
  static constexpr size_t kBars = 0;
  static constexpr size_t kRing = 128;
  static constexpr size_t kPart = kRing + static_cast<size_t>(kStages) * kStageBytes;
  static constexpr size_t kCarry = kPart + sizeof(float) * (kRows / 16) * C * V;
  static constexpr size_t kTotal = kCarry + sizeof(float) * C * V;
};

template <typename T>
__device__ __forceinline__ void add_chunk(const unsigned char* p, float* acc) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  float f[Elem<T>::kPer16B];
  widen16(v, static_cast<const T*>(nullptr), f);
#pragma unroll
  for (int i = 0; i < Elem<T>::kPer16B; ++i) acc[i] += f[i];
}

// Stores V channels of one finished A_L row (fp32, [U, P, D]).
template <int D, int V>
__device__ __forceinline__ void store_row(const float* acc, float scale, int64_t span, int c,
                                          float* out) {
  float4* o = reinterpret_cast<float4*>(out + span * D + c * V);
#pragma unroll
  for (int v = 0; v < V; v += 4)
    o[v / 4] = make_float4(acc[v] * scale, acc[v + 1] * scale, acc[v + 2] * scale, acc[v + 3] * scale);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) dwt_stream_kernel(const T* __restrict__ kp,
                                                                 float* __restrict__ out,
                                                                 const T* __restrict__ q,
                                                                 float* __restrict__ zl, int G,
                                                                 int GZ, float zscale,
                                                                 int64_t n_spans,
                                                                 int64_t spans_per_cta,
                                                                 int levels, int64_t P,
                                                                 float scale, int32_t* status,
                                                                 uint32_t inject_polls) {
  extern __shared__ __align__(128) unsigned char smem[];
  using S = DwtSmem<T, D>;
  constexpr int RB = S::kRowBytes, SR = S::kRows, V = S::V, C = S::C;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBars);
  unsigned char* ring = smem + S::kRing;
  float* part = reinterpret_cast<float*>(smem + S::kPart);
  float* carry = reinterpret_cast<float*>(smem + S::kCarry);
  const int tid = threadIdx.x;
  const int64_t s_begin = static_cast<int64_t>(blockIdx.x) * spans_per_cta;
  const int64_t s_end = min(n_spans, s_begin + spans_per_cta);
  if (s_begin >= s_end) return;  // whole CTA, before any barrier
  const int span_rows = 1 << levels;
  const int64_t rows_total = (s_end - s_begin) << levels;
  const int64_t n_stages = (rows_total + SR - 1) / SR;
  const unsigned char* src = reinterpret_cast<const unsigned char*>(kp + (s_begin << levels) * D);
  // Fault injection (tests of the bounded waits): stage 0 of CTA 0 is never
  // issued and its wait gives up after inject_polls polls.
  const bool inject = inject_polls != 0 && blockIdx.x == 0;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int64_t st) {  // thread 0 only
    const int64_t rows = min(static_cast<int64_t>(SR), rows_total - st * SR);
    const uint32_t bytes = static_cast<uint32_t>(rows * RB);
    uint64_t* bar = &bars[st % kStages];
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(ring + (st % kStages) * kStageBytes, src + st * static_cast<int64_t>(SR) * RB, bytes,
             bar);
  };
  // Stages issued so far (every thread keeps the same count).  After a wait
  // gives up no further stage is issued, but every stage already issued is
  // still waited for (bounded), so no copy is in flight when the CTA exits.
  int64_t issued = min(static_cast<int64_t>(kStages), n_stages);
  if (tid == 0)
    for (int64_t st = 0; st < issued; ++st)
      if (!(inject && st == 0)) issue(st);
  bool aborted = false;
  for (int64_t st = 0; st < issued; ++st) {
    const bool ok = mbar_wait_bounded(&bars[st % kStages], static_cast<uint32_t>((st / kStages) & 1),
                                      status, inject && st == 0 ? inject_polls : kWaitPolls);
    if (__syncthreads_or(!ok)) aborted = true;
    const unsigned char* buf = ring + (st % kStages) * kStageBytes;
    const int rows_in = static_cast<int>(min(static_cast<int64_t>(SR), rows_total - st * SR));
    const int64_t first_row = st * SR;
    if (span_rows <= 16) {
      // One thread per (span, chunk) of this stage; a stage holds whole spans.
      // Whole warps iterate together (the coarse logits are warp-collective).
      const int spans_in = rows_in >> levels;
      const int64_t span0 = first_row >> levels;
      for (int base = 0; base < spans_in * C; base += kThreads) {
        const int item = base + tid;
        const bool act = item < spans_in * C;
        const int sl = item / C, c = item % C;
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.f;
        if (act) {
          const unsigned char* p = buf + (sl << levels) * RB + c * 16;
#pragma unroll
          for (int r = 0; r < 16; ++r)
            if (r < span_rows) add_chunk<T>(p + r * RB, acc);
        }
        if (act) store_row<D, V>(acc, scale, s_begin + span0 + sl, c, out);
      }
    } else {
      // 16-row block partials, then per-span combination in block order.
      const int nblk = rows_in / 16;
      for (int item = tid; item < nblk * C; item += kThreads) {
        const int b = item / C, c = item % C;
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.f;
        const unsigned char* p = buf + (b * 16) * RB + c * 16;
#pragma unroll 4
        for (int r = 0; r < 16; ++r) add_chunk<T>(p + r * RB, acc);
#pragma unroll
        for (int v = 0; v < V; ++v) part[(b * C + c) * V + v] = acc[v];
      }
      __syncthreads();
      const int64_t sp0 = first_row >> levels;
      const int64_t sp1 = (first_row + rows_in - 1) >> levels;
      const int nsp = static_cast<int>(sp1 - sp0 + 1);
      for (int base = 0; base < nsp * C; base += kThreads) {  // whole warps together
        const int item = base + tid;
        const bool in = item < nsp * C;
        const int sl = item / C, c = item % C;
        const int64_t span = sp0 + sl;
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.f;
        bool done = false;
        if (in) {
          const int64_t r_lo = max(span << levels, first_row);
          const int64_t r_hi = min((span + 1) << levels, first_row + rows_in);
          const bool carried = (span << levels) < first_row;
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] = carried ? carry[c * V + v] : 0.f;
          for (int b = static_cast<int>((r_lo - first_row) / 16); b < (r_hi - first_row) / 16; ++b)
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] += part[(b * C + c) * V + v];
          done = ((span + 1) << levels) <= first_row + rows_in;
          if (!done) {
#pragma unroll
            for (int v = 0; v < V; ++v) carry[c * V + v] = acc[v];
          }
        }
        if (done) store_row<D, V>(acc, scale, s_begin + span, c, out);
      }
    }
    __syncthreads();  // stage consumed (and carry / partials settled)
    if (st + kStages < n_stages && !aborted) {
      if (tid == 0) {
        fence_proxy_async();
        issue(st + kStages);
      }
      ++issued;
    }
  }
  // With queries: the coarse logits of this CTA's rows, from the A_L rows it
  // has just written (L2), by all warps.
  if (zl != nullptr) {
    __syncthreads();
    coarse_logits_range<T, D>(out, q, zl, s_begin, s_end, P, G, GZ, zscale, tid >> 5, kWarps);
  }
}

template <typename T, int D>
cudaError_t launch_typed(const LaunchDims& ld, const void* kp, float* out, const void* q,
                         float* zl, int levels, int32_t* status, cudaStream_t stream) {
  const cudaError_t e = ensure_max_smem<dwt_stream_kernel<T, D>>();
  if (e != cudaSuccess) return e;
  const int64_t n_spans = ld.units * (ld.n_prompt >> levels);
  const int64_t grid = std::min<int64_t>(device_sm_count(), n_spans);
  const int64_t per = (n_spans + grid - 1) / grid;
  const int64_t blocks = (n_spans + per - 1) / per;
  const float scale = static_cast<float>(std::pow(2.0, -0.5 * levels));  // 2^(-L/2)
  const float zscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  dwt_stream_kernel<T, D><<<static_cast<unsigned>(blocks), kThreads, DwtSmem<T, D>::kTotal,
                            stream>>>(static_cast<const T*>(kp), out, static_cast<const T*>(q), zl,
                                      ld.n_gen, coarse_logit_pitch(ld.n_gen), zscale, n_spans, per,
                                      levels, static_cast<int64_t>(ld.n_prompt >> levels), scale,
                                      status, consume_wait_injection());
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dwt_lowpass(const LaunchDims& ld, const void* kp, float* out, const void* q,
                               float* zl, int levels, int32_t* status, cudaStream_t stream) {
  if (ld.dtype == WF_BF16) {
    if (ld.head_dim == 128)
      return launch_typed<__nv_bfloat16, 128>(ld, kp, out, q, zl, levels, status, stream);
    return launch_typed<__nv_bfloat16, 64>(ld, kp, out, q, zl, levels, status, stream);
  }
  if (ld.head_dim == 128) return launch_typed<float, 128>(ld, kp, out, q, zl, levels, status, stream);
  return launch_typed<float, 64>(ld, kp, out, q, zl, levels, status, stream);
}

}  // namespace wf
