// KV-cache writes around the filtering path: the cache initialisation of the
// first denoising step (WaveFilter §2.1 eq. (2)) with the level-L Haar
// approximation of the prompt keys (§2.2 eq. (5) pyramid, §3.1) produced in
// the same pass, and the generation-row update of later steps (eq. (4)).
//
// Source: the keys and values the projections produced, token-major
// [batch, n_tok, heads, d] (a token's heads side by side).  Cache:
// head-major [batch, heads, rows, d], the layout every other entry point
// reads.  The write swaps the (token, head) axes at row granularity; a row
// is d·e contiguous bytes on both sides.
//
// Design (HBM-bound: every byte is read once and written once, A_L is an
// extra 1/2^L of the key bytes in fp32): one thread per (tensor, unit,
// coarse span, 16-byte column chunk).  Consecutive threads take consecutive
// chunks of the same span, so each warp-wide load or store covers whole
// 128-512 byte rows.  A thread streams its span's rows in batches of eight
// independent 16-byte loads, stores them to the cache and, for keys, adds
// them in fp32 into 16-row block partials that are combined in block order:
// the summation order of the streaming low-pass kernel, so A_L matches
// wf_dwt_lowpass bit for bit.  Generation rows are one-row items, copied.
// There are no waits and no shared memory; threads never cooperate.
#include <algorithm>
#include <cmath>

#include "wf_common.cuh"
#include "wf_internal.h"

namespace wf {

namespace {

constexpr int kBatchRows = 8;  // independent 16-byte loads in flight per thread

struct CacheParams {
  const unsigned char* k;  // token-major sources
  const unsigned char* v;
  unsigned char* kp;       // head-major caches (prompt part; null when n_prompt == 0)
  unsigned char* vp;
  unsigned char* kg;       // head-major caches (generation part)
  unsigned char* vg;
  float* al;               // nullable
  int64_t units;
  int heads;
  int n_tok;               // source rows per sequence = n_prompt + n_gen
  int n_prompt;
  int n_gen;
  int levels;
  float scale;             // 2^(-L/2)
};

__device__ __forceinline__ uint4 ld_stream(const unsigned char* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_row(unsigned char* p, const uint4& x) {
  *reinterpret_cast<uint4*>(p) = x;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 3) cache_write_kernel(CacheParams p) {
  constexpr int E = static_cast<int>(sizeof(T));
  constexpr int V = Elem<T>::kPer16B;  // elements per 16-byte chunk
  constexpr int C = D / V;             // chunks per row
  constexpr int RB = D * E;            // row bytes
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int span_rows = 1 << p.levels;
  const int64_t P = p.n_prompt >> p.levels;
  const int64_t span_items = p.units * P * C;  // per tensor
  const int64_t gen_items = p.units * p.n_gen * C;
  const int64_t src_row = static_cast<int64_t>(p.heads) * RB;  // token stride of the source

  if (item < 2 * span_items) {
    const bool is_v = item >= span_items;
    const int64_t it = is_v ? item - span_items : item;
    const int c = static_cast<int>(it % C);
    const int64_t sp = it / C;
    const int64_t pos = sp % P;
    const int64_t u = sp / P;
    const int64_t b = u / p.heads, h = u % p.heads;
    const int64_t tok0 = pos << p.levels;
    const unsigned char* src =
        (is_v ? p.v : p.k) + (b * p.n_tok + tok0) * src_row + h * RB + c * 16;
    unsigned char* dst = (is_v ? p.vp : p.kp) + (u * p.n_prompt + tok0) * RB + c * 16;
    float* al = (!is_v && p.al != nullptr) ? p.al + (u * P + pos) * D + c * V : nullptr;
    float acc[V], blk[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = blk[e] = 0.f;
    for (int r0 = 0; r0 < span_rows; r0 += kBatchRows) {
      const int nb = min(kBatchRows, span_rows - r0);
      uint4 x[kBatchRows];
#pragma unroll
      for (int i = 0; i < kBatchRows; ++i)
        if (i < nb) x[i] = ld_stream(src + i * src_row);
#pragma unroll
      for (int i = 0; i < kBatchRows; ++i)
        if (i < nb) st_row(dst + i * RB, x[i]);
      src += kBatchRows * src_row;
      dst += kBatchRows * RB;
      if (al != nullptr) {
#pragma unroll
        for (int i = 0; i < kBatchRows; ++i) {
          if (i < nb) {
            float f[V];
            widen16(x[i], static_cast<const T*>(nullptr), f);
#pragma unroll
            for (int e = 0; e < V; ++e) blk[e] += f[e];
          }
        }
        // A 16-row block ends here (or the span does): fold it in, in order.
        if (((r0 + nb) & 15) == 0 || r0 + nb == span_rows) {
#pragma unroll
          for (int e = 0; e < V; ++e) {
            acc[e] += blk[e];
            blk[e] = 0.f;
          }
        }
      }
    }
    if (al != nullptr) {
      float4* o = reinterpret_cast<float4*>(al);
#pragma unroll
      for (int e = 0; e < V; e += 4)
        o[e / 4] = make_float4(acc[e] * p.scale, acc[e + 1] * p.scale, acc[e + 2] * p.scale,
                               acc[e + 3] * p.scale);
    }
    return;
  }
  const int64_t gi = item - 2 * span_items;
  if (gi >= 2 * gen_items) return;
  const bool is_v = gi >= gen_items;
  const int64_t it = is_v ? gi - gen_items : gi;
  const int c = static_cast<int>(it % C);
  const int64_t rr = it / C;
  const int64_t g = rr % p.n_gen;
  const int64_t u = rr / p.n_gen;
  const int64_t b = u / p.heads, h = u % p.heads;
  const unsigned char* src =
      (is_v ? p.v : p.k) + (b * p.n_tok + p.n_prompt + g) * src_row + h * RB + c * 16;
  unsigned char* dst = (is_v ? p.vg : p.kg) + (u * p.n_gen + g) * RB + c * 16;
  st_row(dst, ld_stream(src));
}

template <typename T, int D>
cudaError_t launch_typed(const CacheParams& p, cudaStream_t stream) {
  constexpr int C = D / Elem<T>::kPer16B;
  const int64_t P = p.n_prompt >> p.levels;
  const int64_t items = 2 * p.units * (P + p.n_gen) * C;
  if (items == 0) return cudaSuccess;
  const int64_t blocks = (items + kThreads - 1) / kThreads;
  cache_write_kernel<T, D><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_cache(const LaunchDims& ld, const CacheParams& p, cudaStream_t stream) {
  if (ld.dtype == WF_BF16) {
    if (ld.head_dim == 128) return launch_typed<__nv_bfloat16, 128>(p, stream);
    return launch_typed<__nv_bfloat16, 64>(p, stream);
  }
  if (ld.head_dim == 128) return launch_typed<float, 128>(p, stream);
  return launch_typed<float, 64>(p, stream);
}

}  // namespace

cudaError_t launch_cache_init(const LaunchDims& ld, const void* k, const void* v, void* kp,
                              void* vp, void* kg, void* vg, float* al, cudaStream_t stream) {
  CacheParams p;
  p.k = static_cast<const unsigned char*>(k);
  p.v = static_cast<const unsigned char*>(v);
  p.kp = static_cast<unsigned char*>(kp);
  p.vp = static_cast<unsigned char*>(vp);
  p.kg = static_cast<unsigned char*>(kg);
  p.vg = static_cast<unsigned char*>(vg);
  p.al = al;
  p.units = ld.units;
  p.heads = static_cast<int>(ld.units / ld.batch);
  p.n_tok = ld.n_prompt + ld.n_gen;
  p.n_prompt = ld.n_prompt;
  p.n_gen = ld.n_gen;
  p.levels = ld.levels;
  p.scale = static_cast<float>(std::pow(2.0, -0.5 * ld.levels));  // 2^(-L/2)
  return launch_cache(ld, p, stream);
}

cudaError_t launch_cache_update(const LaunchDims& ld, const void* k, const void* v, void* kg,
                                void* vg, cudaStream_t stream) {
  CacheParams p;
  p.k = static_cast<const unsigned char*>(k);
  p.v = static_cast<const unsigned char*>(v);
  p.kp = p.vp = nullptr;
  p.kg = static_cast<unsigned char*>(kg);
  p.vg = static_cast<unsigned char*>(vg);
  p.al = nullptr;
  p.units = ld.units;
  p.heads = static_cast<int>(ld.units / ld.batch);
  p.n_tok = ld.n_gen;
  p.n_prompt = 0;
  p.n_gen = ld.n_gen;
  p.levels = 0;
  p.scale = 1.f;
  return launch_cache(ld, p, stream);
}

}  // namespace wf
