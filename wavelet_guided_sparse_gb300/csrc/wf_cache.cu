// KV-cache writes around the filtering path: the cache initialisation of the
// first denoising step (WaveFilter §2.1 eq. (2)) with the level-L Haar
// approximation of the prompt keys (§2.2 eq. (5) pyramid, §3.1) produced in
// the same pass, the generation-row update of later steps (eq. (4)), and
// eq. (4) over an arbitrary position set with the A_L repair it implies.
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

// ------------------------------------------------------------- scattered update
// Eq. (4) over an arbitrary set of positions (prompt or generation): one
// thread per (tensor, new row, head, 16-byte chunk) copies the chunk to the
// row's place in the head-major cache; an index outside [0, N_p + G) is
// skipped and flagged.  Then (optional) one thread per (new row, head,
// chunk) re-forms A_L of the coarse position whose span holds a rewritten
// prompt row, from the updated cache and in the summation order of the
// streaming low-pass kernel (16-row blocks folded in order), so the repaired
// rows equal a fresh wf_dwt_lowpass of the updated keys bit for bit.  Rows
// of one span rewritten together recompute the same values (same bits).
struct ScatterParams {
  const unsigned char* k;  // [batch, rows, heads, d] token-major new rows
  const unsigned char* v;
  const int32_t* pos;      // [batch, rows]
  unsigned char* kp;
  unsigned char* vp;
  unsigned char* kg;
  unsigned char* vg;
  float* al;               // nullable
  int32_t* status;         // nullable
  int64_t units;
  int heads, rows, n_prompt, n_gen, levels;
  float scale;
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) scatter_rows_kernel(ScatterParams p) {
  constexpr int C = D / Elem<T>::kPer16B, RB = D * static_cast<int>(sizeof(T));
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t per_tensor = p.units * p.rows * C;
  if (item >= 2 * per_tensor) return;
  const bool is_v = item >= per_tensor;
  const int64_t it = is_v ? item - per_tensor : item;
  const int c = static_cast<int>(it % C);
  const int64_t rh = it / C;                 // (b, m, h) with h fastest
  const int64_t h = rh % p.heads, bm = rh / p.heads;
  const int64_t b = bm / p.rows;
  const int n = p.pos[bm];
  if (n < 0 || n >= p.n_prompt + p.n_gen) {
    if (!is_v && c == 0 && h == 0) raise_flag(p.status, WF_DEV_BAD_INDEX);
    return;
  }
  const int64_t u = b * p.heads + h;
  const unsigned char* src = (is_v ? p.v : p.k) + (bm * p.heads + h) * RB + c * 16;
  unsigned char* dst = n < p.n_prompt
                           ? (is_v ? p.vp : p.kp) + (u * p.n_prompt + n) * RB + c * 16
                           : (is_v ? p.vg : p.kg) + (u * p.n_gen + (n - p.n_prompt)) * RB + c * 16;
  *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) repair_al_kernel(ScatterParams p) {
  constexpr int V = Elem<T>::kPer16B, C = D / V, RB = D * static_cast<int>(sizeof(T));
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (item >= p.units * p.rows * C) return;
  const int c = static_cast<int>(item % C);
  const int64_t rh = item / C;
  const int64_t h = rh % p.heads, bm = rh / p.heads;
  const int64_t b = bm / p.rows;
  const int n = p.pos[bm];
  if (n < 0 || n >= p.n_prompt) return;  // generation rows do not enter A_L
  const int64_t u = b * p.heads + h;
  const int span_rows = 1 << p.levels;
  const int64_t cpos = n >> p.levels;
  const unsigned char* src = p.kp + (u * p.n_prompt + (cpos << p.levels)) * RB + c * 16;
  float acc[V], blk[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = blk[e] = 0.f;
  for (int r = 0; r < span_rows; ++r) {
    float f[V];
    widen16(__ldcg(reinterpret_cast<const uint4*>(src + static_cast<int64_t>(r) * RB)),
            static_cast<const T*>(nullptr), f);
#pragma unroll
    for (int e = 0; e < V; ++e) blk[e] += f[e];
    if (((r + 1) & 15) == 0 || r + 1 == span_rows) {
#pragma unroll
      for (int e = 0; e < V; ++e) {
        acc[e] += blk[e];
        blk[e] = 0.f;
      }
    }
  }
  float4* o = reinterpret_cast<float4*>(p.al + (u * (p.n_prompt >> p.levels) + cpos) * D + c * V);
#pragma unroll
  for (int e = 0; e < V; e += 4)
    o[e / 4] = make_float4(acc[e] * p.scale, acc[e + 1] * p.scale, acc[e + 2] * p.scale,
                           acc[e + 3] * p.scale);
}

template <typename T, int D>
cudaError_t launch_scatter_typed(const ScatterParams& p, cudaStream_t stream) {
  constexpr int C = D / Elem<T>::kPer16B;
  const int64_t items = p.units * p.rows * C;
  if (items == 0) return cudaSuccess;
  scatter_rows_kernel<T, D><<<static_cast<unsigned>((2 * items + kThreads - 1) / kThreads), kThreads,
                              0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.al == nullptr) return e;
  repair_al_kernel<T, D><<<static_cast<unsigned>((items + kThreads - 1) / kThreads), kThreads, 0,
                           stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cache_scatter(const LaunchDims& ld, const void* k, const void* v,
                                 const int32_t* pos, int rows, void* kp, void* vp, void* kg,
                                 void* vg, float* al, int32_t* status, cudaStream_t stream) {
  ScatterParams p;
  p.k = static_cast<const unsigned char*>(k);
  p.v = static_cast<const unsigned char*>(v);
  p.pos = pos;
  p.kp = static_cast<unsigned char*>(kp);
  p.vp = static_cast<unsigned char*>(vp);
  p.kg = static_cast<unsigned char*>(kg);
  p.vg = static_cast<unsigned char*>(vg);
  p.al = al;
  p.status = status;
  p.units = ld.units;
  p.heads = static_cast<int>(ld.units / ld.batch);
  p.rows = rows;
  p.n_prompt = ld.n_prompt;
  p.n_gen = ld.n_gen;
  p.levels = ld.levels;
  p.scale = static_cast<float>(std::pow(2.0, -0.5 * ld.levels));  // 2^(-L/2)
  if (ld.dtype == WF_BF16) {
    if (ld.head_dim == 128) return launch_scatter_typed<__nv_bfloat16, 128>(p, stream);
    return launch_scatter_typed<__nv_bfloat16, 64>(p, stream);
  }
  if (ld.head_dim == 128) return launch_scatter_typed<float, 128>(p, stream);
  return launch_scatter_typed<float, 64>(p, stream);
}

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
