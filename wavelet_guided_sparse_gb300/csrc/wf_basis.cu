// The filtering path for orthonormal wavelet bases longer than the Haar pair
// (WaveFilter §3.1 leaves the basis psi open).
//
// Readings: the basis is given by its low-pass filter g (2..16 taps; the
// extremal-phase Daubechies filters come from wf_daubechies_lowpass); each
// pyramid level extends its input periodically,
//     A_j[n] = sum_k g[k] A_{j-1}[(2n + k) mod M_{j-1}],   A_0 = Kp;
// the recursive filter keeps the pyramid's index tree (children 2p, 2p+1 of
// every survivor) and scores candidates against that basis's A_j with the
// same attention mass and Top-K order as the Haar path.
//
// Design (a plain, general path beside the fused Haar kernel):
//  * basis_level_kernel: one launch per level, one thread per (unit, output
//    row, 4 channels), F taps read with the periodic wrap; writes every level
//    A_1..A_L in fp32 (level-major blocks), so level j of a candidate is one
//    row read.
//  * basis_filter_kernel: one 8-warp CTA per unit walks the levels L..0.
//    A warp stages eight candidate rows at once (A_j in fp32, or the K_p
//    rows at level 0; eight 16-byte loads in flight per lane) in shared
//    memory and its lanes compute the logits of queries lane and lane + 32
//    against each (queries transposed in shared memory, so the
//    reads are conflict-free), keeping per-query online (max, sum) in the
//    log2 domain; per-warp statistics are merged, each candidate's mass is
//    summed over the queries and the block radix select keeps k_j (larger
//    score first, lower position on ties).  Logits go through the
//    workspace (G floats per candidate).
//  * steps 4-5 reuse the path kernel's gather + attention phase.
// No kernel here waits on anything but __syncthreads().
#include <algorithm>
#include <cmath>
#include <complex>
#include <vector>

#include "wf_common.cuh"
#include "wf_internal.h"
#include "wf_mma.cuh"

namespace wf {

namespace {

constexpr int kMaxG = 64;  // queries per unit (lanes lane and lane + 32)
constexpr int kRowsPerWarp = 8;  // candidate rows a warp stages at once (loads in flight)

__device__ __forceinline__ void load4_f32(const float* p, float* f) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  f[0] = v.x;
  f[1] = v.y;
  f[2] = v.z;
  f[3] = v.w;
}
__device__ __forceinline__ void load4_f32(const __nv_bfloat16* p, float* f) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  f[0] = bf16_lo(v.x);
  f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y);
  f[3] = bf16_hi(v.y);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) basis_level_kernel(const T* __restrict__ src,
                                                               float* __restrict__ dst,
                                                               int64_t units, int m_in,
                                                               BasisTaps taps) {
  constexpr int C4 = D / 4;
  const int m_out = m_in / 2;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (item >= units * m_out * C4) return;
  const int c4 = static_cast<int>(item % C4);
  const int64_t r = item / C4;
  const int n = static_cast<int>(r % m_out);
  const int64_t u = r / m_out;
  const T* base = src + u * m_in * D + c4 * 4;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 16; ++k) {  // constant tap indices: the taps stay in parameter space
    if (k < taps.n) {
      const int row = (2 * n + k) % m_in;
      float x[4];
      load4_f32(base + static_cast<int64_t>(row) * D, x);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = fmaf(taps.g[k], x[e], acc[e]);
    }
  }
  *reinterpret_cast<float4*>(dst + (u * m_out + n) * D + c4 * 4) =
      make_float4(acc[0], acc[1], acc[2], acc[3]);
}

struct FilterSmem {
  TopkSmem tk;
  float stat_m[kWarps][kMaxG];
  float stat_l[kWarps][kMaxG];
  float gm[kMaxG];
  float ginv[kMaxG];
};

template <typename T, int D>
struct FilterLayout {
  static constexpr size_t kQt = (sizeof(FilterSmem) + 15) & ~size_t{15};
  static constexpr size_t kRow = kQt + sizeof(float) * D * kMaxG;
  static constexpr size_t kTotal = kRow + sizeof(float) * kWarps * kRowsPerWarp * D;
};

// Stages rows pos[0..nr) of level j (fp32 A_j, or the K_p rows of type T at
// j = 0) into buf[r][D] as floats; one warp.  Every lane issues its 16-byte
// chunk of all nr rows before widening any, so nr loads are in flight.
template <typename T, int D>
__device__ __forceinline__ void stage_rows(const BasisFilterParams& p, int64_t u, int j,
                                           const int* pos, int nr, float* buf) {
  const int lane = threadIdx.x & 31;
  if (j == 0) {
    constexpr int V = Elem<T>::kPer16B, C = D / V;  // C <= 32 chunks per row
    const T* base = static_cast<const T*>(p.kp) + u * p.n_prompt * D + lane * V;
    uint4 raw[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
      if (r < nr && lane < C) raw[r] = ldg16(base + static_cast<int64_t>(pos[r]) * D);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      if (r < nr && lane < C) {
        float f[V];
        widen16(raw[r], static_cast<const T*>(nullptr), f);
#pragma unroll
        for (int e = 0; e < V; ++e) buf[r * D + lane * V + e] = f[e];
      }
    }
  } else {
    constexpr int C = D / 4;
    const float* base = p.a_all + p.level_off[j] + u * (p.n_prompt >> j) * D + lane * 4;
    uint4 raw[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
      if (r < nr && lane < C) raw[r] = ldg16(base + static_cast<int64_t>(pos[r]) * D);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      if (r < nr && lane < C) {
        float f[4];
        widen16(raw[r], static_cast<const float*>(nullptr), f);
#pragma unroll
        for (int e = 0; e < 4; ++e) buf[r * D + lane * 4 + e] = f[e];
      }
    }
  }
}

__device__ __forceinline__ void online_add(float& m, float& l, float z) {
  const float mn = fmaxf(m, z);
  l = l * fast_exp2(m - mn) + fast_exp2(z - mn);
  m = mn;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) basis_filter_kernel(BasisFilterParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  using L = FilterLayout<T, D>;
  FilterSmem& sm = *reinterpret_cast<FilterSmem*>(smem);
  float* qt = reinterpret_cast<float*>(smem + L::kQt);  // [D][kMaxG], prescaled queries
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t u = blockIdx.x;
  const int G = p.n_gen;
  float* rowbuf = reinterpret_cast<float*>(smem + L::kRow) + warp * kRowsPerWarp * D;
  const T* q = static_cast<const T*>(p.q) + u * G * D;
  for (int e = tid; e < kMaxG * D; e += kThreads) {
    const int i = e % kMaxG, c = e / kMaxG;
    qt[e] = i < G ? to_f32(q[i * D + c]) * p.qscale : 0.f;
  }
  __syncthreads();
  int32_t* cur = p.cand + u * p.cap;             // candidates of the level below
  int32_t* sel = p.cand + (p.units + u) * p.cap;  // survivors of this level
  uint32_t* keys = p.keys + u * p.cap;
  float* z = p.z + u * p.cap * G;
  const int32_t* map = nullptr;                   // level L: candidate i is position i
  int ncand = p.n_prompt >> p.levels;
  for (int j = p.levels; j >= 0; --j) {
    // Logits and per-warp online statistics (queries lane and lane + 32).
    float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
    for (int c0 = warp * kRowsPerWarp; c0 < ncand; c0 += kWarps * kRowsPerWarp) {
      const int nr = min(kRowsPerWarp, ncand - c0);
      int pos[kRowsPerWarp];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) pos[r] = r < nr ? (map ? map[c0 + r] : c0 + r) : 0;
      stage_rows<T, D>(p, u, j, pos, nr, rowbuf);
      __syncwarp();
      for (int r = 0; r < nr; ++r) {
        const float* row = rowbuf + r * D;
        float z0 = 0.f, z1 = 0.f;
#pragma unroll 8
        for (int k = 0; k < D; ++k) {
          const float x = row[k];
          z0 = fmaf(x, qt[k * kMaxG + lane], z0);
          z1 = fmaf(x, qt[k * kMaxG + lane + 32], z1);
        }
        const int64_t c = c0 + r;
        if (lane < G) {
          z[c * G + lane] = z0;
          online_add(m0, l0, z0);
        }
        if (lane + 32 < G) {
          z[c * G + lane + 32] = z1;
          online_add(m1, l1, z1);
        }
      }
      __syncwarp();
    }
    sm.stat_m[warp][lane] = m0;
    sm.stat_l[warp][lane] = l0;
    sm.stat_m[warp][lane + 32] = m1;
    sm.stat_l[warp][lane + 32] = l1;
    __syncthreads();
    if (tid < G) {
      float m = -INFINITY;
      for (int w = 0; w < kWarps; ++w) m = fmaxf(m, sm.stat_m[w][tid]);
      float l = 0.f;
      for (int w = 0; w < kWarps; ++w)
        if (sm.stat_m[w][tid] != -INFINITY) l += sm.stat_l[w][tid] * fast_exp2(sm.stat_m[w][tid] - m);
      sm.gm[tid] = m;
      sm.ginv[tid] = 1.f / l;
    }
    __syncthreads();
    // Attention mass of every candidate: sum over the queries of its softmax weight.
    for (int c = tid; c < ncand; c += kThreads) {
      const float* zc = z + static_cast<int64_t>(c) * G;
      float s = 0.f;
      for (int i = 0; i < G; ++i) s += fast_exp2(zc[i] - sm.gm[i]) * sm.ginv[i];
      keys[c] = __float_as_uint(s);  // s >= 0: the bit pattern orders like the value
    }
    __syncthreads();
    const int kj = p.k[j];
    int32_t* out = j == 0 ? p.idx + u * p.k[0] : sel;
    block_select_topk(keys, ncand, kj, 0, kj, out, sm.tk, false, map);
    if (j > 0) {
      // Children of the survivors, ascending because the survivors are.
      for (int s = tid; s < kj; s += kThreads) {
        const int32_t par = sel[s];
        cur[2 * s] = 2 * par;
        cur[2 * s + 1] = 2 * par + 1;
      }
      __syncthreads();
      map = cur;
      ncand = 2 * kj;
    }
  }
}

// ------------------------------------------------- coarse logits of a basis
//
// With every level between L and 0 keeping all children (k_j = 2 k_{j+1}),
// the step needs only the level-L logits of the basis pyramid: the tokens
// under the coarse survivors are the same dyadic spans as in the Haar case
// and are scored on their own keys.  The L periodic levels compose into one
// periodic filter of the tokens,
//   A_L[c] = Σ_m w[m] · Kp[(2^L c + m) mod N_p],   m < W = (2^L - 1)(F - 1) + 1,
//   w = g for L = 1,   w_j[t] = Σ_k g[k] · w_{j-1}[t - 2^{j-1} k]
// (periodic extension commutes with the composition because 2 (x mod M) mod
// 2M = 2x mod 2M), so the logits are the same filter applied to the token
// logits:  z_L[c][q] = Σ_m w[m] · (Q_q · Kp[(2^L c + m) mod N_p]).
// basis_coarse_kernel: a CTA takes up to kCoarsePos consecutive coarse
// positions, streams the token rows under their filter windows through a
// four-stage cp.async ring of 64-row tiles, forms each tile's token logits on
// the tensor cores (mma.sync, bf16 in, fp32 out) and adds them into its
// (position, query) accumulators with the filter weights.
constexpr int kCoarsePos = 32;   // coarse positions per CTA
constexpr int kCoarseRows = 64;  // token rows per tile
constexpr int kCoarseStages = 4;  // tiles in flight (two CTAs per SM)

template <int D>
struct CoarseSmem {
  static constexpr int kPitch = D * 2 + 16;  // bf16 row pitch (conflict-free fragment loads)
  static constexpr size_t kQ = 0;
  static constexpr size_t kStage = kQ + static_cast<size_t>(64) * kPitch;
  static constexpr size_t kZ = kStage + static_cast<size_t>(kCoarseStages) * kCoarseRows * kPitch;
  static constexpr size_t kW = kZ + sizeof(float) * kCoarseRows * 65;
  static constexpr size_t kTotal = kW + sizeof(float) * kMaxCascade;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2) basis_coarse_kernel(const __grid_constant__ BasisCoarseParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  using S = CoarseSmem<D>;
  constexpr int RB = S::kPitch, C16 = D / 8;  // 16-byte chunks per row
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t u = blockIdx.y;
  const int G = p.n_gen, L = p.levels, N = p.n_prompt, P = N >> L, W = p.w_len;
  const int c0 = blockIdx.x * kCoarsePos;
  const int ncp = min(kCoarsePos, P - c0);
  const int nrows = ((ncp - 1) << L) + W;
  const int nch = (nrows + kCoarseRows - 1) / kCoarseRows;
  const int64_t base = static_cast<int64_t>(c0) << L;
  const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(p.kp) + u * N * D;
  unsigned char* qs = smem + S::kQ;
  float* zt = reinterpret_cast<float*>(smem + S::kZ);
  float* ws = reinterpret_cast<float*>(smem + S::kW);
  const int ZT = G | 1;

  auto issue = [&](int ch, int stage) {
    unsigned char* dst = smem + S::kStage + static_cast<size_t>(stage) * kCoarseRows * RB;
    for (int e = tid; e < kCoarseRows * C16; e += kThreads) {
      const int r = e / C16, c = e % C16;
      const int64_t rel = static_cast<int64_t>(ch) * kCoarseRows + r;
      const int64_t row = (base + (rel < nrows ? rel : 0)) % N;
      cp_async16(dst + r * RB + c * 16, kp + row * D + c * 8);
    }
    cp_async_commit();
  };
  for (int ch = 0; ch < kCoarseStages && ch < nch; ++ch) issue(ch, ch);
  // Queries (rows >= G zero) and the filter weights.
  {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q) + u * G * D;
    for (int e = tid; e < 64 * C16; e += kThreads) {
      const int r = e / C16, c = e % C16;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < G) v = *reinterpret_cast<const uint4*>(q + r * D + c * 8);
      *reinterpret_cast<uint4*>(qs + r * RB + c * 16) = v;
    }
    for (int m = tid; m < W; m += kThreads) ws[m] = p.w[m];
  }
  // Accumulators: item it = tid + kThreads i is (position it / G, query it % G).
  constexpr int kItems = kCoarsePos * 64 / kThreads;
  float acc[kItems];
#pragma unroll
  for (int i = 0; i < kItems; ++i) acc[i] = 0.f;
  const int rb = 16 * (warp & 3);  // this warp's 16 rows of a tile
  const int NT = (G + 7) >> 3;
  const uint32_t qb = smem_u32(qs);
  for (int ch = 0; ch < nch; ++ch) {
    const int stage = ch % kCoarseStages;
    // Tiles issued so far: 0 .. min(ch + kCoarseStages, nch) - 1; tile ch must have landed.
    switch (min(kCoarseStages - 1, nch - 1 - ch)) {
      case 0: cp_async_wait<0>(); break;
      case 1: cp_async_wait<1>(); break;
      case 2: cp_async_wait<2>(); break;
      default: cp_async_wait<3>(); break;
    }
    __syncthreads();  // tile ch landed; every thread is done with the previous logits
    // Token logits of the tile: rows rb..rb+15, query tiles warp / 4 + 2t.
    {
      const uint32_t kb = smem_u32(smem + S::kStage + static_cast<size_t>(stage) * kCoarseRows * RB);
      const uint32_t arow = kb + (rb + (lane & 15)) * RB + (lane >> 4) * 16;
      float c[4][4];
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[t][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(arow + ks * 32, a);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int nt = (warp >> 2) + 2 * t;
          if (nt < NT) {
            const uint32_t ba = qb + (nt * 8 + (lane >> 2)) * RB + ks * 32 + (lane & 3) * 4;
            uint32_t b[2];
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b[0]) : "r"(ba));
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b[1]) : "r"(ba + 16));
            mma_bf16(c[t], a, b);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int nt = (warp >> 2) + 2 * t;
        if (nt >= NT) break;
        const int col = nt * 8 + 2 * (lane & 3);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = rb + (lane >> 2) + 8 * h;
          if (col < G) zt[r * ZT + col] = c[t][2 * h];
          if (col + 1 < G) zt[r * ZT + col + 1] = c[t][2 * h + 1];
        }
      }
    }
    __syncthreads();  // the tile's logits are complete; its stage may be refilled
    if (ch + kCoarseStages < nch) issue(ch + kCoarseStages, stage);
    // Filter the tile's logits into the accumulators.
    const int r0 = ch * kCoarseRows;
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
      const int it = tid + kThreads * i;
      const int cr = it / G, q = it - cr * G;
      if (cr < ncp) {
        const int w0 = cr << L;  // first row of the position's window
        const int lo = max(r0, w0), hi = min(r0 + kCoarseRows, w0 + W);
        float s = acc[i];
        for (int r = lo; r < hi; ++r) s = fmaf(ws[r - w0], zt[(r - r0) * ZT + q], s);
        acc[i] = s;
      }
    }
  }
  float* out = p.zl + (u * P + c0) * p.gz;
#pragma unroll
  for (int i = 0; i < kItems; ++i) {
    const int it = tid + kThreads * i;
    const int cr = it / G, q = it - cr * G;
    if (cr < ncp) out[cr * p.gz + q] = acc[i] * p.zscale;
  }
}

template <typename T, int D>
cudaError_t launch_pyramid_typed(const LaunchDims& ld, const void* kp, float* a_all,
                                 const BasisTaps& taps, cudaStream_t stream) {
  size_t off = 0;
  for (int j = 1; j <= ld.levels; ++j) {
    const int m_in = ld.n_prompt >> (j - 1);
    const int64_t items = ld.units * (m_in / 2) * (D / 4);
    const unsigned blocks = static_cast<unsigned>((items + kThreads - 1) / kThreads);
    float* dst = a_all + off;
    if (j == 1) {
      basis_level_kernel<T, D><<<blocks, kThreads, 0, stream>>>(static_cast<const T*>(kp), dst,
                                                               ld.units, m_in, taps);
    } else {
      const float* src = a_all + off - static_cast<size_t>(ld.units) * m_in * D;
      basis_level_kernel<float, D><<<blocks, kThreads, 0, stream>>>(src, dst, ld.units, m_in,
                                                                   taps);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    off += static_cast<size_t>(ld.units) * (m_in / 2) * D;
  }
  return cudaSuccess;
}

template <typename T, int D>
cudaError_t launch_filter_typed(const LaunchDims& ld, const BasisFilterParams& p,
                                cudaStream_t stream) {
  const cudaError_t e = ensure_max_smem<basis_filter_kernel<T, D>>();
  if (e != cudaSuccess) return e;
  basis_filter_kernel<T, D><<<static_cast<unsigned>(ld.units), kThreads,
                              FilterLayout<T, D>::kTotal, stream>>>(p);
  return cudaGetLastError();
}

// Roots of a real polynomial (coefficients highest power first, degree >= 1)
// by the Durand-Kerner simultaneous iteration.
std::vector<std::complex<double>> poly_roots(const std::vector<double>& c) {
  const int n = static_cast<int>(c.size()) - 1;
  std::vector<std::complex<double>> r(n);
  const std::complex<double> seed(0.4, 0.9);
  std::complex<double> pw(1.0, 0.0);
  for (int i = 0; i < n; ++i) {
    r[i] = pw;
    pw *= seed;
  }
  auto eval = [&](std::complex<double> x) {
    std::complex<double> v(c[0] / c[0], 0.0);
    for (int i = 1; i <= n; ++i) v = v * x + c[i] / c[0];
    return v;
  };
  for (int it = 0; it < 2000; ++it) {
    double change = 0.0;
    for (int i = 0; i < n; ++i) {
      std::complex<double> den(1.0, 0.0);
      for (int k = 0; k < n; ++k)
        if (k != i) den *= r[i] - r[k];
      const std::complex<double> step = eval(r[i]) / den;
      r[i] -= step;
      change = std::max(change, std::abs(step));
    }
    if (change < 1e-15) break;
  }
  return r;
}

}  // namespace

int daubechies_lowpass(int n_moments, double* out) {
  const int n = n_moments;
  std::vector<std::complex<double>> zeros(n, std::complex<double>(-1.0, 0.0));
  if (n > 1) {
    // P(y) = sum_{k<N} binom(N-1+k, k) y^k, highest power first.
    std::vector<double> pc(n);
    for (int k = 0; k < n; ++k) {
      double b = 1.0;  // binom(N-1+k, k)
      for (int i = 1; i <= k; ++i) b = b * (n - 1 + i) / i;
      pc[n - 1 - k] = b;
    }
    for (const std::complex<double>& y : poly_roots(pc)) {
      // z + 1/z = 2 - 4y: of the two reciprocal roots keep the inner one.
      const std::complex<double> b = 1.0 - 2.0 * y;
      const std::complex<double> s = std::sqrt(b * b - 1.0);
      const std::complex<double> z1 = b + s, z2 = b - s;
      zeros.push_back(std::abs(z1) < 1.0 ? z1 : z2);
    }
  }
  // Monic polynomial with these zeros, highest power first.
  std::vector<std::complex<double>> c(1, std::complex<double>(1.0, 0.0));
  for (const std::complex<double>& zr : zeros) {
    std::vector<std::complex<double>> nc(c.size() + 1, std::complex<double>(0.0, 0.0));
    for (size_t i = 0; i < c.size(); ++i) {
      nc[i] += c[i];
      nc[i + 1] -= c[i] * zr;
    }
    c.swap(nc);
  }
  double sum = 0.0;
  for (const auto& v : c) sum += v.real();
  const double scale = std::sqrt(2.0) / sum;
  for (size_t i = 0; i < c.size(); ++i) out[i] = c[i].real() * scale;
  return static_cast<int>(c.size());
}

cudaError_t launch_basis_pyramid(const LaunchDims& ld, const void* kp, float* a_all,
                                 const BasisTaps& taps, cudaStream_t stream) {
  if (ld.dtype == WF_BF16) {
    if (ld.head_dim == 128)
      return launch_pyramid_typed<__nv_bfloat16, 128>(ld, kp, a_all, taps, stream);
    return launch_pyramid_typed<__nv_bfloat16, 64>(ld, kp, a_all, taps, stream);
  }
  if (ld.head_dim == 128) return launch_pyramid_typed<float, 128>(ld, kp, a_all, taps, stream);
  return launch_pyramid_typed<float, 64>(ld, kp, a_all, taps, stream);
}

cudaError_t launch_basis_filter(const LaunchDims& ld, const BasisFilterParams& p,
                                cudaStream_t stream) {
  if (ld.dtype == WF_BF16) {
    if (ld.head_dim == 128) return launch_filter_typed<__nv_bfloat16, 128>(ld, p, stream);
    return launch_filter_typed<__nv_bfloat16, 64>(ld, p, stream);
  }
  if (ld.head_dim == 128) return launch_filter_typed<float, 128>(ld, p, stream);
  return launch_filter_typed<float, 64>(ld, p, stream);
}

int basis_cascade_len(int taps, int levels) {
  const int64_t len = ((int64_t{1} << levels) - 1) * (taps - 1) + 1;
  return len > kMaxCascade ? -1 : static_cast<int>(len);
}

int basis_cascade(const double* g, int taps, int levels, float* w) {
  const int W = basis_cascade_len(taps, levels);
  if (W < 0) return -1;
  std::vector<double> cur(g, g + taps), next;
  for (int j = 2; j <= levels; ++j) {
    const int len = ((1 << j) - 1) * (taps - 1) + 1, step = 1 << (j - 1);
    next.assign(len, 0.0);
    for (int k = 0; k < taps; ++k)
      for (size_t m = 0; m < cur.size(); ++m) next[k * step + m] += g[k] * cur[m];
    cur.swap(next);
  }
  for (int m = 0; m < W; ++m) w[m] = static_cast<float>(cur[m]);
  return W;
}

cudaError_t launch_basis_coarse(const LaunchDims& ld, const BasisCoarseParams& p,
                                cudaStream_t stream) {
  if (ld.dtype != WF_BF16 || p.w_len < 1 || p.w_len > kMaxCascade || ld.n_gen > 64)
    return cudaErrorInvalidValue;
  const int P = ld.n_prompt >> ld.levels;
  const dim3 grid(static_cast<unsigned>((P + kCoarsePos - 1) / kCoarsePos),
                  static_cast<unsigned>(ld.units));
  if (ld.head_dim == 128) {
    const cudaError_t e = ensure_max_smem<basis_coarse_kernel<128>>();
    if (e != cudaSuccess) return e;
    basis_coarse_kernel<128><<<grid, kThreads, CoarseSmem<128>::kTotal, stream>>>(p);
  } else {
    const cudaError_t e = ensure_max_smem<basis_coarse_kernel<64>>();
    if (e != cudaSuccess) return e;
    basis_coarse_kernel<64><<<grid, kThreads, CoarseSmem<64>::kTotal, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace wf
