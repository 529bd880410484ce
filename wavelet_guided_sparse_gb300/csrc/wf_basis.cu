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

}  // namespace wf
