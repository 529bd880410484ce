// Step 2: importance of every coarse position and the coarse Top-K.
//
// WaveFilter (arXiv 2606.00724) Fig. 2(c) and §1: the queries of the
// generation block are scored against the low-frequency keys A_L with the
// eq. (3) logits, and a Top-K keeps the candidate regions.  Score of coarse
// position p (attention mass):
//   z[i,p] = Q[i]·A_L[p]/√d,   s[p] = Σ_i exp(z[i,p] - m_i) / l_i,
//   m_i = max_p z[i,p],        l_i = Σ_p exp(z[i,p] - m_i).
//
// Design: one thread-block cluster per (sequence, head) unit; the P = N_p/2^L
// coarse positions are split into equal contiguous slices, one per CTA.  A
// CTA computes its slice of z with fp32 FMAs (A_L is fp32, so the logits are
// fp32-accurate, as the index-set parity needs), the per-query max/sum are
// merged across the cluster through DSMEM, and the exact radix Top-K of
// wf_common.cuh selects k_L positions with the lower-position tie-break.
#include "wf_common.cuh"
#include "wf_internal.h"

namespace wf {

namespace {

constexpr int kChunkRows = 32;  // A_L rows staged per pass

struct ScoreParams {
  const void* q;
  const float* al;
  int32_t* idx_out;
  float* scores_out;
  int32_t* status;
  int P;        // coarse positions per unit
  int per_cta;  // positions per CTA
  int G;
  int k;
  float inv_sqrt_d;
};

// Shared-memory carve-up (dynamic).
template <int D>
struct ScoreSmem {
  static constexpr int kRow = D + 4;  // fp32 row pitch (conflict-free float4 columns)
  size_t qs, as, z, keys, take, stats, topk, total;
  __host__ __device__ ScoreSmem(int G, int per_cta) {
    size_t o = 0;
    auto take_bytes = [&](size_t bytes) {
      const size_t at = o;
      o = (o + bytes + 15) & ~size_t(15);
      return at;
    };
    qs = take_bytes(sizeof(float) * 64 * kRow);
    as = take_bytes(sizeof(float) * kChunkRows * kRow);
    z = take_bytes(sizeof(float) * G * per_cta);
    keys = take_bytes(sizeof(uint32_t) * per_cta);
    take = take_bytes(per_cta);
    stats = take_bytes(sizeof(float) * 4 * 64);
    topk = take_bytes(sizeof(TopkSmem));
    total = o;
  }
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) score_topk_kernel(ScoreParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int64_t unit = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, Pc = p.per_cta;
  const ScoreSmem<D> L(G, Pc);
  constexpr int R = ScoreSmem<D>::kRow;
  float* qs = reinterpret_cast<float*>(smem + L.qs);
  float* as = reinterpret_cast<float*>(smem + L.as);
  float* z = reinterpret_cast<float*>(smem + L.z);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + L.keys);
  uint8_t* take = smem + L.take;
  float* loc_m = reinterpret_cast<float*>(smem + L.stats);
  float* loc_l = loc_m + 64;
  float* gm = loc_m + 128;
  float* ginv = loc_m + 192;
  TopkSmem& tk = *reinterpret_cast<TopkSmem*>(smem + L.topk);

  // Queries -> fp32 shared rows (rows >= G zero).
  const T* qsrc = static_cast<const T*>(p.q) + unit * G * D;
  constexpr int V = Elem<T>::kPer16B;
  for (int e = tid; e < 64 * (D / V); e += kThreads) {
    const int r = e / (D / V), c = (e % (D / V)) * V;
    float f[V];
    if (r < G) {
      load16_f32(qsrc + r * D + c, f);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) f[v] = 0.f;
    }
#pragma unroll
    for (int v = 0; v < V; ++v) qs[r * R + c + v] = f[v];
  }

  // z for this CTA's slice, kChunkRows A_L rows at a time.  Thread -> row
  // (lane) of the chunk and queries warp, warp + 8, ... (at most 8).
  const float* asrc = p.al + (unit * p.P + static_cast<int64_t>(rank) * Pc) * D;
  for (int c0 = 0; c0 < Pc; c0 += kChunkRows) {
    __syncthreads();
    const int rows = min(kChunkRows, Pc - c0);
    for (int e = tid; e < rows * (D / 4); e += kThreads) {
      const int r = e / (D / 4), c = (e % (D / 4)) * 4;
      *reinterpret_cast<float4*>(as + r * R + c) =
          __ldg(reinterpret_cast<const float4*>(asrc + static_cast<int64_t>(c0 + r) * D + c));
    }
    __syncthreads();
    if (lane < rows) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      const float* arow = as + lane * R;
#pragma unroll 4
      for (int c = 0; c < D; c += 4) {
        const float4 a = *reinterpret_cast<const float4*>(arow + c);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 b = *reinterpret_cast<const float4*>(qs + (warp + 8 * i) * R + c);
          acc[i] = fmaf(a.x, b.x, acc[i]);
          acc[i] = fmaf(a.y, b.y, acc[i]);
          acc[i] = fmaf(a.z, b.z, acc[i]);
          acc[i] = fmaf(a.w, b.w, acc[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int qi = warp + 8 * i;
        if (qi < G) z[qi * Pc + c0 + lane] = acc[i] * p.inv_sqrt_d;
      }
    }
  }
  __syncthreads();

  // Per-query max and sum of exponentials over this slice (warp per query).
  for (int qi = warp; qi < G; qi += kWarps) {
    float m = -INFINITY;
    for (int c = lane; c < Pc; c += 32) m = fmaxf(m, z[qi * Pc + c]);
    m = warp_max(m);
    float l = 0.f;
    for (int c = lane; c < Pc; c += 32) l += expf(z[qi * Pc + c] - m);
    l = warp_sum(l);
    if (lane == 0) {
      loc_m[qi] = m;
      loc_l[qi] = l;
    }
  }
  cluster.sync();
  // Merge over the cluster in rank order (deterministic).
  for (int qi = tid; qi < G; qi += kThreads) {
    float m = -INFINITY;
    for (int r = 0; r < static_cast<int>(cluster.num_blocks()); ++r)
      m = fmaxf(m, cluster.map_shared_rank(loc_m, r)[qi]);
    float l = 0.f;
    for (int r = 0; r < static_cast<int>(cluster.num_blocks()); ++r) {
      const float mr = cluster.map_shared_rank(loc_m, r)[qi];
      l += cluster.map_shared_rank(loc_l, r)[qi] * expf(mr - m);
    }
    gm[qi] = m;
    ginv[qi] = 1.f / l;
  }
  __syncthreads();

  // Scores of this slice.
  for (int c = tid; c < Pc; c += kThreads) {
    float s = 0.f;
    for (int qi = 0; qi < G; ++qi) s += expf(z[qi * Pc + c] - gm[qi]) * ginv[qi];
    keys[c] = __float_as_uint(s);
    if (p.scores_out != nullptr) p.scores_out[unit * p.P + rank * Pc + c] = s;
  }
  __syncthreads();

  const TopkResult res = cluster_topk(keys, Pc, p.k, take, tk);
  // Selected positions in ascending order.
  int carry = 0;
  for (int base = 0; base < Pc; base += kThreads) {
    const int c = base + tid;
    const int t = c < Pc ? take[c] : 0;
    int tot;
    const int pos = block_excl_scan(t, tk.scan, &tot);
    const int slot = res.offset + carry + pos;
    if (t && slot < p.k) p.idx_out[unit * p.k + slot] = rank * Pc + c;
    carry += tot;
  }
  cluster.sync();  // peers may still read this CTA's shared memory
}

template <typename T, int D>
cudaError_t launch_typed(const LaunchDims& ld, const ScorePlan& plan, const ScoreParams& prm,
                         cudaStream_t stream) {
  auto kern = score_topk_kernel<T, D>;
  const cudaError_t e = ensure_max_smem<score_topk_kernel<T, D>>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.cluster, static_cast<unsigned>(ld.units), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace

bool plan_score(const LaunchDims& ld, ScorePlan* plan) {
  const int P = ld.n_prompt >> ld.levels;
  int cs = 1;
  while (cs < kMaxCluster && P / (2 * cs) >= 32 && P % (2 * cs) == 0) cs *= 2;
  plan->cluster = cs;
  plan->per_cta = P / cs;
  plan->smem_bytes = ld.head_dim == 128 ? ScoreSmem<128>(ld.n_gen, P / cs).total
                                        : ScoreSmem<64>(ld.n_gen, P / cs).total;
  return plan->smem_bytes <= kMaxSmem;
}

cudaError_t launch_score_topk(const LaunchDims& ld, const ScorePlan& plan, const void* q,
                              const float* al, int k_l, int32_t* idx_l, float* scores,
                              int32_t* status, cudaStream_t stream) {
  ScoreParams prm;
  prm.q = q;
  prm.al = al;
  prm.idx_out = idx_l;
  prm.scores_out = scores;
  prm.status = status;
  prm.P = ld.n_prompt >> ld.levels;
  prm.per_cta = plan.per_cta;
  prm.G = ld.n_gen;
  prm.k = k_l;
  prm.inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(ld.head_dim)));
  if (ld.dtype == WF_BF16) {
    if (ld.head_dim == 128) return launch_typed<__nv_bfloat16, 128>(ld, plan, prm, stream);
    return launch_typed<__nv_bfloat16, 64>(ld, plan, prm, stream);
  }
  if (ld.head_dim == 128) return launch_typed<float, 128>(ld, plan, prm, stream);
  return launch_typed<float, 64>(ld, plan, prm, stream);
}

}  // namespace wf
