// Step 3: multi-scale recursive filtering down to token resolution.
//
// WaveFilter (arXiv 2606.00724) Fig. 2(d) and §1: the candidate regions kept
// by the coarse Top-K are refined scale by scale until the final key tokens
// remain.  For j = L-1 .. 0 the candidates are the children {2p, 2p+1} of the
// level-(j+1) survivors, each is scored like step 2 against its A_j (softmax
// over the current candidate set, summed over the queries), and k_j survive.
//
// Linearity makes every level cheap: A_j[c] = 2^(-j/2) Σ_{n in span(c)} Kp[n],
// so Q·A_j[c] = 2^(-j/2) Σ_{n in span(c)} Q·Kp[n].  The kernel therefore
// computes the token logits t[n, i] = Q[i]·Kp[n] ONCE for the 2^L·k_L rows
// under the coarse survivors (every later candidate lies inside them) and
// forms each level's logits by summing t over the candidate's leaves.  For
// bf16 inputs t comes from bf16 tensor-core MMAs whose products are exact
// and whose sums are fp32, so the logits stay fp32-accurate.
//
// Design: one thread-block cluster per unit.  The sorted coarse survivors are
// split into contiguous slices, one per CTA, so CTA ranks hold ascending,
// disjoint position ranges and every descendant of a CTA's spans stays in
// that CTA.  Span rows are staged into padded shared-memory rows by bulk
// copies (TMA engine) in a two-stage mbarrier pipeline.  The per-query
// softmax statistics of a level are merged across the cluster through DSMEM
// and the selection is the exact cluster Top-K of wf_common.cuh.  Levels
// whose k_j keeps every candidate skip scoring.
#include <climits>
#include <cmath>

#include "wf_common.cuh"
#include "wf_internal.h"

namespace wf {

namespace {

constexpr int kTileRows = 64;

struct FilterParams {
  const void* q;
  const void* kp;
  const int32_t* idx_l;
  int32_t* idx_out;
  int32_t* status;
  float* t_ws;  // token logits in global memory (nullptr: shared memory)
  int n_prompt, G, levels, kL, budget;
  int spans_cap, rows_cap, sorted_cap;
  int k[WF_MAX_LEVELS + 1];
  float scale[WF_MAX_LEVELS + 1];  // 2^(-j/2) / sqrt(d)
};

template <typename T, int D>
struct FilterSmem {
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(T)) + 16;  // padded row pitch
  size_t bars, qs, kst, sorted, sp, sr, cp, cr, keys, take, part, stats, misc, topk, t, total;
  __host__ __device__ FilterSmem(int G, int rows_cap, int sorted_cap, bool t_in_smem) {
    size_t o = 0;
    auto take_bytes = [&](size_t bytes) {
      const size_t at = o;
      o = (o + bytes + 15) & ~size_t(15);
      return at;
    };
    bars = take_bytes(2 * sizeof(uint64_t));
    qs = take_bytes(static_cast<size_t>(64) * kRowBytes);
    kst = take_bytes(static_cast<size_t>(2) * kTileRows * kRowBytes);
    sorted = take_bytes(sizeof(int32_t) * sorted_cap);
    sp = take_bytes(sizeof(int32_t) * rows_cap);
    sr = take_bytes(sizeof(int32_t) * rows_cap);
    cp = take_bytes(sizeof(int32_t) * rows_cap);
    cr = take_bytes(sizeof(int32_t) * rows_cap);
    keys = take_bytes(sizeof(uint32_t) * rows_cap);
    take = take_bytes(rows_cap);
    part = take_bytes(sizeof(float) * 2 * kWarps * 64);
    stats = take_bytes(sizeof(float) * 4 * 64);
    misc = take_bytes(sizeof(int32_t) * 8);
    topk = take_bytes(sizeof(TopkSmem));
    t = t_in_smem ? take_bytes(sizeof(float) * static_cast<size_t>(rows_cap) * G) : 0;
    total = o;
  }
};

// ------------------------------------------------------------- tensor-core helpers
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// t rows [row0, row0 + 64) of this CTA from the staged key rows (bf16, MMA).
// Warp w: 16-row block (w & 3), n-blocks (w >> 2) + 2i of 8 queries each.
template <int D>
__device__ __forceinline__ void token_logits_tile(const unsigned char* kst, const uint32_t (&bq)[4][D / 16][2],
                                                  float* t, int row0, int rows_valid, int G,
                                                  __nv_bfloat16*) {
  constexpr int RB = FilterSmem<__nv_bfloat16, D>::kRowBytes;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int mb = warp & 3, ng = warp >> 2;
  const int NB = (G + 7) >> 3;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
  const uint32_t abase = smem_u32(kst) + (mb * 16 + (lane & 15)) * RB + (lane >> 4) * 16;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t a[4];
    ldsm_x4(abase + ks * 32, a);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (ng + 2 * i < NB) mma_bf16(acc[i], a, bq[i][ks]);
  }
  const int r_lo = mb * 16 + (lane >> 2);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int nb = ng + 2 * i;
    if (nb >= NB) continue;
    const int q0 = nb * 8 + (lane & 3) * 2;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = r_lo + 8 * h;
      if (r >= rows_valid) continue;
      float* dst = t + static_cast<int64_t>(row0 + r) * G;
      if (q0 < G) dst[q0] = acc[i][2 * h];
      if (q0 + 1 < G) dst[q0 + 1] = acc[i][2 * h + 1];
    }
  }
}

// fp32 inputs: plain FMAs.  Thread -> row (tid & 63), queries (tid >> 6) + 4i.
template <int D>
__device__ __forceinline__ void token_logits_tile(const unsigned char* kst, const float* qs,
                                                  float* t, int row0, int rows_valid, int G,
                                                  float*) {
  constexpr int RB = FilterSmem<float, D>::kRowBytes;
  constexpr int RF = RB / 4;
  const int r = threadIdx.x & 63, g = threadIdx.x >> 6;
  if (r >= rows_valid) return;
  const float* krow = reinterpret_cast<const float*>(kst + r * RB);
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll 2
  for (int c = 0; c < D; c += 4) {
    const float4 a = *reinterpret_cast<const float4*>(krow + c);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float4 b = *reinterpret_cast<const float4*>(qs + (g + 4 * i) * RF + c);
      acc[i] = fmaf(a.x, b.x, acc[i]);
      acc[i] = fmaf(a.y, b.y, acc[i]);
      acc[i] = fmaf(a.z, b.z, acc[i]);
      acc[i] = fmaf(a.w, b.w, acc[i]);
    }
  }
  float* dst = t + static_cast<int64_t>(row0 + r) * G;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (g + 4 * i < G) dst[g + 4 * i] = acc[i];
}

__device__ __forceinline__ void online_update(float& m, float& l, float z) {
  if (z > m) {
    l = l * expf(m - z) + 1.f;
    m = z;
  } else {
    l += expf(z - m);
  }
}

// Merge (m, l) pairs; pairs with m = -inf (no candidates) are skipped.
__device__ __forceinline__ void merge_ml(float& m, float& l, float m2, float l2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    l = l2;
    return;
  }
  const float mx = fmaxf(m, m2);
  l = l * expf(m - mx) + l2 * expf(m2 - mx);
  m = mx;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) recursive_filter_kernel(FilterParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int64_t unit = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, levels = p.levels, kL = p.kL;
  const FilterSmem<T, D> L(G, p.rows_cap, p.sorted_cap, p.t_ws == nullptr);
  constexpr int RB = FilterSmem<T, D>::kRowBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  unsigned char* qs = smem + L.qs;
  unsigned char* kst = smem + L.kst;
  int32_t* sorted = reinterpret_cast<int32_t*>(smem + L.sorted);
  int32_t* sp = reinterpret_cast<int32_t*>(smem + L.sp);
  int32_t* sr = reinterpret_cast<int32_t*>(smem + L.sr);
  int32_t* cp = reinterpret_cast<int32_t*>(smem + L.cp);
  int32_t* cr = reinterpret_cast<int32_t*>(smem + L.cr);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + L.keys);
  uint8_t* take = smem + L.take;
  float* part_m = reinterpret_cast<float*>(smem + L.part);
  float* part_l = part_m + kWarps * 64;
  float* loc_m = reinterpret_cast<float*>(smem + L.stats);
  float* loc_l = loc_m + 64;
  float* gm = loc_m + 128;
  float* ginv = loc_m + 192;
  int32_t* misc = reinterpret_cast<int32_t*>(smem + L.misc);
  TopkSmem& tk = *reinterpret_cast<TopkSmem*>(smem + L.topk);
  float* t = p.t_ws == nullptr
                 ? reinterpret_cast<float*>(smem + L.t)
                 : p.t_ws + (static_cast<int64_t>(unit) * cs + rank) * p.rows_cap * G;

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
    misc[0] = 0;  // aborted (a bounded wait gave up)
  }
  // ---- coarse survivors: load, sort ascending, validate
  const int P = p.n_prompt >> levels;
  for (int i = tid; i < p.sorted_cap; i += kThreads)
    sorted[i] = i < kL ? p.idx_l[unit * kL + i] : INT_MAX;
  __syncthreads();
  for (int kk = 2; kk <= p.sorted_cap; kk <<= 1) {
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
      for (int i = tid; i < p.sorted_cap; i += kThreads) {
        const int ixj = i ^ jj;
        if (ixj > i) {
          const int a = sorted[i], b = sorted[ixj];
          const bool asc = (i & kk) == 0;
          if ((a > b) == asc) {
            sorted[i] = b;
            sorted[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  int bad = 0;
  for (int i = tid; i < kL; i += kThreads) {
    const int v = sorted[i];
    if (v < 0 || v >= P) bad |= WF_DEV_BAD_INDEX;
    if (i > 0 && sorted[i - 1] == v) bad |= WF_DEV_DUP_INDEX;
  }
  __syncthreads();
  for (int i = tid; i < kL; i += kThreads) sorted[i] = min(max(sorted[i], 0), P - 1);
  if (bad && rank == 0) raise_flag(p.status, bad);

  // ---- this CTA's slice of coarse survivors and its token rows
  const int s0 = static_cast<int>((static_cast<int64_t>(rank) * kL) / cs);
  const int s1 = static_cast<int>((static_cast<int64_t>(rank + 1) * kL) / cs);
  const int ns = s1 - s0;
  const int R = ns << levels;

  // ---- queries into shared memory (rows >= G zero)
  {
    const T* qsrc = static_cast<const T*>(p.q) + unit * G * D;
    constexpr int V = Elem<T>::kPer16B;
    for (int e = tid; e < 64 * (D / V); e += kThreads) {
      const int r = e / (D / V), c = (e % (D / V)) * V;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < G) v = ldg16(qsrc + r * D + c);
      *reinterpret_cast<uint4*>(qs + r * RB + c * sizeof(T)) = v;
    }
  }
  __syncthreads();

  // ---- token logits t = Kp[rows] · Q^T, two-stage bulk-copy pipeline
  const T* kp = static_cast<const T*>(p.kp);
  const int ntiles = (R + kTileRows - 1) / kTileRows;
  auto issue = [&](int tile, int stage) {  // warp 0 only
    const int r0 = tile * kTileRows;
    const int nr = min(kTileRows, R - r0);
    if (lane == 0) mbar_arrive_expect_tx(&bars[stage], nr * D * static_cast<int>(sizeof(T)));
    __syncwarp();
    for (int i = lane; i < nr; i += 32) {
      const int lr = r0 + i;
      const int64_t grow = unit * p.n_prompt +
                           (static_cast<int64_t>(sorted[s0 + (lr >> levels)]) << levels) +
                           (lr & ((1 << levels) - 1));
      bulk_g2s(kst + (stage * kTileRows + i) * RB, kp + grow * D, D * sizeof(T), &bars[stage]);
    }
  };
  if (warp == 0) {
    if (ntiles > 0) issue(0, 0);
    if (ntiles > 1) issue(1, 1);
  }
  uint32_t bq[4][D / 16][2];
  if constexpr (sizeof(T) == 2) {
    const int NB = (G + 7) >> 3, ng = warp >> 2;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int nb = min(ng + 2 * i, NB - 1);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        ldsm_x2(smem_u32(qs) + (nb * 8 + (lane & 7)) * RB + ks * 32 + ((lane >> 3) & 1) * 16,
                bq[i][ks]);
    }
  }
  for (int tile = 0; tile < ntiles; ++tile) {
    const int stage = tile & 1;
    int ok = 1;
    if (misc[0] == 0) ok = mbar_wait_bounded(&bars[stage], (tile >> 1) & 1, p.status) ? 1 : 0;
    if (__syncthreads_or(!ok) && tid == 0) misc[0] = 1;
    const unsigned char* buf = kst + stage * kTileRows * RB;
    const int rows_valid = min(kTileRows, R - tile * kTileRows);
    if constexpr (sizeof(T) == 2) {
      token_logits_tile<D>(buf, bq, t, tile * kTileRows, rows_valid, G,
                           static_cast<__nv_bfloat16*>(nullptr));
    } else {
      token_logits_tile<D>(buf, reinterpret_cast<const float*>(qs), t, tile * kTileRows,
                           rows_valid, G, static_cast<float*>(nullptr));
    }
    __syncthreads();
    if (warp == 0 && tile + 2 < ntiles && misc[0] == 0) {
      fence_proxy_async();
      issue(tile + 2, stage);
    }
  }
  __syncthreads();

  // ---- level loop
  int n_surv = ns;
  for (int i = tid; i < ns; i += kThreads) {
    sp[i] = sorted[s0 + i];
    sr[i] = i << levels;
  }
  __syncthreads();
  for (int j = levels - 1; j >= 0; --j) {
    for (int i = tid; i < n_surv; i += kThreads) {
      const int pos = sp[i], row = sr[i];
      cp[2 * i] = 2 * pos;
      cp[2 * i + 1] = 2 * pos + 1;
      cr[2 * i] = row;
      cr[2 * i + 1] = row + (1 << j);
    }
    const int n_cand = 2 * n_surv;
    __syncthreads();
    if (p.k[j] >= 2 * p.k[j + 1]) {  // keeps every candidate: no scoring needed
      int32_t* x = sp; sp = cp; cp = x;
      x = sr; sr = cr; cr = x;
      n_surv = n_cand;
      continue;
    }
    const int leaves = 1 << j;
    const float sc = p.scale[j];
    // Pass 1: per-query max / sum of exponentials over this CTA's candidates.
    float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
    for (int c = warp; c < n_cand; c += kWarps) {
      const float* tp = t + static_cast<int64_t>(cr[c]) * G;
      if (lane < G) {
        float acc = 0.f;
        for (int i = 0; i < leaves; ++i) acc += tp[i * G + lane];
        online_update(m0, l0, acc * sc);
      }
      if (lane + 32 < G) {
        float acc = 0.f;
        for (int i = 0; i < leaves; ++i) acc += tp[i * G + lane + 32];
        online_update(m1, l1, acc * sc);
      }
    }
    part_m[warp * 64 + lane] = m0;
    part_l[warp * 64 + lane] = l0;
    part_m[warp * 64 + lane + 32] = m1;
    part_l[warp * 64 + lane + 32] = l1;
    __syncthreads();
    if (tid < G) {
      float m = -INFINITY, l = 0.f;
      for (int w = 0; w < kWarps; ++w) merge_ml(m, l, part_m[w * 64 + tid], part_l[w * 64 + tid]);
      loc_m[tid] = m;
      loc_l[tid] = l;
    }
    cluster.sync();
    if (tid < G) {
      float m = -INFINITY, l = 0.f;
      for (int r = 0; r < cs; ++r)
        merge_ml(m, l, cluster.map_shared_rank(loc_m, r)[tid], cluster.map_shared_rank(loc_l, r)[tid]);
      gm[tid] = m;
      ginv[tid] = 1.f / l;
    }
    __syncthreads();
    // Pass 2: attention mass of every candidate.
    for (int c = warp; c < n_cand; c += kWarps) {
      const float* tp = t + static_cast<int64_t>(cr[c]) * G;
      float s = 0.f;
      if (lane < G) {
        float acc = 0.f;
        for (int i = 0; i < leaves; ++i) acc += tp[i * G + lane];
        s += expf(acc * sc - gm[lane]) * ginv[lane];
      }
      if (lane + 32 < G) {
        float acc = 0.f;
        for (int i = 0; i < leaves; ++i) acc += tp[i * G + lane + 32];
        s += expf(acc * sc - gm[lane + 32]) * ginv[lane + 32];
      }
      s = warp_sum(s);
      if (lane == 0) keys[c] = __float_as_uint(s);
    }
    __syncthreads();
    (void)cluster_topk(keys, n_cand, p.k[j], take, tk);
    n_surv = compact2(cp, cr, take, n_cand, sp, sr, tk.scan);
  }

  // ---- output: this CTA's tokens at the offset of the lower ranks
  if (tid == 0) misc[1] = n_surv;
  cluster.sync();
  int offset = 0;
  for (int r = 0; r < rank; ++r) offset += cluster.map_shared_rank(misc, r)[1];
  for (int i = tid; i < n_surv; i += kThreads)
    if (offset + i < p.budget) p.idx_out[unit * p.budget + offset + i] = sp[i];
  cluster.sync();  // peers may still read this CTA's shared memory
}

template <typename T, int D>
cudaError_t launch_typed(const LaunchDims& ld, const FilterPlan& plan, const FilterParams& prm,
                         cudaStream_t stream) {
  auto kern = recursive_filter_kernel<T, D>;
  const cudaError_t e = ensure_max_smem<recursive_filter_kernel<T, D>>();
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

template <typename T, int D>
size_t smem_for(int G, int rows_cap, int sorted_cap, bool t_in_smem) {
  return FilterSmem<T, D>(G, rows_cap, sorted_cap, t_in_smem).total;
}

size_t filter_smem(const LaunchDims& ld, int rows_cap, int sorted_cap, bool t_in_smem) {
  if (ld.dtype == WF_BF16)
    return ld.head_dim == 128 ? smem_for<__nv_bfloat16, 128>(ld.n_gen, rows_cap, sorted_cap, t_in_smem)
                              : smem_for<__nv_bfloat16, 64>(ld.n_gen, rows_cap, sorted_cap, t_in_smem);
  return ld.head_dim == 128 ? smem_for<float, 128>(ld.n_gen, rows_cap, sorted_cap, t_in_smem)
                            : smem_for<float, 64>(ld.n_gen, rows_cap, sorted_cap, t_in_smem);
}

}  // namespace

bool plan_filter(const LaunchDims& ld, const int32_t* k, FilterPlan* plan) {
  const int kL = k[ld.levels];
  const int64_t rows = static_cast<int64_t>(kL) << ld.levels;
  // About 256 token rows per CTA, at most kMaxCluster CTAs, at least one span each.
  int cs = 1;
  while (cs < kMaxCluster && rows / (2 * cs) >= 256 && kL >= 2 * cs) cs *= 2;
  plan->cluster = cs;
  plan->spans_cap = (kL + cs - 1) / cs;
  plan->rows_cap = plan->spans_cap << ld.levels;
  int sc = 1;
  while (sc < kL) sc <<= 1;
  plan->sorted_cap = sc;
  const size_t with_t = filter_smem(ld, plan->rows_cap, sc, true);
  plan->t_in_smem = with_t <= kMaxSmem;
  plan->smem_bytes = plan->t_in_smem ? with_t : filter_smem(ld, plan->rows_cap, sc, false);
  plan->t_bytes = plan->t_in_smem ? 0
                                  : sizeof(float) * static_cast<size_t>(ld.units) * cs *
                                        plan->rows_cap * ld.n_gen;
  return plan->smem_bytes <= kMaxSmem;
}

cudaError_t launch_recursive_filter(const LaunchDims& ld, const FilterPlan& plan, const void* q,
                                    const void* kp, const int32_t* idx_l, const int32_t* k,
                                    int32_t* idx, float* t_ws, int32_t* status,
                                    cudaStream_t stream) {
  FilterParams prm = {};
  prm.q = q;
  prm.kp = kp;
  prm.idx_l = idx_l;
  prm.idx_out = idx;
  prm.status = status;
  prm.t_ws = plan.t_in_smem ? nullptr : t_ws;
  prm.n_prompt = ld.n_prompt;
  prm.G = ld.n_gen;
  prm.levels = ld.levels;
  prm.kL = k[ld.levels];
  prm.budget = k[0];
  prm.spans_cap = plan.spans_cap;
  prm.rows_cap = plan.rows_cap;
  prm.sorted_cap = plan.sorted_cap;
  for (int j = 0; j <= ld.levels; ++j) {
    prm.k[j] = k[j];
    prm.scale[j] = static_cast<float>(std::pow(2.0, -0.5 * j) / std::sqrt(static_cast<double>(ld.head_dim)));
  }
  if (ld.dtype == WF_BF16) {
    if (ld.head_dim == 128) return launch_typed<__nv_bfloat16, 128>(ld, plan, prm, stream);
    return launch_typed<__nv_bfloat16, 64>(ld, plan, prm, stream);
  }
  if (ld.head_dim == 128) return launch_typed<float, 128>(ld, plan, prm, stream);
  return launch_typed<float, 64>(ld, plan, prm, stream);
}

}  // namespace wf
