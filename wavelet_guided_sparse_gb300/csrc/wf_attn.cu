// Steps 4-5: gather the sparse KV cache and attend over it.
//
// WaveFilter (arXiv 2606.00724) §2.1 eq. (3), with the cached index set I
// replaced by the selected prompt tokens S plus every generation position
// I_g (Fig. 2(d); §1: the final tokens build a sparse KV cache that takes
// part in attention with the current queries):
//   O[i] = Σ_j softmax_j(Q[i]·K_j/√d) V_j,   j over Kp[S] ∪ Kg (no mask).
//
// Design: one cluster per unit, split-KV.  The key list (B selected prompt
// rows, then G generation rows) is cut into tiles; each CTA owns a
// contiguous run of tiles.  Rows are gathered straight into padded shared
// memory by per-row bulk copies (TMA engine) in a two-stage mbarrier
// pipeline; the sparse cache is never materialised in HBM.  bf16 inputs use
// m16n8k16 tensor-core MMAs for Q·K^T and P·V with an online softmax in
// registers (P rounded to bf16, fp32 accumulation); fp32 inputs use FMAs.
// Partial (max, sum, O) triples are merged inside the CTA and then across
// the cluster through DSMEM.
#include <cmath>

#include "wf_common.cuh"
#include "wf_internal.h"

namespace wf {

namespace {

constexpr float kLn2 = 0.6931471805599453f;

struct AttnParams {
  const void* q;
  const void* kp;
  const void* vp;
  const void* kg;
  const void* vg;
  const int32_t* idx;
  float* o;
  float* lse;
  int32_t* status;
  int n_prompt, G, B, n_keys, tile_keys, n_tiles;
  float scale_log2;  // log2(e) / sqrt(d)
};

template <typename T, int D>
struct AttnSmem {
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(T)) + 16;
  // bf16 path: the per-warp partials are written after the last tile, so they
  // share bytes with the K/V stages; the fp32 path needs its scratch during
  // the tile loop.
  static constexpr bool kAliasWork = sizeof(T) == 2;
  size_t bars, qs, kst, vst, work, cta_o, cta_ml, total;
  __host__ __device__ AttnSmem(int tile_keys) {
    size_t o = 0;
    auto take_bytes = [&](size_t bytes) {
      const size_t at = o;
      o = (o + bytes + 15) & ~size_t(15);
      return at;
    };
    bars = take_bytes(2 * sizeof(uint64_t));
    qs = take_bytes(static_cast<size_t>(64) * kRowBytes);
    const size_t stage = static_cast<size_t>(2) * tile_keys * kRowBytes;
    const size_t work_bytes =
        kAliasWork ? sizeof(float) * (kWarps * 16 * D + 2 * kWarps * 16)
                   : sizeof(float) * (64 * 33 + 3 * 64);
    if (kAliasWork) {
      kst = o;
      vst = o + stage;
      work = o;
      take_bytes(2 * stage > work_bytes ? 2 * stage : work_bytes);
    } else {
      kst = take_bytes(stage);
      vst = take_bytes(stage);
      work = take_bytes(work_bytes);
    }
    cta_o = take_bytes(sizeof(float) * 64 * D);
    cta_ml = take_bytes(sizeof(float) * 2 * 64);
    total = o;
  }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Key j of the unit's list: a valid row pointer pair and whether it counts.
template <typename T, int D>
__device__ __forceinline__ bool key_source(const AttnParams& p, int64_t unit, int j, int key_end,
                                           const T** ksrc, const T** vsrc) {
  const T* kg = static_cast<const T*>(p.kg) + unit * p.G * D;
  const T* vg = static_cast<const T*>(p.vg) + unit * p.G * D;
  *ksrc = kg;
  *vsrc = vg;
  if (j >= key_end) return false;
  if (j >= p.B) {
    *ksrc = kg + static_cast<int64_t>(j - p.B) * D;
    *vsrc = vg + static_cast<int64_t>(j - p.B) * D;
    return true;
  }
  const int row = __ldg(p.idx + unit * p.B + j);
  if (row < 0 || row >= p.n_prompt) return false;
  *ksrc = static_cast<const T*>(p.kp) + (unit * p.n_prompt + row) * D;
  *vsrc = static_cast<const T*>(p.vp) + (unit * p.n_prompt + row) * D;
  return true;
}

__device__ __forceinline__ bool key_valid(const AttnParams& p, int64_t unit, int j, int key_end) {
  if (j >= key_end) return false;
  if (j >= p.B) return true;
  const int row = __ldg(p.idx + unit * p.B + j);
  return row >= 0 && row < p.n_prompt;
}

// (m, l) merge in the log2 domain; m = -inf means "nothing yet".
__device__ __forceinline__ float safe_exp2_diff(float m, float mx) {
  return m == -INFINITY ? 0.f : exp2f(m - mx);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) sparse_attn_kernel(AttnParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int64_t unit = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, TK = p.tile_keys;
  const AttnSmem<T, D> L(TK);
  constexpr int RB = AttnSmem<T, D>::kRowBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  unsigned char* qs = smem + L.qs;
  unsigned char* kst = smem + L.kst;
  unsigned char* vst = smem + L.vst;
  float* work = reinterpret_cast<float*>(smem + L.work);
  float* cta_o = reinterpret_cast<float*>(smem + L.cta_o);
  float* cta_m = reinterpret_cast<float*>(smem + L.cta_ml);
  float* cta_l = cta_m + 64;
  __shared__ int aborted;

  const int t0 = static_cast<int>((static_cast<int64_t>(rank) * p.n_tiles) / cs);
  const int t1 = static_cast<int>((static_cast<int64_t>(rank + 1) * p.n_tiles) / cs);
  const int key_begin = t0 * TK;
  const int key_end = min(t1 * TK, p.n_keys);
  const int ntiles = t1 - t0;

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
    aborted = 0;
  }
  // Bad prompt indices of this CTA's keys are reported once.
  for (int j = key_begin + tid; j < min(key_end, p.B); j += kThreads) {
    const int row = __ldg(p.idx + unit * p.B + j);
    if (row < 0 || row >= p.n_prompt) raise_flag(p.status, WF_DEV_BAD_INDEX);
  }
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

  // Every slot of a tile is filled (invalid slots with a finite dummy row) so
  // masked probabilities multiply finite values.
  auto issue = [&](int tile, int stage) {  // warp 0 only
    const int base = key_begin + tile * TK;
    if (lane == 0) mbar_arrive_expect_tx(&bars[stage], 2u * TK * D * sizeof(T));
    __syncwarp();
    for (int i = lane; i < TK; i += 32) {
      const T* ks;
      const T* vs;
      (void)key_source<T, D>(p, unit, base + i, key_end, &ks, &vs);
      bulk_g2s(kst + (stage * TK + i) * RB, ks, D * sizeof(T), &bars[stage]);
      bulk_g2s(vst + (stage * TK + i) * RB, vs, D * sizeof(T), &bars[stage]);
    }
  };
  if (warp == 0) {
    if (ntiles > 0) issue(0, 0);
    if (ntiles > 1) issue(1, 1);
  }

  if constexpr (sizeof(T) == 2) {
    // ------------------------------------------------ bf16 tensor-core path
    const int MB = G <= 16 ? 1 : (G <= 32 ? 2 : 4);
    const int mb = warp % MB, kgrp = warp / MB;  // 16 keys per warp per tile
    uint32_t qa[D / 16][4];
    {
      const uint32_t qbase = smem_u32(qs) + (mb * 16 + (lane & 15)) * RB + (lane >> 4) * 16;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) ldsm_x4(qbase + ks * 32, qa[ks]);
    }
    float oacc[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[i][e] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

    for (int tile = 0; tile < ntiles; ++tile) {
      const int stage = tile & 1;
      int ok = 1;
      if (aborted == 0) ok = mbar_wait_bounded(&bars[stage], (tile >> 1) & 1, p.status) ? 1 : 0;
      if (__syncthreads_or(!ok) && tid == 0) aborted = 1;
      const uint32_t kb = smem_u32(kst + (stage * TK + kgrp * 16) * RB);
      const uint32_t vb = smem_u32(vst + (stage * TK + kgrp * 16) * RB);
      // S = Q K^T for 16 rows x 16 keys.
      float s[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nb][e] = 0.f;
      const uint32_t kaddr = kb + ((lane & 7) + ((lane >> 4) << 3)) * RB + ((lane >> 3) & 1) * 16;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t b[4];
        ldsm_x4(kaddr + ks * 32, b);
        mma_bf16(s[0], qa[ks], b);
        mma_bf16(s[1], qa[ks], b + 2);
      }
      // Scale, mask, online softmax (rows lane/4 and lane/4 + 8).
      const int jbase = key_begin + tile * TK + kgrp * 16 + (lane & 3) * 2;
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool v = key_valid(p, unit, jbase + nb * 8 + e, key_end);
          s[nb][e] = v ? s[nb][e] * p.scale_log2 : -INFINITY;
          s[nb][e + 2] = v ? s[nb][e + 2] * p.scale_log2 : -INFINITY;
          mx_lo = fmaxf(mx_lo, s[nb][e]);
          mx_hi = fmaxf(mx_hi, s[nb][e + 2]);
        }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float base_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
      const float base_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
      const float corr_lo = exp2f(m_lo - base_lo), corr_hi = exp2f(m_hi - base_hi);
      float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s[nb][e] = exp2f(s[nb][e] - base_lo);
          s[nb][e + 2] = exp2f(s[nb][e + 2] - base_hi);
          sum_lo += s[nb][e];
          sum_hi += s[nb][e + 2];
        }
      sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, 1);
      sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, 2);
      sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, 1);
      sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, 2);
      l_lo = l_lo * corr_lo + sum_lo;
      l_hi = l_hi * corr_hi + sum_hi;
      m_lo = mn_lo;
      m_hi = mn_hi;
      uint32_t pa[4];
      pa[0] = pack_bf16(s[0][0], s[0][1]);
      pa[1] = pack_bf16(s[0][2], s[0][3]);
      pa[2] = pack_bf16(s[1][0], s[1][1]);
      pa[3] = pack_bf16(s[1][2], s[1][3]);
      const uint32_t vaddr = vb + (lane & 15) * RB + (lane >> 4) * 16;
#pragma unroll
      for (int dn = 0; dn < D / 8; dn += 2) {
        oacc[dn][0] *= corr_lo; oacc[dn][1] *= corr_lo;
        oacc[dn][2] *= corr_hi; oacc[dn][3] *= corr_hi;
        oacc[dn + 1][0] *= corr_lo; oacc[dn + 1][1] *= corr_lo;
        oacc[dn + 1][2] *= corr_hi; oacc[dn + 1][3] *= corr_hi;
        uint32_t b[4];
        ldsm_x4_t(vaddr + dn * 16, b);
        mma_bf16(oacc[dn], pa, b);
        mma_bf16(oacc[dn + 1], pa, b + 2);
      }
      __syncthreads();
      if (warp == 0 && tile + 2 < ntiles && aborted == 0) {
        fence_proxy_async();
        issue(tile + 2, stage);
      }
    }
    // Per-warp partials -> shared memory (rows of the warp's m-block).
    float* opart = work;                        // [kWarps][16][D]
    float* mpart = work + kWarps * 16 * D;      // [kWarps][16]
    float* lpart = mpart + kWarps * 16;         // [kWarps][16]
    __syncthreads();
    const int r_lo = lane >> 2;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      const int c = dn * 8 + (lane & 3) * 2;
      opart[(warp * 16 + r_lo) * D + c] = oacc[dn][0];
      opart[(warp * 16 + r_lo) * D + c + 1] = oacc[dn][1];
      opart[(warp * 16 + r_lo + 8) * D + c] = oacc[dn][2];
      opart[(warp * 16 + r_lo + 8) * D + c + 1] = oacc[dn][3];
    }
    if ((lane & 3) == 0) {
      mpart[warp * 16 + r_lo] = m_lo;
      lpart[warp * 16 + r_lo] = l_lo;
      mpart[warp * 16 + r_lo + 8] = m_hi;
      lpart[warp * 16 + r_lo + 8] = l_hi;
    }
    __syncthreads();
    const int KGW = kWarps / MB;
    for (int e = tid; e < G * D; e += kThreads) {
      const int qi = e / D, c = e % D;
      const int qmb = qi >> 4, r = qi & 15;
      float mx = -INFINITY;
      for (int g = 0; g < KGW; ++g) mx = fmaxf(mx, mpart[(qmb + MB * g) * 16 + r]);
      float acc = 0.f, l = 0.f;
      for (int g = 0; g < KGW; ++g) {
        const int w = qmb + MB * g;
        const float f = safe_exp2_diff(mpart[w * 16 + r], mx);
        acc += f * opart[(w * 16 + r) * D + c];
        l += f * lpart[w * 16 + r];
      }
      cta_o[qi * D + c] = acc;
      if (c == 0) {
        cta_m[qi] = mx;
        cta_l[qi] = l;
      }
    }
  } else {
    // ------------------------------------------------ fp32 FMA path
    constexpr int RF = RB / 4;
    float* sS = work;                   // [64][33] logits / probabilities
    float* m_run = work + 64 * 33;      // [64]
    float* l_run = m_run + 64;          // [64]
    float* corr_s = l_run + 64;         // [64]
    const float* qf = reinterpret_cast<const float*>(qs);
    constexpr int C4 = D / 4;                 // float4 columns
    constexpr int QG = kThreads / C4;         // query groups in the O phase
    constexpr int QPT = 64 / QG;              // queries per thread in the O phase
    float oacc[QPT][4];
#pragma unroll
    for (int i = 0; i < QPT; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[i][e] = 0.f;
    if (tid < 64) {
      m_run[tid] = -INFINITY;
      l_run[tid] = 0.f;
    }
    __syncthreads();
    for (int tile = 0; tile < ntiles; ++tile) {
      const int stage = tile & 1;
      int ok = 1;
      if (aborted == 0) ok = mbar_wait_bounded(&bars[stage], (tile >> 1) & 1, p.status) ? 1 : 0;
      if (__syncthreads_or(!ok) && tid == 0) aborted = 1;
      const float* kb = reinterpret_cast<const float*>(kst + stage * TK * RB);
      const float* vb = reinterpret_cast<const float*>(vst + stage * TK * RB);
      {  // logits: thread -> key (tid & 31), queries (tid >> 5) + 8i
        const int kk = tid & 31, g = tid >> 5;
        const bool v = key_valid(p, unit, key_begin + tile * TK + kk, key_end);
        for (int qi = g; qi < G; qi += 8) {
          float acc = 0.f;
          for (int c = 0; c < D; c += 4) {
            const float4 a = *reinterpret_cast<const float4*>(kb + kk * RF + c);
            const float4 b = *reinterpret_cast<const float4*>(qf + qi * RF + c);
            acc = fmaf(a.x, b.x, acc);
            acc = fmaf(a.y, b.y, acc);
            acc = fmaf(a.z, b.z, acc);
            acc = fmaf(a.w, b.w, acc);
          }
          sS[qi * 33 + kk] = v ? acc * p.scale_log2 : -INFINITY;
        }
      }
      __syncthreads();
      for (int qi = warp; qi < G; qi += kWarps) {  // row softmax update, lane = key
        const float sv = sS[qi * 33 + lane];
        const float mx = warp_max(sv);
        const float mo = m_run[qi];
        const float mn = fmaxf(mo, mx);
        const float base = mn == -INFINITY ? 0.f : mn;
        const float pv = exp2f(sv - base);
        const float sum = warp_sum(pv);
        sS[qi * 33 + lane] = pv;
        if (lane == 0) {
          const float corr = exp2f(mo - base);
          corr_s[qi] = corr;
          l_run[qi] = l_run[qi] * corr + sum;
          m_run[qi] = mn;
        }
      }
      __syncthreads();
      {
        const int c4 = tid % C4, qg = tid / C4;
#pragma unroll
        for (int i = 0; i < QPT; ++i) {
          const int qi = qg + QG * i;
          if (qi >= G) continue;
          const float corr = corr_s[qi];
          float a0 = oacc[i][0] * corr, a1 = oacc[i][1] * corr, a2 = oacc[i][2] * corr,
                a3 = oacc[i][3] * corr;
          for (int kk = 0; kk < TK; ++kk) {
            const float pv = sS[qi * 33 + kk];
            const float4 vv = *reinterpret_cast<const float4*>(vb + kk * RF + c4 * 4);
            a0 = fmaf(pv, vv.x, a0);
            a1 = fmaf(pv, vv.y, a1);
            a2 = fmaf(pv, vv.z, a2);
            a3 = fmaf(pv, vv.w, a3);
          }
          oacc[i][0] = a0; oacc[i][1] = a1; oacc[i][2] = a2; oacc[i][3] = a3;
        }
      }
      __syncthreads();
      if (warp == 0 && tile + 2 < ntiles && aborted == 0) {
        fence_proxy_async();
        issue(tile + 2, stage);
      }
    }
    {
      const int c4 = tid % C4, qg = tid / C4;
#pragma unroll
      for (int i = 0; i < QPT; ++i) {
        const int qi = qg + QG * i;
        if (qi >= G) continue;
        *reinterpret_cast<float4*>(cta_o + qi * D + c4 * 4) =
            make_float4(oacc[i][0], oacc[i][1], oacc[i][2], oacc[i][3]);
      }
      if (tid < G) {
        cta_m[tid] = m_run[tid];
        cta_l[tid] = l_run[tid];
      }
    }
  }

  // ---- merge the CTAs of the cluster; rank r finalises a slice of query rows
  cluster.sync();
  const int q0 = (rank * G) / cs, q1 = ((rank + 1) * G) / cs;
  for (int e = q0 * D + tid; e < q1 * D; e += kThreads) {
    const int qi = e / D, c = e % D;
    float mx = -INFINITY;
    for (int r = 0; r < cs; ++r) mx = fmaxf(mx, cluster.map_shared_rank(cta_m, r)[qi]);
    float acc = 0.f, l = 0.f;
    for (int r = 0; r < cs; ++r) {
      const float f = safe_exp2_diff(cluster.map_shared_rank(cta_m, r)[qi], mx);
      acc += f * cluster.map_shared_rank(cta_o, r)[qi * D + c];
      l += f * cluster.map_shared_rank(cta_l, r)[qi];
    }
    p.o[(unit * G + qi) * D + c] = acc / l;
    if (c == 0 && p.lse != nullptr) p.lse[unit * G + qi] = (mx + log2f(l)) * kLn2;
  }
  cluster.sync();  // peers may still read this CTA's shared memory
}

template <typename T, int D>
cudaError_t launch_typed(const LaunchDims& ld, const AttnPlan& plan, const AttnParams& prm,
                         cudaStream_t stream) {
  auto kern = sparse_attn_kernel<T, D>;
  const cudaError_t e = ensure_max_smem<sparse_attn_kernel<T, D>>();
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

bool plan_attn(const LaunchDims& ld, int budget, AttnPlan* plan) {
  const int G = ld.n_gen;
  int tk;
  if (ld.dtype == WF_BF16) {
    const int mb = G <= 16 ? 1 : (G <= 32 ? 2 : 4);
    tk = 16 * (kWarps / mb);
  } else {
    tk = 32;
  }
  const int n_keys = budget + G;
  plan->tile_keys = tk;
  plan->n_tiles = (n_keys + tk - 1) / tk;
  plan->cluster = plan->n_tiles < kMaxCluster ? plan->n_tiles : kMaxCluster;
  if (ld.dtype == WF_BF16)
    plan->smem_bytes = ld.head_dim == 128 ? AttnSmem<__nv_bfloat16, 128>(tk).total
                                          : AttnSmem<__nv_bfloat16, 64>(tk).total;
  else
    plan->smem_bytes = ld.head_dim == 128 ? AttnSmem<float, 128>(tk).total
                                          : AttnSmem<float, 64>(tk).total;
  return plan->smem_bytes <= kMaxSmem;
}

cudaError_t launch_sparse_attn(const LaunchDims& ld, const AttnPlan& plan, const void* q,
                               const void* kp, const void* vp, const void* kg, const void* vg,
                               const int32_t* idx, int budget, float* o, float* lse,
                               int32_t* status, cudaStream_t stream) {
  AttnParams prm = {};
  prm.q = q;
  prm.kp = kp;
  prm.vp = vp;
  prm.kg = kg;
  prm.vg = vg;
  prm.idx = idx;
  prm.o = o;
  prm.lse = lse;
  prm.status = status;
  prm.n_prompt = ld.n_prompt;
  prm.G = ld.n_gen;
  prm.B = budget;
  prm.n_keys = budget + ld.n_gen;
  prm.tile_keys = plan.tile_keys;
  prm.n_tiles = plan.n_tiles;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(ld.head_dim)));
  if (ld.dtype == WF_BF16) {
    if (ld.head_dim == 128) return launch_typed<__nv_bfloat16, 128>(ld, plan, prm, stream);
    return launch_typed<__nv_bfloat16, 64>(ld, plan, prm, stream);
  }
  if (ld.head_dim == 128) return launch_typed<float, 128>(ld, plan, prm, stream);
  return launch_typed<float, 64>(ld, plan, prm, stream);
}

}  // namespace wf
