// The WaveFilter path in one thread-block-cluster kernel (steps 2-5, and
// step 1 too where a CTA's coarse slice is small enough).
//
// WaveFilter (arXiv 2606.00724):
//  * step 1, §2.2 eq. (5) + pyramid, §3.1: A_L = 2^(-L/2) x span sums of K_p;
//  * step 2, Fig. 2(c) / §1: score the low-frequency keys A_L against the
//    generation-block queries with the eq. (3) logits and keep a coarse Top-K;
//  * step 3, Fig. 2(d) / §1: multi-scale recursive filtering — children of
//    the survivors are re-scored level by level down to tokens;
//  * steps 4-5, Fig. 2(d) / §2.1 eq. (3): the selected prompt tokens plus all
//    generation positions form a sparse KV cache that the queries attend.
// Score of a candidate c among the candidate set C at level j (attention
// mass): z[i,c] = Q[i]·A_j[c]/√d,  s[c] = Σ_i softmax_{c∈C}(z[i,·])[c].
//
// One cluster of `cs` CTAs handles one (sequence, head) unit; the kernel runs
// any contiguous subset of the phases (score / filter / attend), which is how
// wf_score_topk, wf_recursive_filter, wf_sparse_gather_attn, wf_step and
// wf_step_cached_al share it.  Between phases the work is rebalanced across
// the cluster through DSMEM: the coarse survivors are all-gathered (every CTA
// then takes an equal slice) and the final tokens are pushed to the CTA that
// attends over their slot of the key list.
//
// Phase details:
//  step 1 — (fused plans) each CTA streams the spans of its P/cs coarse
//           positions through a ring of bulk copies and writes A_L straight
//           into shared memory as hi/mid/lo bf16 planes.
//  score  — z = Q·A_L^T per CTA slice: with the fused stream, bf16 on the
//           fifth-generation tensor cores (tcgen05.mma, accumulators in
//           tensor memory, three bf16 planes reproduce fp32 A_L), fp32 by
//           FMAs; otherwise read from the coarse logits the streaming launch
//           (or the cached-A_L logits kernel) wrote; per-query (max, sum)
//           merged over the cluster; every CTA selects the coarse Top-K.
//  filter — by linearity Q·A_j[c] = 2^(-j/2) Σ_{n∈span(c)} Q·Kp[n]: token
//           logits t = Kp[rows]·Q^T are computed once (tcgen05, exact bf16
//           products, fp32 sums) for the rows under this CTA's coarse
//           survivors, fetched by 2-D tensor copies of whole spans (or 16-byte
//           cp.async) into the 128-byte-swizzled operand layout; levels that
//           keep every child are skipped, the others sum t over leaves.
//  attend — split-KV: each CTA gathers the K/V rows of its key slot range by
//           cp.async, runs Q·K^T and P·V on tensor cores (mma.sync) with an
//           online softmax, and the partial (max, sum, O) rows are pushed to
//           the CTA that finalises those query rows.
#include <algorithm>
#include <climits>
#include <cmath>

#include <cuda.h>

#include "wf_common.cuh"
#include "wf_internal.h"
#include "wf_mma.cuh"
#include "wf_umma.cuh"

namespace wf {

namespace {

constexpr int kTileRows = 64;    // filter: token rows per staged tile
constexpr int kScoreChunk = 64;  // score: coarse positions per staged chunk (fused step 1)
constexpr int kZRows = 256;      // score: coarse-logit rows per staged chunk (from global)
static_assert(kScoreChunk == 8 * kWarps, "score pass 1 takes eight rows per warp per chunk");
constexpr int kFuseStages = 3;               // fused step 1: bulk-copy ring depth
constexpr int kFuseStageBytes = 32 * 1024;   // fused step 1: bytes per ring stage
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum : int { kModeScore = 1, kModeFilter = 2, kModeAttend = 4 };

struct PathParams {
  // K_p as a 2-D tensor [units * N_p rows, d columns] for tensor copies of whole
  // spans (box: 64 columns x 2^L rows, 128-byte swizzle); valid if use_tma_spans.
  alignas(64) CUtensorMap tmap_spans;
  // A cached fp32 A_L as a 2-D tensor [units * P rows, d columns] (box: 32
  // columns x 64 rows, 128-byte swizzle); valid if al_stage.
  alignas(64) CUtensorMap tmap_al;
  int use_tma_spans;
  const void* q;
  const void* kp;
  const void* vp;
  const void* kg;
  const void* vg;
  const float* zl;           // score without the fused stream: coarse logits [U, P, GZ]
  const float* al;           // or an fp32 A_L [U, P, d] whose logits this kernel forms
  const int32_t* idx_l_in;   // filter without score: S_L [U, k_L]
  const int32_t* idx_in;     // attend without filter: S [U, B]
  int32_t* idx_l_out;        // score without filter: S_L out [U, k_L]
  float* scores_out;         // nullable [U, P]
  int32_t* idx_out;          // nullable in path mode [U, B]
  float* o;
  float* lse;                // nullable [U, G]
  int32_t* status;
  float* t_ws;               // token logits in global memory (nullptr: shared)
  int mode;
  int n_prompt, G, GZ, levels, P, kL, budget, n_keys;
  int cs, per_cta_p, rows_cap, sorted_cap, keys_cap, gather_all, klist_cap, tile_keys;
  int f_stages, a_stages;  // ring depths (filter tiles, attention tiles)
  int filter_fast;         // token logits: 0 general path; 1 tensor-memory resident; 2 streamed twice
  int f_nb;                // fast filter: tensor-memory accumulator slots
  int fuse_dwt;            // score: A_L from K_p inside this kernel
  int al_stage;            // score: this CTA's rows of the cached fp32 A_L arrive by bulk
                           // copies, 64 rows a stage (per_cta_p <= kZRows), through a
                           // ring of al_ring stages (every stage resident when it fits)
  int al_ring;
  uint32_t inject_polls;   // fault injection (tests): see the fused step 1 below
  float al_scale;          // 2^(-L/2), the orthonormal Haar low-pass gain
  int k[WF_MAX_LEVELS + 1];
  float scale[WF_MAX_LEVELS + 1];  // 2^(-j/2)/sqrt(d)
  float inv_sqrt_d, scale_log2;
};

template <typename T, int D>
struct PathSmem {
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(T)) + 16;  // padded row pitch
  static constexpr int kRowF = D + 4;                                      // fp32 row pitch
  size_t qs, stat_in, gm, loc, part, cnt_a, cnt_b, misc, bars, sl_all, sp, sr, cp, cr, keys,
      take, topk, keys_all, pos_all, klist;
  size_t s_stage, s_as, s_z, s_ring;  // score phase
  size_t f_kst, f_t;               // filter phase (general path)
  size_t f_ring, f_stage, f_bars, f_gather;  // filter phase (fast path)
  size_t a_kst, a_vst, a_work, a_recv, a_rml;  // attend phase
  size_t total;
  __host__ __device__ explicit PathSmem(const PathParams& p) {
    size_t o = 0;
    auto take_bytes = [&](size_t bytes, size_t align = 16) {
      o = (o + align - 1) & ~(align - 1);
      const size_t at = o;
      o = (o + bytes + 15) & ~size_t(15);
      return at;
    };
    sp = sr = cp = cr = keys = take = 0;
    f_kst = f_t = f_ring = f_stage = f_bars = f_gather = 0;
    qs = take_bytes(static_cast<size_t>(kMaxQ) * kRowBytes);
    stat_in = take_bytes(sizeof(float) * kMaxCluster * 2 * kMaxQ);
    gm = take_bytes(sizeof(float) * 2 * kMaxQ);
    loc = take_bytes(sizeof(float) * 2 * kMaxQ);
    part = take_bytes(sizeof(float) * 2 * kWarps * kMaxQ);
    cnt_a = take_bytes(sizeof(int32_t) * kMaxCluster);
    cnt_b = take_bytes(sizeof(int32_t) * kMaxCluster);
    misc = take_bytes(sizeof(int32_t) * 8);
    bars = take_bytes(sizeof(uint64_t) * (kFuseStages + 2));  // ring, tensor-core commits, span copies
    sl_all = take_bytes(sizeof(int32_t) * p.sorted_cap);
    topk = take_bytes(sizeof(TopkSmem));
    // All-gathered keys: the P coarse scores, and (final level, gather mode)
    // every CTA's candidates with their positions.
    // (The fast filter keeps its all-gather buffers in its own region.)
    const size_t gather_n =
        p.gather_all && !p.filter_fast ? static_cast<size_t>(p.cs) * p.rows_cap : 0;
    const size_t score_n = (p.mode & kModeScore) ? static_cast<size_t>(p.P) : 0;
    keys_all = take_bytes(sizeof(uint32_t) * (gather_n > score_n ? gather_n : score_n));
    pos_all = take_bytes(sizeof(int32_t) * gather_n);
    klist = take_bytes(sizeof(int32_t) * p.klist_cap);
    const size_t u = o;
    size_t end = u;
    s_ring = 0;
    if ((p.mode & kModeScore) && p.fuse_dwt) {
      // Fused step 1: the bulk-copy ring of K_p rows, then A_L in the tile
      // operand layout (bf16: hi / mid / lo planes; fp32: rows).  The logits
      // overwrite the ring once every stage has been consumed.
      o = u;
      s_ring = take_bytes(static_cast<size_t>(kFuseStages) * kFuseStageBytes);
      s_as = take_bytes((sizeof(T) == 2 ? 3 : 1) * kScoreChunk * kRowBytes, 1024);
      s_stage = s_z = s_ring;
      end = end > o ? end : o;
    } else if ((p.mode & kModeScore) && p.al_stage) {
      // Cached A_L by bulk copies of 64 fp32 rows: one stage, which the
      // logits then overwrite, when the CTA has at most 64 positions; else a
      // ring of kFuseStages stages with the logits tile beside it.
      o = u;
      const size_t stage_b = sizeof(float) * kScoreChunk * D;
      const size_t z_b = sizeof(float) * static_cast<size_t>(p.per_cta_p) * (p.G | 1);
      if (p.per_cta_p <= kScoreChunk) {
        s_ring = take_bytes(stage_b > z_b ? stage_b : z_b, 1024);
        s_z = s_ring;
      } else {
        s_ring = take_bytes(static_cast<size_t>(p.al_ring) * stage_b, 1024);
        s_z = take_bytes(z_b);
      }
      s_stage = s_as = s_ring;
      end = end > o ? end : o;
    } else if (p.mode & kModeScore) {
      // Coarse logits of up to kZRows positions, padded rows of GZ + 4 floats.
      o = u;
      s_z = take_bytes(sizeof(float) * static_cast<size_t>(p.per_cta_p < kZRows ? p.per_cta_p : kZRows) *
                       (p.GZ + 4));
      s_stage = s_as = s_z;
      end = end > o ? end : o;
    }
    if ((p.mode & kModeFilter) && p.filter_fast) {
      // Ring of 128-row key tiles in the swizzled operand layout, the staging
      // tile of the statistics pass, row scores, selection flags, survivors.
      // The all-gather of (score, position) pairs for the final selection
      // starts after every CTA's statistics pass: with resident logits the
      // ring is idle by then and holds it; otherwise it has its own bytes.
      o = u;
      f_kst = f_t = 0;
      const size_t ring_b = static_cast<size_t>(p.f_stages) * D * 256;
      const size_t gath_b = p.gather_all ? sizeof(uint32_t) * 2 * static_cast<size_t>(p.cs) * p.rows_cap : 0;
      // The distributed selection's flags and survivor list are formed after
      // the last tile has been consumed, so they overlay the ring as well.
      const bool overlay = p.filter_fast == 1;
      const size_t sel_b = static_cast<size_t>(p.rows_cap) * (sizeof(int32_t) + 1);
      size_t ring_sz = ring_b > sel_b ? ring_b : sel_b;
      if (overlay && gath_b > ring_sz) ring_sz = gath_b;
      f_ring = take_bytes(ring_sz, 1024);
      f_gather = overlay ? f_ring : (gath_b ? take_bytes(gath_b) : 0);
      sp = f_ring;
      take = f_ring + sizeof(int32_t) * static_cast<size_t>(p.rows_cap);
      // The statistics pass's staging tile is done before the scores are
      // formed: the row scores share its bytes.
      const size_t stage_b = sizeof(float) * 128 * static_cast<size_t>(p.GZ + 4);
      const size_t keys_b = sizeof(uint32_t) * static_cast<size_t>(p.rows_cap);
      f_stage = take_bytes(stage_b > keys_b ? stage_b : keys_b);
      keys = f_stage;
      f_bars = take_bytes(sizeof(uint64_t) * (p.f_stages + 2 * p.f_nb), 8);
      end = end > o ? end : o;
    } else if (p.mode & kModeFilter) {
      o = u;
      f_ring = f_stage = f_bars = f_gather = 0;
      f_kst = take_bytes(static_cast<size_t>(p.f_stages) * kTileRows * kRowBytes, 1024);
      sp = take_bytes(sizeof(int32_t) * p.rows_cap);  // survivor / candidate lists
      sr = take_bytes(sizeof(int32_t) * p.rows_cap);
      cp = take_bytes(sizeof(int32_t) * p.rows_cap);
      cr = take_bytes(sizeof(int32_t) * p.rows_cap);
      keys = take_bytes(sizeof(uint32_t) * p.keys_cap);
      take = take_bytes(p.keys_cap);
      f_t = p.t_ws == nullptr ? take_bytes(sizeof(float) * static_cast<size_t>(p.rows_cap) * (p.G | 1)) : 0;
      end = end > o ? end : o;
    }
    if (p.mode & kModeAttend) {
      o = u;
      const size_t stage = static_cast<size_t>(p.a_stages) * p.tile_keys * kRowBytes;
      if (sizeof(T) == 2) {  // warp partials overwrite the stages after the last tile
        const size_t work = sizeof(float) * (kWarps * 16 * (D + 8) + 2 * kWarps * 16 + kMaxQ * kWarps);
        a_kst = o;
        a_vst = o + stage;
        a_work = o;
        take_bytes(2 * stage > work ? 2 * stage : work);
      } else {
        a_kst = take_bytes(stage);
        a_vst = take_bytes(stage);
        a_work = take_bytes(sizeof(float) * (kMaxQ * 33 + 3 * kMaxQ));
      }
      const int rpo = (p.G + p.cs - 1) / p.cs;  // query rows finalised per CTA
      a_recv = take_bytes(sizeof(float) * static_cast<size_t>(p.cs) * rpo * D);
      a_rml = take_bytes(sizeof(float) * static_cast<size_t>(p.cs) * rpo * 2);
      end = end > o ? end : o;
    }
    total = end;
  }
};

struct Ctx {
  int cs, rank, tid, lane, warp;
  int64_t unit;
};

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ int key_slot_start(int r, int cs, int n_keys) {
  return static_cast<int>((static_cast<int64_t>(r) * n_keys) / cs);
}
__device__ __forceinline__ int key_slot_owner(int g, int cs, int n_keys) {
  int r = cs - 1;
  while (r > 0 && key_slot_start(r, cs, n_keys) > g) --r;
  return r;
}

// Selection among this CTA's candidates (keys[0..n)), exact over the cluster.
__device__ __forceinline__ TopkResult cluster_select(const uint32_t* keys, int n, int k,
                                                     uint8_t* take, TopkSmem& tk) {
  return topk_distributed(keys, n, k, take, tk);
}

// ------------------------------------------------------------------ logits GEMM
// bf16 logits tile on the fifth-generation tensor cores:
//   out[(row0 + r) * pitch + q] = scale * Σ_planes Σ_k A_p[r][k] * Q[q][k]
// for r < rows and q < G.  A (nplanes planes plane_bytes apart, summed: one
// plane for key rows; hi + mid + lo planes reproduce an fp32 row exactly) is
// bf16 in the 128-byte-swizzled layout with m_alloc rows per column block;
// Q is bf16 in the core-matrix layout (8-row groups 16 * D bytes apart).
// The rows go in 128-row (M = 128) pieces, then 64-row (M = 64) pieces, each
// into its own tensor-memory accumulator of N = G rounded up to 16 columns;
// one thread issues every MMA, one commit signals `bar`, and the warps read
// the accumulators back (M = 128: row = lane of the warp's lane quarter;
// M = 64: rows 16q + l in lanes 32q + l, l < 16).  Rows up to the next
// multiple of 64 are read from shared memory.  Block-wide; every thread keeps
// the same `phase` count of completed commits on `bar`.
template <int D>
__device__ __noinline__ void umma_logits(const unsigned char* a, int nplanes, int plane_bytes,
                                         int m_alloc, int rows, const unsigned char* qs, int G,
                                         float* out, int row0, int pitch, float scale,
                                         uint32_t tmem, uint64_t* bar, uint32_t& phase,
                                         int32_t* status) {
  constexpr int SBO = D * 16;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int N = (G + 15) & ~15;
  fence_proxy_async();  // operands written through the generic proxy
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t a0 = smem_u32(a), q0 = smem_u32(qs);
    int piece = 0;
    for (int r0 = 0; r0 < rows; r0 += rows - r0 >= 128 ? 128 : 64, ++piece) {
      const int m = rows - r0 >= 128 ? 128 : 64;
      const uint32_t idesc = umma_idesc_bf16(m, N);
      for (int pl = 0; pl < nplanes; ++pl)
        for (int ks = 0; ks < D / 16; ++ks)
          umma_bf16(tmem + piece * N,
                    umma_desc_sw128(a0 + pl * plane_bytes + ((ks * 16) >> 6) * (m_alloc * 128) +
                                    (r0 >> 3) * 1024 + ((ks * 16) & 63) * 2),
                    umma_desc(q0 + ks * 256, 128, SBO), idesc, (pl | ks) != 0);
    }
    umma_commit(bar);
  }
  const bool ok = mbar_wait_bounded(bar, phase & 1u, status);
  // The count advances even after a wait gave up: the commit still completes
  // this phase when the multiply ends, so the next wait is for the next
  // commit; if it never comes, every later wait gives up as well.
  ++phase;
  tc_fence_after();
  if (ok) {
    const int q4 = warp & 3;
    int piece = 0;
    for (int r0 = 0; r0 < rows; r0 += rows - r0 >= 128 ? 128 : 64, ++piece) {
      const int m = rows - r0 >= 128 ? 128 : 64;
      const int r = m == 128 ? q4 * 32 + lane : q4 * 16 + (lane & 15);
      const bool has = (m == 128 || lane < 16) && r0 + r < rows;
      float* dst = out + static_cast<int64_t>(row0 + r0 + r) * pitch;
      for (int c = (warp >> 2) * 16; c < N; c += 32) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(q4 * 32) << 16) + piece * N + c, v);
        if (has) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c + i < G) dst[c + i] = v[i] * scale;
        }
      }
    }
  }
  tc_fence_before();  // later MMAs into these columns follow these reads
}

// fp32: plain FMAs.  Thread -> row (tid & 63), queries (tid >> 6) + 4i.
template <int D>
__device__ __forceinline__ void logits_tile_f32(const unsigned char* kst, const float* qs,
                                                float* t, int row0, int rows_valid, int G,
                                                int pitch, float scale) {
  constexpr int RF = D + 4;
  const int r = threadIdx.x & 63, g = threadIdx.x >> 6;
  if (r >= rows_valid) return;
  const float* krow = reinterpret_cast<const float*>(kst) + r * RF;
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
  float* dst = t + static_cast<int64_t>(row0 + r) * pitch;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (g + 4 * i < G) dst[g + 4 * i] = acc[i] * scale;
}

// Running (max, Σ 2^(z - max)) update (log2 domain) with 8 logits at once
// (entries that do not exist are -inf); the 8 loads and exponentials are
// independent, so one warp keeps them in flight together.
__device__ __forceinline__ void online8(float& m, float& l, const float (&z)[8]) {
  float cm = m;
#pragma unroll
  for (int u = 0; u < 8; ++u) cm = fmaxf(cm, z[u]);
  if (cm == -INFINITY) return;
  float acc = l * fast_exp2(m - cm);
#pragma unroll
  for (int u = 0; u < 8; ++u) acc += fast_exp2(z[u] - cm);
  l = acc;
  m = cm;
}

// Waits until at most `pending` of this thread's most recent cp.async groups
// are still in flight (0 <= pending < 8).
__device__ __forceinline__ void cp_async_wait_pending(int pending) {
  switch (pending) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    default: cp_async_wait<7>(); break;
  }
}

__device__ __forceinline__ float safe_exp2_diff(float m, float mx) {
  return m == -INFINITY ? 0.f : fast_exp2(m - mx);
}

// Prompt row of key slot g (g < B) of this unit, or -1 if out of range.
// klist holds the rows of this CTA's slots [k0, k1): the filter's list, or
// the caller's copied there at the start of the attend phase.
__device__ __forceinline__ int prompt_row(const PathParams& p, const int32_t* klist, int k0,
                                          int g) {
  const int row = klist[g - k0];
  return (row >= 0 && row < p.n_prompt) ? row : -1;
}

// Key slots of one CTA's attention: slot g < B is prompt row idx[g] (the
// filter's list or the caller's), B <= g < n_keys generation row g - B.
template <typename T>
struct AttnRows {
  const T *kg, *vg, *kp, *vp;  // this unit's rows
  const int32_t* klist;
  int k0, k1, B;               // this CTA's slots [k0, k1)
};

template <typename T>
__device__ __forceinline__ bool attn_key_valid(const PathParams& p, int mode, const Ctx& c,
                                               const AttnRows<T>& ar, int g) {
  if (g >= ar.k1) return false;
  if (g >= ar.B) return true;
  return prompt_row(p, ar.klist, ar.k0, g) >= 0;
}

// Gathers the key and value rows of slots [k0 + tile TK, ...) into ring stage
// `stage` by 16-byte cp.async (one commit group; all threads).
template <typename T, int D>
__device__ __forceinline__ void attn_issue(const PathParams& p, int mode, const Ctx& c,
                                           const AttnRows<T>& ar, unsigned char* kst,
                                           unsigned char* vst, int TK, int tile, int stage) {
  constexpr int C16 = D * static_cast<int>(sizeof(T)) / 16;
  constexpr int RB = PathSmem<T, D>::kRowBytes;
  const int base = ar.k0 + tile * TK;
  // Not unrolled: the loop runs once per tile between other phases' code, and
  // its smaller body costs fewer instruction fetches.
#pragma unroll 1
  for (int e = threadIdx.x; e < TK * C16; e += kThreads) {
    const int i = e / C16, ch = e % C16;
    const int g = base + i;
    const T* ks = ar.kg;
    const T* vs = ar.vg;
    if (g < ar.k1) {
      if (g >= ar.B) {
        ks = ar.kg + static_cast<int64_t>(g - ar.B) * D;
        vs = ar.vg + static_cast<int64_t>(g - ar.B) * D;
      } else {
        const int row = prompt_row(p, ar.klist, ar.k0, g);
        if (row >= 0) {
          ks = ar.kp + static_cast<int64_t>(row) * D;
          vs = ar.vp + static_cast<int64_t>(row) * D;
        }
      }
    }
    cp_async16(kst + (stage * TK + i) * RB + ch * 16, reinterpret_cast<const unsigned char*>(ks) + ch * 16);
    cp_async16(vst + (stage * TK + i) * RB + ch * 16, reinterpret_cast<const unsigned char*>(vs) + ch * 16);
  }
  cp_async_commit();
}

// Producer of the fast filter (one thread): fills a ring of S 128-row tiles
// by 2-D tensor copies (whole spans of the coarse survivors, 128-byte
// swizzle) and issues one tcgen05.mma pass per tile into tensor-memory slot
// g % NB (N columns each), committing to done[slot]; a slot is reused once
// the consumers released it (empty[slot]).  Tiles g >= ntiles are the second
// pass over the same rows.  Every wait is bounded; on a timeout the producer
// stops issuing, sets *abort, waits (bounded) for the copies it issued and
// the last multiply, and returns.
template <int D>
struct FilterProducer {
  static constexpr int TR = 128;
  static constexpr int kStageBytes = D * 256;
  unsigned char* ring;
  uint64_t *full, *done;
  const void* tmap;
  const int32_t* sl;
  const unsigned char* qs;
  int32_t* status;
  volatile int32_t* abort;
  uint32_t tmem;
  int s0, levels, row_base, R, ntiles, total, S, NB, N;
  int next_tma = 0, g_mma = 0, g_full = 0;
  bool ok = true;

  __device__ __forceinline__ void copy_tile(int g) {
    const int t = g % ntiles, st = g % S;
    const int box_rows = min(1 << levels, TR);
    const int rows = min(TR, R - t * TR);
    mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(rows) * D * 2);
    for (int b = 0; b * box_rows < rows; ++b) {
      const int lr = t * TR + b * box_rows;
      const int y = row_base + (sl[s0 + (lr >> levels)] << levels) + (lr & ((1 << levels) - 1));
      for (int kb = 0; kb < D / 64; ++kb)
        tma_load_2d(ring + st * kStageBytes + kb * (TR * 128) + b * box_rows * 128, tmap, kb * 64,
                    y, &full[st]);
    }
  }

  __device__ __forceinline__ void run(int g_end) {
    if (next_tma == 0)
      for (; next_tma < min(S, total); ++next_tma) copy_tile(next_tma);
    const uint32_t q0 = smem_u32(qs);
    const uint32_t idesc = umma_idesc_bf16(TR, N);
    int g = g_mma;
    for (; ok && g < g_end; ++g) {
      const int st = g % S, slot = g % NB;
      ok = mbar_wait_bounded(&full[st], static_cast<uint32_t>((g / S) & 1), status);
      if (!ok) break;
      g_full = g + 1;
      if (g >= NB) ok = mbar_wait_bounded(&empty_bar(slot), static_cast<uint32_t>(((g / NB) - 1) & 1), status);
      if (!ok) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(ring + st * kStageBytes);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        umma_bf16(tmem + slot * N, umma_desc_sw128(a0 + ((ks * 16) >> 6) * (TR * 128) + ((ks * 16) & 63) * 2),
                  umma_desc(q0 + ks * 256, 128, D * 16), idesc, ks != 0);
      umma_commit(&done[slot]);
      // Refill a stage once the multiply that read it has finished: that of
      // tile g - 1 (so tile g's multiply is queued behind it meanwhile), or
      // with a single stage that of tile g itself.
      const int j = S > 1 ? g - 1 : g;
      if (j >= 0 && j + S < total) {
        ok = mbar_wait_bounded(&done[j % NB], static_cast<uint32_t>((j / NB) & 1), status);
        if (!ok) {
          ++g;
          break;
        }
        copy_tile(next_tma++);  // tile j + S into stage j % S
      }
    }
    g_mma = g;
    if (!ok) {
      *abort = 1;
      for (int h = g_full; h < next_tma; ++h)
        (void)mbar_wait_bounded(&full[h % S], static_cast<uint32_t>((h / S) & 1), status);
      if (g_mma > 0)
        (void)mbar_wait_bounded(&done[(g_mma - 1) % NB], static_cast<uint32_t>(((g_mma - 1) / NB) & 1),
                                status);
      g_full = next_tma;
    }
  }
  __device__ __forceinline__ uint64_t& empty_bar(int slot) { return done[NB + slot]; }
};

// Token position of row `row` of a CTA's span rows (survivor spans
// sl[s0 ..], 2^levels rows each).
__device__ __forceinline__ int span_token(const int32_t* sl, int s0, int row, int levels) {
  return (sl[s0 + (row >> levels)] << levels) + (row & ((1 << levels) - 1));
}

// Attention mass of the token whose logits sit in this thread's tensor-memory
// lane at taddr (N columns, the G queries first): Σ_q 2^(v_q sc2 - gm_q) /
// sum_q, with four partial sums in a fixed order.  Sixteen columns per
// iteration keep the loop body (and the code to fetch) small.
// Warp-collective.
__device__ __forceinline__ float token_score_tmem(uint32_t taddr, int N, int G, float sc2,
                                                  const float* gm, const float* ginv) {
  float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int c = 0; c < N; c += 16) {
    float v[16];
    tmem_ld16(taddr + c, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int q = c + i;
      if (q < G) sq[i & 3] += fast_exp2(v[i] * sc2 - gm[q]) * ginv[q];
    }
  }
  return (sq[0] + sq[1]) + (sq[2] + sq[3]);
}

// Copies the first `cols` (a multiple of 4) logits of this thread's lane at
// taddr to dst (fp32, 16-byte aligned) if `store`.  Warp-collective.
__device__ __forceinline__ void tmem_row_to_smem(uint32_t taddr, int N, int cols, bool store,
                                                 float* dst) {
#pragma unroll 1
  for (int c = 0; c < N; c += 16) {
    float v[16];
    tmem_ld16(taddr + c, v);
    if (store) {
#pragma unroll
      for (int i = 0; i < 16; i += 4)
        if (c + i < cols) *reinterpret_cast<float4*>(dst + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
  }
}

// Coarse logits of `rows` (<= 128) rows of an fp32 A_L in shared memory
// (64-row stages one after another, each in the 128-byte-swizzled layout of
// 32-column blocks a tensor copy writes) against the unit's queries in the
// tensor-core operand layout (qs, bf16, rows >= G zero), into z (row pitch
// `pitch`, scaled by zscale), on the warps' mma.sync units: each A_L value is
// split exactly into three bf16 parts in registers, whose products with the
// bf16 queries are exact (fp32 accumulation).  Warp w takes rows 16w .. 16w
// + 15 against every query tile, so each value is split once; for at most 64
// rows warps w and w + 4 share a row tile and take alternate query tiles
// instead (all eight warps busy).  z may overlay
// the A_L rows: every warp has read its rows (block barrier) before any
// result is stored.  Block-wide (every thread calls it).
template <int D>
__device__ __forceinline__ void coarse_logits_ring(const float* a, int rows, const unsigned char* qs,
                                                   int G, float* z, int pitch, float zscale) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gid = lane >> 2, tig = lane & 3;
  const bool shared_rows = rows <= 64;
  const int rb = 16 * (shared_rows ? (warp & 3) : warp);
  const int t0 = shared_rows ? (warp >> 2) : 0, tstep = shared_rows ? 2 : 1;  // query tiles
  const int NT = (G + 7) >> 3;
  constexpr int kMaxTiles = 8;  // G <= 64
  float c[kMaxTiles][4];
#pragma unroll
  for (int t = 0; t < kMaxTiles; ++t)
#pragma unroll
    for (int e = 0; e < 4; ++e) c[t][e] = 0.f;
  if (rb < rows) {
    const bool r0ok = rb + gid < rows, r1ok = rb + gid + 8 < rows;
    // Element (r, k): stage r / 64, then 16-byte chunk k / 4 of row r % 64.
    const unsigned char* ab = reinterpret_cast<const unsigned char*>(a) +
                              static_cast<size_t>(rb >> 6) * kScoreChunk * D * sizeof(float);
    const int r0 = (rb & 63) + gid, r1 = r0 + 8;
    auto at = [&](int r, int k) {
      return *reinterpret_cast<const float2*>(ab + sw_offset(r, k >> 2, kScoreChunk) + (k & 3) * 4);
    };
    const uint32_t q0 = smem_u32(qs);
#pragma unroll 2
    for (int ks = 0; ks < D / 16; ++ks) {
      const int k0 = ks * 16 + 2 * tig;
      float2 v[4];  // (row gid, k0), (row gid + 8, k0), (row gid, k0 + 8), (row gid + 8, k0 + 8)
      v[0] = r0ok ? at(r0, k0) : make_float2(0.f, 0.f);
      v[1] = r1ok ? at(r1, k0) : make_float2(0.f, 0.f);
      v[2] = r0ok ? at(r0, k0 + 8) : make_float2(0.f, 0.f);
      v[3] = r1ok ? at(r1, k0 + 8) : make_float2(0.f, 0.f);
      uint32_t af[3][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float h0, m0, l0, h1, m1, l1;
        split3_bf16(v[i].x, h0, m0, l0);
        split3_bf16(v[i].y, h1, m1, l1);
        af[0][i] = pack_bf16(h0, h1);
        af[1][i] = pack_bf16(m0, m1);
        af[2][i] = pack_bf16(l0, l1);
      }
#pragma unroll
      for (int t = 0; t < kMaxTiles; ++t) {
        const int nt = t0 + tstep * t;
        if (nt >= NT) break;
        // Queries nt * 8 + gid, k0 and k0 + 8: two bf16 each, from the core-matrix layout.
        const uint32_t qa = q0 + cm_offset(nt * 8 + gid, k0 >> 3, D * 16) + (k0 & 7) * 2;
        uint32_t b[2];
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b[0]) : "r"(qa));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b[1]) : "r"(qa + 128));
#pragma unroll
        for (int pl = 0; pl < 3; ++pl) mma_bf16(c[t], af[pl], b);
      }
    }
  }
  __syncthreads();  // every warp has read its A_L rows
  if (rb >= rows) return;
#pragma unroll
  for (int t = 0; t < kMaxTiles; ++t) {
    const int nt = t0 + tstep * t;
    if (nt >= NT) break;
    const int col = nt * 8 + 2 * tig;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rb + gid + 8 * h;
      if (r >= rows) continue;
      if (col < G) z[r * pitch + col] = c[t][2 * h] * zscale;
      if (col + 1 < G) z[r * pitch + col + 1] = c[t][2 * h + 1] * zscale;
    }
  }
}

// ============================================================== the kernel
// kVar selects an instantiation with the common decisions constant:
// 0: general (every decision read from the parameters); 1: the single-launch
// step (fused step 1, every phase, all-gather final selection, resident token
// logits); 2: the same step from a cached fp32 A_L (no stream).
template <typename T, int D, int kVar>
__global__ void __launch_bounds__(kThreads, 1) path_kernel(const __grid_constant__ PathParams p) {
  constexpr bool kFast = kVar != 0;
  extern __shared__ __align__(1024) unsigned char smem[];  // swizzled operands need 1024
  cg::cluster_group cluster = cg::this_cluster();
  Ctx c;
  c.cs = static_cast<int>(cluster.num_blocks());
  c.rank = static_cast<int>(cluster.block_rank());
  c.tid = threadIdx.x;
  c.lane = c.tid & 31;
  c.warp = c.tid >> 5;
  c.unit = blockIdx.y;
  const int tid = c.tid, lane = c.lane, warp = c.warp, cs = c.cs, rank = c.rank;
  const int64_t unit = c.unit;
  const int G = p.G, levels = p.levels;
  const int mode = kFast ? (kModeScore | kModeFilter | kModeAttend) : p.mode;
  const bool fuse_dwt = kVar == 1 || (kVar == 0 && p.fuse_dwt);
  const bool cached_al = kVar == 2 || (kVar == 0 && p.al != nullptr);
  const bool al_stage = kVar != 1 && p.al_stage;
  const bool gather_all = kFast || p.gather_all;
  float* const t_ws = kFast ? nullptr : p.t_ws;
  const PathSmem<T, D> L(p);
  constexpr int RB = PathSmem<T, D>::kRowBytes;
  constexpr int RF = PathSmem<T, D>::kRowF;
  // bf16 A_L planes (hi / mid / lo) of one score chunk, core-matrix layout.
  constexpr int kPlaneBytes = kScoreChunk * D * 2;
  unsigned char* qs = smem + L.qs;
  float* stat_in = reinterpret_cast<float*>(smem + L.stat_in);
  float* gm = reinterpret_cast<float*>(smem + L.gm);
  float* ginv = gm + kMaxQ;
  float* loc_m = reinterpret_cast<float*>(smem + L.loc);
  float* loc_l = loc_m + kMaxQ;
  const int TS = G | 1;  // odd row pitch of logit tiles: conflict-free row-wise passes
  float* part_m = reinterpret_cast<float*>(smem + L.part);
  float* part_l = part_m + kWarps * kMaxQ;
  int32_t* cnt_a = reinterpret_cast<int32_t*>(smem + L.cnt_a);
  int32_t* cnt_b = reinterpret_cast<int32_t*>(smem + L.cnt_b);
  int32_t* misc = reinterpret_cast<int32_t*>(smem + L.misc);
  int32_t* sl_all = reinterpret_cast<int32_t*>(smem + L.sl_all);
  int32_t* sp = reinterpret_cast<int32_t*>(smem + L.sp);
  int32_t* sr = reinterpret_cast<int32_t*>(smem + L.sr);
  int32_t* cp = reinterpret_cast<int32_t*>(smem + L.cp);
  int32_t* cr = reinterpret_cast<int32_t*>(smem + L.cr);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + L.keys);
  uint8_t* take = smem + L.take;
  TopkSmem& tk = *reinterpret_cast<TopkSmem*>(smem + L.topk);
  uint32_t* keys_all = reinterpret_cast<uint32_t*>(smem + L.keys_all);
  int32_t* pos_all = reinterpret_cast<int32_t*>(smem + L.pos_all);
  int32_t* klist = reinterpret_cast<int32_t*>(smem + L.klist);

  cluster_arrive_relaxed();  // waited for after the prologue, before any peer access

  // Fused step 1: this CTA's K_p rows (the spans of its per_cta_p coarse
  // positions, one contiguous byte range) stream through a ring of bulk
  // copies; the first stages are in flight before anything else happens.
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* mma_bar = bars + kFuseStages;  // tensor-core commits (phase count in mma_phase)
  uint64_t* span_bar = bars + kFuseStages + 1;  // tensor copies of the filter's span rows (one use)
  uint32_t mma_phase = 0;
  // bf16 logits tiles run on the tensor cores with accumulators in tensor
  // memory: 256 columns (at most four pieces of N <= 64 queries), or 512.
  // The fast filter keeps up to 512 columns of token logits.
  const uint32_t kTmemCols = (kFast || p.filter_fast) ? 512u : 256u;
  const bool use_tmem = sizeof(T) == 2 && (mode & (kModeScore | kModeFilter)) != 0;
  const int fuse_sr = kFuseStageBytes / (D * static_cast<int>(sizeof(T)));  // rows per stage
  const int fuse_rows = fuse_dwt ? (p.per_cta_p << levels) : 0;
  const int fuse_nst = (fuse_rows + fuse_sr - 1) / fuse_sr;
  const unsigned char* fuse_src =
      reinterpret_cast<const unsigned char*>(static_cast<const T*>(p.kp)) +
      (unit * p.n_prompt + (static_cast<int64_t>(rank) * p.per_cta_p << levels)) * D *
          static_cast<int64_t>(sizeof(T));
  auto fuse_issue = [&](int st) {  // thread 0 only
    const int rows = min(fuse_sr, fuse_rows - st * fuse_sr);
    const uint32_t bytes = static_cast<uint32_t>(rows) * D * static_cast<uint32_t>(sizeof(T));
    uint64_t* bar = &bars[st % kFuseStages];
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(smem + L.s_ring + (st % kFuseStages) * kFuseStageBytes,
             fuse_src + static_cast<int64_t>(st) * kFuseStageBytes, bytes, bar);
  };
  int fuse_issued = min(kFuseStages, fuse_nst);
  // Cached A_L: stages of kScoreChunk fp32 rows of this CTA's contiguous range.
  const int al_nst = al_stage ? (p.per_cta_p + kScoreChunk - 1) / kScoreChunk : 0;
  const int al_nring = al_nst > 1 ? p.al_ring : 1;
  // A stage is D / 32 tensor copies of 64 rows x 32 columns (128-byte
  // swizzle; rows past the tensor's end arrive as zeros, rows of the next
  // CTA's slice are ignored), so the fragment loads below hit distinct banks.
  auto al_issue = [&](int st) {  // thread 0 only
    uint64_t* bar = &bars[st % al_nring];
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kScoreChunk * D * sizeof(float)));
    unsigned char* dst = smem + L.s_ring + static_cast<size_t>(st % al_nring) * kScoreChunk * D * sizeof(float);
    const int y = static_cast<int>(unit * p.P) + rank * p.per_cta_p + st * kScoreChunk;
    for (int kb = 0; kb < D / 32; ++kb)
      tma_load_2d(dst + kb * (kScoreChunk * 128), &p.tmap_al, kb * 32, y, bar);
  };
  int al_issued = min(al_nring, al_nst);
  // Fault injection (tests of the bounded waits): in the first CTA, stage 0
  // of the ring is never issued and its wait gives up after inject_polls polls.
  const bool inject = fuse_dwt && p.inject_polls != 0 && blockIdx.x == 0 && blockIdx.y == 0;
  if (tid == 0) {
    if (fuse_dwt)
      for (int i = 0; i < kFuseStages; ++i) mbar_init(&bars[i], 1);
    if (al_stage)
      for (int i = 0; i < al_nring; ++i) mbar_init(&bars[i], 1);
    mbar_init(mma_bar, 1);
    mbar_init(span_bar, 1);
    fence_mbar_init();
    if (fuse_dwt)
      for (int st = 0; st < fuse_issued; ++st)
        if (!(inject && st == 0)) fuse_issue(st);
    if (al_stage) prefetch_tensormap(&p.tmap_al);
    for (int st = 0; st < al_issued; ++st) al_issue(st);
    if (p.use_tma_spans) prefetch_tensormap(&p.tmap_spans);  // used by the filter phase
  }
  __syncwarp();
  if (use_tmem && warp == 0) tmem_alloc(reinterpret_cast<uint32_t*>(misc + 7), kTmemCols);

  // The Top-K histograms start zeroed (the first selection skips that step).
  topk_zero(tk);
  bool tk_clean = true;

  // Queries (input dtype, padded rows; rows >= G are zero), by cp.async: with
  // fused step 1 they land while the ring streams and are waited for just
  // before the first logits tile.
  {
    // bf16: core-matrix layout (tensor-core operand); fp32: padded rows.
    const T* qsrc = static_cast<const T*>(p.q) + unit * G * D;
    constexpr int V = Elem<T>::kPer16B;
    for (int e = tid; e < kMaxQ * (D / V); e += kThreads) {
      const int r = e / (D / V), col = (e % (D / V)) * V;
      unsigned char* dst = sizeof(T) == 2 ? qs + cm_offset(r, col / 8, D * 16)
                                          : qs + r * RB + col * sizeof(T);
      if (r < G)
        cp_async16(dst, qsrc + r * D + col);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
    if (!fuse_dwt && !al_stage) cp_async_wait<0>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = use_tmem ? static_cast<uint32_t>(misc[7]) : 0u;  // accumulator base
  cluster_wait();  // every CTA of the cluster has started: shared memory may be shared

  // ================================================================ score
  if (mode & kModeScore) {
    // Each CTA scores P/cs coarse positions; the per-query statistics are
    // merged over the cluster, then every CTA receives all P scores and
    // selects locally (so every CTA knows the sorted coarse survivors).
    const int Pc = p.per_cta_p;
    unsigned char* as = smem + L.s_as;
    float* zc = reinterpret_cast<float*>(smem + L.s_z);  // [position][query], log2 domain
    const float zscale = p.inv_sqrt_d * kLog2e;
    // Row pitch of zc: the fused stream's logits tile (odd pitch), or padded
    // rows of the coarse logits read from global memory (16-byte aligned).
    const int ZP = fuse_dwt || al_stage ? TS : p.GZ + 4;
    const int zrows = fuse_dwt || al_stage ? Pc : min(Pc, kZRows);  // positions resident at a time
    const int nz = (Pc + zrows - 1) / zrows;
    const int64_t row0 = unit * p.P + static_cast<int64_t>(rank) * Pc;  // this CTA's first position
    const float* zsrc = fuse_dwt || p.zl == nullptr ? nullptr : p.zl + row0 * p.GZ;
    if (fuse_dwt) {
      // Step 1: A_L[c] = 2^(-L/2) * (sum of the 2^L rows of span c), fp32,
      // written straight into the tile operand layout.  Two threads per
      // (span, 16-byte column chunk) of a stage (a stage holds whole spans):
      // each sums half of the span's rows, one shuffle per value combines
      // the halves, and each thread stores half of the chunk's values.
      constexpr int V = Elem<T>::kPer16B, C = D / V, VH = V / 2;
      const int half_rows = 1 << (levels - 1);
      bool aborted = false;
      for (int st = 0; st < fuse_issued; ++st) {
        // Every issued stage is waited for (bounded), even after a timeout,
        // so no copy is still landing when the ring is reused; a timeout
        // only stops further issues (the status word reports it).
        const bool ok = mbar_wait_bounded(&bars[st % kFuseStages],
                                          static_cast<uint32_t>((st / kFuseStages) & 1), p.status,
                                          inject && st == 0 ? p.inject_polls : kWaitPolls);
        if (__syncthreads_or(!ok)) aborted = true;
        const unsigned char* buf = smem + L.s_ring + (st % kFuseStages) * kFuseStageBytes;
        const int rows_in = min(fuse_sr, fuse_rows - st * fuse_sr);
        const int span0 = (st * fuse_sr) >> levels;
        const int n_half = 2 * (rows_in >> levels) * C;  // (span, chunk, half) items, even
        for (int base = 0; base < n_half; base += kThreads) {  // whole warps iterate together
          const int it = base + tid, item = it >> 1, h = it & 1;
          const bool active = it < n_half;
          const int sl = item / C, ch = item % C;
          float acc[V];
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] = 0.f;
          if (active) {
            const unsigned char* src =
                buf + static_cast<size_t>((sl << levels) + h * half_rows) * D * sizeof(T) + ch * 16;
#pragma unroll 8
            for (int r = 0; r < half_rows; ++r) {
              float f[V];
              widen16(*reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * D * sizeof(T)),
                      static_cast<const T*>(nullptr), f);
#pragma unroll
              for (int v = 0; v < V; ++v) acc[v] += f[v];
            }
          }
          float mine[VH];  // this thread's half of the chunk: values h * VH ..
#pragma unroll
          for (int v = 0; v < V; ++v) {
            const float tot = acc[v] + __shfl_xor_sync(0xffffffffu, acc[v], 1);
            if ((v >= VH) == (h == 1)) mine[v % VH] = tot * p.al_scale;
          }
          if (!active) continue;
          const int row = span0 + sl;
          if constexpr (sizeof(T) == 2) {
            uint32_t w[3][VH / 2];
#pragma unroll
            for (int v = 0; v < VH; v += 2) {
              float hv[2], mv[2], lv[2];
#pragma unroll
              for (int e2 = 0; e2 < 2; ++e2) {  // a = hi + mid + lo exactly (to 2^-25 relative)
                const float a = mine[v + e2];
                hv[e2] = __bfloat162float(__float2bfloat16_rn(a));
                const float r1 = a - hv[e2];
                mv[e2] = __bfloat162float(__float2bfloat16_rn(r1));
                lv[e2] = r1 - mv[e2];
              }
              w[0][v / 2] = pack_bf16(hv[0], hv[1]);
              w[1][v / 2] = pack_bf16(mv[0], mv[1]);
              w[2][v / 2] = pack_bf16(lv[0], lv[1]);
            }
#pragma unroll
            for (int pl = 0; pl < 3; ++pl)
              *reinterpret_cast<uint2*>(as + pl * kPlaneBytes + sw_offset(row, ch, kScoreChunk) + h * 8) =
                  make_uint2(w[pl][0], w[pl][1]);
          } else {
            *reinterpret_cast<float2*>(as + row * RB + ch * 16 + h * 8) = make_float2(mine[0], mine[1]);
          }
        }
        __syncthreads();  // stage consumed
        if (!aborted && st + kFuseStages < fuse_nst) {
          if (tid == 0) {
            fence_proxy_async();
            fuse_issue(st + kFuseStages);
          }
          ++fuse_issued;
        }
      }
      cp_async_wait<0>();  // the queries
      if (sizeof(T) == 2) {
        umma_logits<D>(as, 3, kPlaneBytes, kScoreChunk, Pc, qs, G, zc, 0, TS, zscale, tmem, mma_bar,
                       mma_phase, p.status);
      } else {
        __syncthreads();
        logits_tile_f32<D>(as, reinterpret_cast<const float*>(qs), zc, 0, Pc, G, TS, zscale);
      }
      __syncthreads();
    } else if (sizeof(T) == 2 && al_stage) {
      // Cached A_L: stages of 64 rows (fp32, D floats apart) land in the
      // ring; the warps form each stage's logits with the queries straight
      // from there.  Every issued stage is waited for (bounded), even after a
      // timeout, so no copy lands after the ring is reused; a timeout only
      // stops further issues (the status word reports it).
      const float* ring = reinterpret_cast<const float*>(smem + L.s_ring);
      cp_async_wait<0>();  // the queries (visible after the loop's first barrier)
      bool aborted = false;
      // With every stage resident two stages (128 rows, one 16-row tile per
      // warp) go through the tensor cores at a time; with a refilled ring one.
      const int step = al_nring == al_nst ? 2 : 1;
      for (int st = 0; st < al_issued; st += step) {
        const int n_st = min(step, al_issued - st);
        bool ok = true;
        for (int j = 0; j < n_st; ++j)
          ok = mbar_wait_bounded(&bars[(st + j) % al_nring],
                                 static_cast<uint32_t>(((st + j) / al_nring) & 1), p.status) && ok;
        if (__syncthreads_or(!ok)) aborted = true;
        const int r0 = st * kScoreChunk;
        coarse_logits_ring<D>(ring + static_cast<size_t>(st % al_nring) * kScoreChunk * D,
                              min(n_st * kScoreChunk, Pc - r0), qs, G, zc + r0 * TS, TS, zscale);
        __syncthreads();  // stage consumed
        if (step == 1 && !aborted && st + al_nring < al_nst) {
          if (tid == 0) {
            fence_proxy_async();
            al_issue(st + al_nring);
          }
          ++al_issued;
        }
      }
    }
    // Coarse logits of positions [c0, c0 + rows) into zc: read from global
    // memory, or formed here from a cached fp32 A_L (16 rows per warp task).
    auto load_z = [&](int c0, int rows) {
      __syncthreads();  // earlier readers of zc are done
      if (cached_al) {
        coarse_logits_range<T, D>(p.al + (row0 + c0) * D, static_cast<const T*>(p.q) + unit * G * D,
                                  zc, 0, rows, int64_t{1} << 40, G, ZP, zscale, warp, kWarps);
      } else {
        const int c4 = p.GZ >> 2;
        for (int e = tid; e < rows * c4; e += kThreads) {
          const int r = e / c4, k = e - r * c4;
          cp_async16(zc + r * ZP + 4 * k, zsrc + static_cast<int64_t>(c0 + r) * p.GZ + 4 * k);
        }
        cp_async_commit();
        cp_async_wait<0>();
      }
      __syncthreads();
    };
    // Pass 1: per-query (max, sum) over this CTA's positions; thread ->
    // queries lane / lane + 32, positions warp + 8u of every 64-row block.
    float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
    for (int zc0 = 0; zc0 < Pc; zc0 += zrows) {
      const int zr = min(zrows, Pc - zc0);
      if (!fuse_dwt && !al_stage) load_z(zc0, zr);
      const int q0 = lane < G ? lane : 0, q1 = lane + 32 < G ? lane + 32 : 0;
      for (int c0 = 0; c0 < zr; c0 += kScoreChunk) {
        float z[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int r = c0 + warp + kWarps * u;
          z[u] = r < zr && lane < G ? zc[r * ZP + q0] : -INFINITY;
        }
        online8(m0, l0, z);
        if (G > 32) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int r = c0 + warp + kWarps * u;
            z[u] = r < zr && lane + 32 < G ? zc[r * ZP + q1] : -INFINITY;
          }
          online8(m1, l1, z);
        }
      }
    }
    part_m[warp * kMaxQ + lane] = m0;
    part_l[warp * kMaxQ + lane] = l0;
    part_m[warp * kMaxQ + lane + 32] = m1;
    part_l[warp * kMaxQ + lane + 32] = l1;
    __syncthreads();
    if (tid < G) {
      float cm = -INFINITY, cl = 0.f;
      for (int w = 0; w < kWarps; ++w) merge_ml(cm, cl, part_m[w * kMaxQ + tid], part_l[w * kMaxQ + tid]);
      loc_m[tid] = cm;
      loc_l[tid] = cl;
    }
    __syncthreads();
    cluster_merge_stats(loc_m, loc_l, G, stat_in, gm, ginv);
    // Pass 2: attention mass of every position (4 threads per position).
    for (int zc0 = 0; zc0 < Pc; zc0 += zrows) {
      const int zr = min(zrows, Pc - zc0);
      if (nz > 1) load_z(zc0, zr);  // one chunk: zc still holds it
      for (int c0 = 0; c0 < zr; c0 += kThreads / 4) {
        const int r = c0 + (tid >> 2), sub = tid & 3;
        float sa = 0.f, sb = 0.f;
        if (r < zr) {
          int qi = sub;
          for (; qi + 4 < G; qi += 8) {
            sa += fast_exp2(zc[r * ZP + qi] - gm[qi]) * ginv[qi];
            sb += fast_exp2(zc[r * ZP + qi + 4] - gm[qi + 4]) * ginv[qi + 4];
          }
          if (qi < G) sa += fast_exp2(zc[r * ZP + qi] - gm[qi]) * ginv[qi];
        }
        float sacc = sa + sb;
        sacc += __shfl_xor_sync(0xffffffffu, sacc, 1);
        sacc += __shfl_xor_sync(0xffffffffu, sacc, 2);
        if (r < zr && sub == 0) {
          const int pos = rank * Pc + zc0 + r;
          for (int rr = 0; rr < cs; ++rr) peer(keys_all, rr)[pos] = __float_as_uint(sacc);
          if (p.scores_out != nullptr) p.scores_out[unit * p.P + pos] = sacc;
        }
      }
    }
    cluster.sync();  // every CTA holds all P scores
    // Exact Top-k_L over all coarse positions (ties: lower position first).
    const bool to_filter = (mode & kModeFilter) != 0;
    block_select_topk(keys_all, p.P, p.kL, 0, p.kL, sl_all, tk, tk_clean);
    tk_clean = false;
    if (!to_filter && rank == 0)
      for (int i = tid; i < p.kL; i += kThreads) p.idx_l_out[unit * p.kL + i] = sl_all[i];
  } else if (mode & kModeFilter) {
    // Coarse survivors from the caller: load, sort ascending, validate.
    const int kL = p.kL, P = p.P;
    for (int i = tid; i < p.sorted_cap; i += kThreads)
      sl_all[i] = i < kL ? p.idx_l_in[unit * kL + i] : INT_MAX;
    __syncthreads();
    for (int kk = 2; kk <= p.sorted_cap; kk <<= 1) {
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        for (int i = tid; i < p.sorted_cap; i += kThreads) {
          const int ixj = i ^ jj;
          if (ixj > i) {
            const int a = sl_all[i], b = sl_all[ixj];
            if ((a > b) == ((i & kk) == 0)) {
              sl_all[i] = b;
              sl_all[ixj] = a;
            }
          }
        }
        __syncthreads();
      }
    }
    int bad = 0;
    for (int i = tid; i < kL; i += kThreads) {
      const int v = sl_all[i];
      if (v < 0 || v >= P) bad |= WF_DEV_BAD_INDEX;
      if (i > 0 && sl_all[i - 1] == v) bad |= WF_DEV_DUP_INDEX;
    }
    __syncthreads();
    for (int i = tid; i < kL; i += kThreads) sl_all[i] = min(max(sl_all[i], 0), P - 1);
    if (bad && rank == 0) raise_flag(p.status, bad);
    __syncthreads();
  }

  // ================================================================ filter
  if (mode & kModeFilter) {
    const int kL = p.kL;
    const int s0 = static_cast<int>((static_cast<int64_t>(rank) * kL) / cs);
    const int s1 = static_cast<int>((static_cast<int64_t>(rank + 1) * kL) / cs);
    const int ns = s1 - s0;
    const int R = ns << levels;
    bool global_done = false;  // final token list already distributed
    int n_surv = 0;
    if (sizeof(T) == 2 && (kFast || p.filter_fast)) {
      // -------- fast path (token-level selection only; every level between
      // L and 0 keeps all children): the R = ns 2^L rows under this CTA's
      // coarse survivors go through a ring of 128-row tiles filled by 2-D
      // tensor copies (whole spans, 128-byte swizzle), one tcgen05.mma pass
      // per tile into its own tensor-memory accumulator (N = G rounded up to
      // 16 columns).  Thread 0 issues copies and MMAs; warps 4-7 (one per
      // tensor-memory lane quarter) read each finished accumulator, stage it
      // in shared memory and fold it into per-query (max, sum) statistics.
      // After the cluster-wide merge the token scores are formed from the
      // accumulators again: still resident (filter_fast == 1, ntiles * N <=
      // 512 columns), or recomputed by a second pass over the tiles through
      // a few rotating accumulators (filter_fast == 2, which never spills).
      constexpr int TR = 128;
      constexpr int kStageBytes = D * 256;  // D / 64 column blocks of 128 rows x 128 B
      const int box_rows = min(1 << levels, TR);
      const int ntiles = (R + TR - 1) / TR;
      const int S = p.f_stages, NB = p.f_nb;
      const bool resident = kFast || p.filter_fast == 1;
      const int N = (G + 15) & ~15;
      const int total = resident ? ntiles : 2 * ntiles;
      const int ZT2 = p.GZ + 4;
      unsigned char* ring = smem + L.f_ring;
      float* fst = reinterpret_cast<float*>(smem + L.f_stage);
      uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.f_bars);
      uint64_t* done = full + S;
      uint64_t* empty = done + NB;
      volatile int32_t* fabort = misc + 6;
      const float sc2 = p.scale[0] * kLog2e;
      if (tid == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&full[i], 1);
        for (int i = 0; i < NB; ++i) {
          mbar_init(&done[i], 1);
          mbar_init(&empty[i], 4);  // one arrival per consumer warp
        }
        fence_mbar_init();
        *fabort = 0;
      }
      if (!tk_clean) {
        topk_zero(tk);
        tk_clean = true;
      }
      tc_fence_before();
      __syncthreads();
      tc_fence_after();

      // ---- producer (thread 0): next tile to copy, next tile to multiply
      FilterProducer<D> prod{ring, full, done, &p.tmap_spans, sl_all, qs, p.status, fabort, tmem,
                             s0, levels, static_cast<int>(unit * p.n_prompt), R, ntiles, total, S,
                             NB, N};
      const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
      const int row_l = (warp & 3) * 32 + lane;

      // ---- pass A: statistics
      float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
      if (warp == 0) {
        if (lane == 0) prod.run(resident ? total : min(total, ntiles + NB));
        __syncwarp();
      } else if (warp >= 4) {
        const int qw = warp & 3;
        for (int t = 0; t < ntiles; ++t) {
          const int slot = t % NB;
          bool okc = *fabort == 0 &&
                     mbar_wait_bounded(&done[slot], static_cast<uint32_t>((t / NB) & 1), p.status);
          okc = __all_sync(0xffffffffu, okc);
          tc_fence_after();
          const int rows_valid = min(TR, R - t * TR);
          if (okc) tmem_row_to_smem(t_lane + slot * N, N, p.GZ, row_l < rows_valid, fst + row_l * ZT2);
          if (!resident) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
          }
          // Each warp stages and then reads only its own 32 rows: a warp-level
          // barrier orders the staging stores before the reads.
          __syncwarp();
          const int qa = lane < G ? lane : 0, qb = lane + 32 < G ? lane + 32 : 0;
#pragma unroll
          for (int u0 = 0; u0 < 32; u0 += 8) {
            float z[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int r = qw * 32 + u0 + u;
              z[u] = okc && r < rows_valid && lane < G ? fst[r * ZT2 + qa] * sc2 : -INFINITY;
            }
            online8(m0, l0, z);
            if (G > 32) {
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int r = qw * 32 + u0 + u;
                z[u] = okc && r < rows_valid && lane + 32 < G ? fst[r * ZT2 + qb] * sc2 : -INFINITY;
              }
              online8(m1, l1, z);
            }
          }
          __syncwarp();  // the next tile's staging overwrites these rows
        }
      }
      if (warp >= 4) {
        const int w4 = warp - 4;
        part_m[w4 * kMaxQ + lane] = m0;
        part_l[w4 * kMaxQ + lane] = l0;
        part_m[w4 * kMaxQ + lane + 32] = m1;
        part_l[w4 * kMaxQ + lane + 32] = l1;
      }
      __syncthreads();
      if (tid < G) {
        float m = -INFINITY, l = 0.f;
        for (int w = 0; w < 4; ++w) merge_ml(m, l, part_m[w * kMaxQ + tid], part_l[w * kMaxQ + tid]);
        loc_m[tid] = m;
        loc_l[tid] = l;
      }
      __syncthreads();
      cluster_merge_stats(loc_m, loc_l, G, stat_in, gm, ginv, R, gather_all ? cnt_b : nullptr);

      // ---- pass B: token scores s = Σ_q 2^(z - gm_q) / sum_q
      if (resident) {
        // Every multiply has completed (pass A waited for each): all eight
        // warps read the accumulators, warps w and w + 4 sharing a lane
        // quarter and taking alternate tiles.
        tc_fence_after();
        if (*fabort == 0) {
          for (int t = warp >> 2; t < ntiles; t += 2) {
            const float sc = token_score_tmem(t_lane + t * N, N, G, sc2, gm, ginv);
            const int row = t * TR + row_l;
            if (row < R) keys[row] = __float_as_uint(sc);
          }
        }
      } else if (warp == 0) {
        if (lane == 0) prod.run(total);
        __syncwarp();
      } else if (warp >= 4) {
        for (int t = 0; t < ntiles; ++t) {
          const int g = ntiles + t, slot = g % NB;
          bool okc = *fabort == 0 &&
                     mbar_wait_bounded(&done[slot], static_cast<uint32_t>((g / NB) & 1), p.status);
          okc = __all_sync(0xffffffffu, okc);
          tc_fence_after();
          if (okc) {
            const float sc = token_score_tmem(t_lane + slot * N, N, G, sc2, gm, ginv);
            const int row = t * TR + row_l;
            if (row < R) keys[row] = __float_as_uint(sc);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
        }
      }
      tc_fence_before();
      __syncthreads();
      tc_fence_after();

      // ---- selection of the budget among the unit's token candidates
      const int B = p.budget;
      if (gather_all) {
        // Every CTA receives every candidate (score, position) and selects
        // the budget locally, keeping its slot range of the key list.
        int off = 0, n_all = 0;
        for (int r = 0; r < cs; ++r) {
          if (r < rank) off += cnt_b[r];
          n_all += cnt_b[r];
        }
        uint32_t* gkeys = reinterpret_cast<uint32_t*>(smem + L.f_gather);
        int32_t* gpos = reinterpret_cast<int32_t*>(gkeys + cs * p.rows_cap);
        // Four candidates per 16-byte store (R and every offset are multiples of 8).
        const int R4 = R >> 2;
        for (int e = tid; e < R4 * cs; e += kThreads) {
          const int i = (e % R4) * 4, r = e / R4;
          *reinterpret_cast<uint4*>(peer(gkeys, r) + off + i) = *reinterpret_cast<const uint4*>(keys + i);
          *reinterpret_cast<int4*>(peer(gpos, r) + off + i) =
              make_int4(span_token(sl_all, s0, i, levels), span_token(sl_all, s0, i + 1, levels),
                        span_token(sl_all, s0, i + 2, levels), span_token(sl_all, s0, i + 3, levels));
        }
        cluster.sync();
        if (mode & kModeAttend) {
          // This CTA's slots of the key list, [a0, min(a1, B)).
          const int a0 = key_slot_start(rank, cs, p.n_keys), a1 = key_slot_start(rank + 1, cs, p.n_keys);
          const int b1 = min(a1, B);
          block_select_topk(gkeys, n_all, B, a0, b1, klist, tk, tk_clean, gpos);
          if (p.idx_out != nullptr)
            for (int sl = a0 + tid; sl < b1; sl += kThreads) p.idx_out[unit * B + sl] = klist[sl - a0];
        } else {
          // No key list: this CTA's share of the output slots, straight to idx.
          const int w0 = key_slot_start(rank, cs, B), w1 = key_slot_start(rank + 1, cs, B);
          block_select_topk(gkeys, n_all, B, w0, w1, p.idx_out + unit * B + w0, tk, tk_clean, gpos);
        }
        tk_clean = false;
        global_done = true;
      } else {
        (void)cluster_select(keys, R, B, take, tk);
        tk_clean = false;
        int carry = 0;
        for (int base = 0; base < R; base += kThreads) {
          const int i = base + tid;
          const int tf = i < R ? take[i] : 0;
          int tot;
          const int at = block_excl_scan(tf, tk.scan, &tot);
          if (tf) sp[carry + at] = span_token(sl_all, s0, i, levels);
          carry += tot;
        }
        __syncthreads();
        n_surv = carry;
      }
    } else {
      unsigned char* kst = smem + L.f_kst;
      // Row pitch of t: odd in shared memory (conflict-free row-wise passes),
      // a multiple of 4 floats when spilled to the workspace (16-byte loads).
      const int TT = t_ws == nullptr ? TS : ((G + 3) & ~3);
      float* t = t_ws == nullptr
                     ? reinterpret_cast<float*>(smem + L.f_t)
                     : t_ws + (static_cast<int64_t>(unit) * cs + rank) * p.rows_cap * TT;
      const T* kp = static_cast<const T*>(p.kp);
      const int ntiles = (R + kTileRows - 1) / kTileRows;
      constexpr int C16 = D * static_cast<int>(sizeof(T)) / 16;  // 16-byte chunks per row
      // Offset of a ring stage: bf16, rows of the 128-byte-swizzled layout
      // (column blocks of FS * kTileRows rows); fp32, padded rows.
      constexpr int kStageB = sizeof(T) == 2 ? kTileRows * 128 : kTileRows * RB;
      const int FS = p.f_stages;
      auto issue = [&](int tile, int stage) {  // all threads; one cp.async group
        const int r0 = tile * kTileRows;
        const int nr = min(kTileRows, R - r0);
        for (int e = tid; e < nr * C16; e += kThreads) {
          const int i = e / C16, ch = e % C16;
          const int lr = r0 + i;
          const int64_t grow = unit * p.n_prompt +
                               (static_cast<int64_t>(sl_all[s0 + (lr >> levels)]) << levels) +
                               (lr & ((1 << levels) - 1));
          // bf16: core-matrix layout, stages back to back (a tensor-core
          // operand may span stages); fp32: padded rows.
          unsigned char* dst = sizeof(T) == 2
                                   ? kst + sw_offset(stage * kTileRows + i, ch, FS * kTileRows)
                                   : kst + (stage * kTileRows + i) * RB + ch * 16;
          cp_async16(dst, reinterpret_cast<const unsigned char*>(kp + grow * D) + ch * 16);
        }
        cp_async_commit();
      };
      // bf16 with every row in the ring at once: one tensor copy per (span,
      // 64-column block) lands the span's 2^L rows straight in the swizzled
      // operand layout (8-row groups, so 2^L >= 8); otherwise 16-byte cp.async.
      const bool tma_spans = sizeof(T) == 2 && p.use_tma_spans && ntiles <= FS;
      if (tma_spans) {
        constexpr int KB = D / 64;  // 64-column blocks per row
        if (tid == 0) mbar_arrive_expect_tx(span_bar, static_cast<uint32_t>(R) * D * sizeof(T));
        for (int i = tid; i < ns * KB; i += kThreads) {
          const int sp_i = i / KB, kb = i - sp_i * KB;
          tma_load_2d(kst + kb * (FS * kTileRows * 128) + ((sp_i << levels) >> 3) * 1024,
                      &p.tmap_spans, kb * 64,
                      static_cast<int>(unit * p.n_prompt + (sl_all[s0 + sp_i] << levels)), span_bar);
        }
      } else {
        for (int tl = 0; tl < FS && tl < ntiles; ++tl) issue(tl, tl);
      }
      if (!tk_clean) {  // while the key rows are in flight (the tile barriers order it)
        topk_zero(tk);
        tk_clean = true;
      }
      if (ntiles <= FS && sizeof(T) == 2) {
        // Every row is in flight: one wait, then one tensor-core pass over all
        // R rows (tiles sit back to back in the ring).  If the wait gives up
        // (the status word reports it) no multiply reads the ring.
        bool rows_ok = true;
        if (tma_spans)
          rows_ok = mbar_wait_bounded(span_bar, 0, p.status);
        else
          cp_async_wait<0>();
        if (!__syncthreads_or(!rows_ok))
          umma_logits<D>(kst, 1, 0, FS * kTileRows, R, qs, G, t, 0, TT, 1.f, tmem, mma_bar,
                         mma_phase, p.status);
        __syncthreads();
      } else
      for (int tile = 0; tile < ntiles; ++tile) {
        const int stage = tile % FS;
        cp_async_wait_pending(min(ntiles, tile + FS) - 1 - tile);
        const int rows_valid = min(kTileRows, R - tile * kTileRows);
        if constexpr (sizeof(T) == 2) {
          umma_logits<D>(kst + stage * kStageB, 1, 0, FS * kTileRows, rows_valid, qs, G, t,
                         tile * kTileRows, TT, 1.f, tmem, mma_bar, mma_phase, p.status);
        } else {
          __syncthreads();
          logits_tile_f32<D>(kst + stage * kStageB, reinterpret_cast<const float*>(qs), t,
                             tile * kTileRows, rows_valid, G, TT, 1.f);
        }
        __syncthreads();
        if (tile + FS < ntiles) issue(tile + FS, stage);
      }
      __syncthreads();

      // Levels that keep every child need no scoring: start from the survivors
      // of the lowest of them (all descendants of the coarse survivors, in
      // position order) and walk down from the first level that selects.
      int j_top = levels - 1;
      while (j_top >= 0 && p.k[j_top] >= 2 * p.k[j_top + 1]) --j_top;
      const int jj = j_top + 1, dsh = levels - jj;  // survivors at level jj: 2^dsh per span
      n_surv = ns << dsh;
      for (int e = tid; e < n_surv; e += kThreads) {
        const int i = e >> dsh, m = e & ((1 << dsh) - 1);
        sp[e] = (sl_all[s0 + i] << dsh) + m;
        sr[e] = (i << levels) + (m << jj);
      }
      __syncthreads();
      for (int j = j_top; j >= 0; --j) {
        for (int i = tid; i < n_surv; i += kThreads) {
          const int pos = sp[i], row = sr[i];
          cp[2 * i] = 2 * pos;
          cp[2 * i + 1] = 2 * pos + 1;
          cr[2 * i] = row;
          cr[2 * i + 1] = row + (1 << j);
        }
        const int n_cand = 2 * n_surv;
        __syncthreads();
        if (p.k[j] >= 2 * p.k[j + 1]) {  // every candidate survives: no scoring
          int32_t* x = sp; sp = cp; cp = x;
          x = sr; sr = cr; cr = x;
          n_surv = n_cand;
          continue;
        }
        // Scores of this level's candidates (log2 domain, z = sc2 * Σ_leaves t):
        //  pass A  per query, online (max, Σ 2^(z - max)) over this CTA's
        //          candidates (lanes = queries q and q + 32; a warp takes 8
        //          candidates at a time, their loads issued together);
        //  CTA and cluster merges give the global max gm and 1 / sum ginv;
        //  pass B  s_c = Σ_q 2^(z[c,q] - gm_q) * ginv_q, one thread per candidate.
        const int leaves = 1 << j;
        const float sc2 = p.scale[j] * kLog2e;
        const bool final_gather = j == 0 && gather_all;
        const bool qa = lane < G, qb = lane + 32 < G;
        const int la = qa ? lane : 0, lb = qb ? lane + 32 : 0;
        // Leaf sum of t for candidate row offset `row` (row index * TT), query q.
        auto leaf_sum = [&](int row, int q) {
          float a = 0.f;
  #pragma unroll 1
          for (int i = 0; i < leaves; ++i) a += t[row + i * TT + q];
          return a;
        };
        float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
        if (leaves == 1) {
          // Sixteen candidates per warp step, every load of a step (both query
          // halves) issued before the first exponential.
          for (int ci0 = warp * 16; ci0 < n_cand; ci0 += kWarps * 16) {
            int rows[16];
  #pragma unroll
            for (int u = 0; u < 16; ++u) rows[u] = cr[min(ci0 + u, n_cand - 1)] * TT;
            float za[2][8], zb[2][8];
  #pragma unroll
            for (int u = 0; u < 16; ++u) za[u >> 3][u & 7] = t[rows[u] + la];
            if (G > 32) {
  #pragma unroll
              for (int u = 0; u < 16; ++u) zb[u >> 3][u & 7] = t[rows[u] + lb];
            }
  #pragma unroll
            for (int u = 0; u < 16; ++u) {
              const bool ok = ci0 + u < n_cand;
              za[u >> 3][u & 7] = ok && qa ? za[u >> 3][u & 7] * sc2 : -INFINITY;
              zb[u >> 3][u & 7] = ok && qb ? zb[u >> 3][u & 7] * sc2 : -INFINITY;
            }
            online8(m0, l0, za[0]);
            online8(m0, l0, za[1]);
            if (G > 32) {
              online8(m1, l1, zb[0]);
              online8(m1, l1, zb[1]);
            }
          }
        } else {
          for (int ci0 = warp * 8; ci0 < n_cand; ci0 += kWarps * 8) {
            float z[8];
  #pragma unroll 1
            for (int u = 0; u < 8; ++u) {
              const int row = cr[min(ci0 + u, n_cand - 1)] * TT;
              z[u] = ci0 + u < n_cand && qa ? leaf_sum(row, la) * sc2 : -INFINITY;
            }
            online8(m0, l0, z);
            if (G > 32) {  // queries 32..63
  #pragma unroll 1
              for (int u = 0; u < 8; ++u) {
                const int row = cr[min(ci0 + u, n_cand - 1)] * TT;
                z[u] = ci0 + u < n_cand && qb ? leaf_sum(row, lb) * sc2 : -INFINITY;
              }
              online8(m1, l1, z);
            }
          }
        }
        part_m[warp * kMaxQ + lane] = m0;
        part_m[warp * kMaxQ + lane + 32] = m1;
        part_l[warp * kMaxQ + lane] = l0;
        part_l[warp * kMaxQ + lane + 32] = l1;
        __syncthreads();
        if (tid < G) {
          float m = -INFINITY, l = 0.f;
          for (int w = 0; w < kWarps; ++w) merge_ml(m, l, part_m[w * kMaxQ + tid], part_l[w * kMaxQ + tid]);
          loc_m[tid] = m;
          loc_l[tid] = l;
        }
        __syncthreads();
        cluster_merge_stats(loc_m, loc_l, G, stat_in, gm, ginv, n_cand, final_gather ? cnt_b : nullptr);
        // Pass B: one thread per candidate (odd row pitch in shared memory:
        // conflict-free); four independent partial sums over the queries.
        for (int ci = tid; ci < n_cand; ci += kThreads) {
          const int row = cr[ci] * TT;
          float sq[4] = {0.f, 0.f, 0.f, 0.f};
          if (leaves == 1 && t_ws != nullptr) {
            // Spilled rows (L2): 16-byte loads, four in flight; columns >= G are padding.
            const float4* r4 = reinterpret_cast<const float4*>(t + row);
  #pragma unroll 4
            for (int q4 = 0; q4 < TT / 4; ++q4) {
              const float4 v = r4[q4];
              const float vv[4] = {v.x, v.y, v.z, v.w};
  #pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int q = 4 * q4 + k;
                if (q < G) sq[k] += fast_exp2(vv[k] * sc2 - gm[q]) * ginv[q];
              }
            }
          } else if (leaves == 1) {
            int q = 0;
  #pragma unroll 2
            for (; q + 4 <= G; q += 4) {
  #pragma unroll
              for (int k = 0; k < 4; ++k) sq[k] += fast_exp2(t[row + q + k] * sc2 - gm[q + k]) * ginv[q + k];
            }
            for (; q < G; ++q) sq[0] += fast_exp2(t[row + q] * sc2 - gm[q]) * ginv[q];
          } else {
  #pragma unroll 1
            for (int q = 0; q < G; ++q) sq[q & 3] += fast_exp2(leaf_sum(row, q) * sc2 - gm[q]) * ginv[q];
          }
          keys[ci] = __float_as_uint((sq[0] + sq[1]) + (sq[2] + sq[3]));
        }
        __syncthreads();
        if (final_gather) {
          // Every CTA receives every candidate (score, position) at its dense
          // offset, selects the budget locally and keeps what it needs: its
          // slot range of the key list (attend) and of the output (idx).
          int off = 0, n_all = 0;
          for (int r = 0; r < cs; ++r) {
            if (r < rank) off += cnt_b[r];
            n_all += cnt_b[r];
          }
          for (int e = tid; e < n_cand * cs; e += kThreads) {
            const int i = e % n_cand, r = e / n_cand;
            peer(keys_all, r)[off + i] = keys[i];
            peer(pos_all, r)[off + i] = cp[i];
          }
          cluster.sync();
          const int B = p.budget;
          if (mode & kModeAttend) {
            // This CTA's slots of the key list: [a0, min(a1, B)); klist
            // receives the selected candidates' token positions.
            const int a0 = key_slot_start(rank, cs, p.n_keys), a1 = key_slot_start(rank + 1, cs, p.n_keys);
            const int b1 = min(a1, B);
            block_select_topk(keys_all, n_all, B, a0, b1, klist, tk, tk_clean, pos_all);  // positions
            if (p.idx_out != nullptr)
              for (int sl = a0 + tid; sl < b1; sl += kThreads) p.idx_out[unit * B + sl] = klist[sl - a0];
          } else {
            // No key list: this CTA's share of the output slots, straight to idx.
            const int w0 = key_slot_start(rank, cs, B), w1 = key_slot_start(rank + 1, cs, B);
            block_select_topk(keys_all, n_all, B, w0, w1, p.idx_out + unit * B + w0, tk, tk_clean,
                              pos_all);
          }
          tk_clean = false;
          global_done = true;
          break;
        }
        (void)cluster_select(keys, n_cand, p.k[j], take, tk);
        tk_clean = false;
        n_surv = compact2(cp, cr, take, n_cand, sp, sr, tk.scan);
      }
    }
    // Tokens of this CTA: sp[0, n_surv), ascending.
    if (!global_done) {
    int all;
    const int offset = cluster_excl_count(n_surv, cnt_a, &all);
    const int B = p.budget;
    if (mode & kModeAttend) {
      for (int i = tid; i < n_surv; i += kThreads) {
        const int g = offset + i;
        if (g >= B) continue;
        const int owner = key_slot_owner(g, cs, p.n_keys);
        peer(klist, owner)[g - key_slot_start(owner, cs, p.n_keys)] = sp[i];
        if (p.idx_out != nullptr) p.idx_out[unit * B + g] = sp[i];
      }
      cluster.sync();
    } else {
      for (int i = tid; i < n_surv; i += kThreads)
        if (offset + i < B) p.idx_out[unit * B + offset + i] = sp[i];
    }
    }
  }

  // ================================================================ attend
  if (mode & kModeAttend) {
    const int B = p.budget, TK = p.tile_keys;
    const int k0 = key_slot_start(rank, cs, p.n_keys);
    const int k1 = key_slot_start(rank + 1, cs, p.n_keys);
    const int ntiles = (k1 - k0 + TK - 1) / TK;
    unsigned char* kst = smem + L.a_kst;
    unsigned char* vst = smem + L.a_vst;
    float* work = reinterpret_cast<float*>(smem + L.a_work);
    float* recv_o = reinterpret_cast<float*>(smem + L.a_recv);
    float* recv_ml = reinterpret_cast<float*>(smem + L.a_rml);
    const int rpo = (G + cs - 1) / cs;
    const T* kgp = static_cast<const T*>(p.kg) + unit * G * D;
    const T* vgp = static_cast<const T*>(p.vg) + unit * G * D;
    const T* kpp = static_cast<const T*>(p.kp) + unit * p.n_prompt * D;
    const T* vpp = static_cast<const T*>(p.vp) + unit * p.n_prompt * D;
    if (!(mode & kModeFilter)) {
      // The caller's rows of this slot range, staged once (the copies below
      // then need no dependent global load); bad ones are reported.
      const int32_t* src = p.idx_in + unit * B;
      bool bad = false;
      for (int g = k0 + tid; g < min(k1, B); g += kThreads) {
        const int row = __ldg(src + g);
        klist[g - k0] = row;
        bad |= row < 0 || row >= p.n_prompt;
      }
      if (bad) raise_flag(p.status, WF_DEV_BAD_INDEX);
    }
    // Every slot of a tile is filled (invalid slots with a finite dummy row),
    // so masked probabilities multiply finite values.
    const AttnRows<T> ar{kgp, vgp, kpp, vpp, klist, k0, k1, B};
    __syncthreads();  // filter-phase readers of the union are done
    const int AS = p.a_stages;
    for (int tl = 0; tl < AS && tl < ntiles; ++tl) attn_issue<T, D>(p, mode, c, ar, kst, vst, TK, tl, tl);

    if constexpr (sizeof(T) == 2) {
      const int MB = G <= 16 ? 1 : (G <= 32 ? 2 : 4);
      // Keys per warp per tile (the plan's tile / key-group warps): 16, or 32
      // with four query-row blocks in the general instantiation, so a tile
      // still holds 64 keys and its fixed cost (wait, barrier, copies) is
      // spread over as many keys as with fewer queries.  The constant-folded
      // instantiations keep the 16-key body (their code stays smaller).
      const bool two = !kFast && TK * MB / kWarps == 32;
      const int KB = two ? 32 : 16;
      const int mb = warp % MB, kgrp = warp / MB;
      uint32_t qa[D / 16][4];
      {
        // Q rows mb * 16 + (lane & 15), chunk 2 ks + (lane >> 4), core-matrix layout.
        const uint32_t qbase = smem_u32(qs) + cm_offset(mb * 16 + (lane & 15), lane >> 4, D * 16);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) ldsm_x4(qbase + ks * 256, qa[ks]);
      }
      float oacc[D / 8][4];
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[i][e] = 0.f;
      float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
      for (int tile = 0; tile < ntiles; ++tile) {
        const int stage = tile % AS;
        // Tiles issued before this iteration's refill: 0 .. min(ntiles, AS + tile - 1) - 1.
        cp_async_wait_pending(tile == 0 ? min(ntiles, AS) - 1 : min(ntiles - tile - 1, AS - 2));
        __syncthreads();  // this tile's rows are visible; every warp is done with tile - 1
        const uint32_t kb = smem_u32(kst + (stage * TK + kgrp * KB) * RB);
        const uint32_t vb = smem_u32(vst + (stage * TK + kgrp * KB) * RB);
        // Logits of the warp's keys: n-blocks of 8 keys (two per 16-key block).
        float s[4][4];
#pragma unroll
        for (int nb = 0; nb < 4; ++nb)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[nb][e] = 0.f;
        const uint32_t kaddr = kb + ((lane & 7) + ((lane >> 4) << 3)) * RB + ((lane >> 3) & 1) * 16;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t b[4];
          ldsm_x4(kaddr + ks * 32, b);
          mma_bf16(s[0], qa[ks], b);
          mma_bf16(s[1], qa[ks], b + 2);
          if (two) {
            uint32_t b2[4];
            ldsm_x4(kaddr + 16 * RB + ks * 32, b2);
            mma_bf16(s[2], qa[ks], b2);
            mma_bf16(s[3], qa[ks], b2 + 2);
          }
        }
        const int NB = two ? 4 : 2;
        const int jbase = k0 + tile * TK + kgrp * KB + (lane & 3) * 2;
        float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
        for (int nb = 0; nb < 4; ++nb)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            if (nb >= NB) continue;
            const bool v = attn_key_valid(p, mode, c, ar, jbase + nb * 8 + e);
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
        const float corr_lo = fast_exp2(m_lo - base_lo), corr_hi = fast_exp2(m_hi - base_hi);
        float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
        for (int nb = 0; nb < 4; ++nb)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            if (nb >= NB) continue;
            s[nb][e] = fast_exp2(s[nb][e] - base_lo);
            s[nb][e + 2] = fast_exp2(s[nb][e + 2] - base_hi);
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
        // Probabilities as the A operand (16 rows x 16 keys per block).
        uint32_t pa[2][4];
#pragma unroll
        for (int kb2 = 0; kb2 < 2; ++kb2) {
          pa[kb2][0] = pack_bf16(s[2 * kb2][0], s[2 * kb2][1]);
          pa[kb2][1] = pack_bf16(s[2 * kb2][2], s[2 * kb2][3]);
          pa[kb2][2] = pack_bf16(s[2 * kb2 + 1][0], s[2 * kb2 + 1][1]);
          pa[kb2][3] = pack_bf16(s[2 * kb2 + 1][2], s[2 * kb2 + 1][3]);
        }
        const uint32_t vaddr = vb + (lane & 15) * RB + (lane >> 4) * 16;
#pragma unroll
        for (int dn = 0; dn < D / 8; dn += 2) {
          oacc[dn][0] *= corr_lo; oacc[dn][1] *= corr_lo;
          oacc[dn][2] *= corr_hi; oacc[dn][3] *= corr_hi;
          oacc[dn + 1][0] *= corr_lo; oacc[dn + 1][1] *= corr_lo;
          oacc[dn + 1][2] *= corr_hi; oacc[dn + 1][3] *= corr_hi;
          uint32_t b[4];
          ldsm_x4_t(vaddr + dn * 16, b);
          mma_bf16(oacc[dn], pa[0], b);
          mma_bf16(oacc[dn + 1], pa[0], b + 2);
          if (two) {
            uint32_t b2[4];
            ldsm_x4_t(vaddr + 16 * RB + dn * 16, b2);
            mma_bf16(oacc[dn], pa[1], b2);
            mma_bf16(oacc[dn + 1], pa[1], b2 + 2);
          }
        }
        // Refill the stage tile - 1 used (every warp left it before this
        // iteration's barrier) after this warp's multiplies: the warps reach
        // the copies one by one instead of all at once after the barrier.
        if (tile >= 1 && tile - 1 + AS < ntiles)
          attn_issue<T, D>(p, mode, c, ar, kst, vst, TK, tile - 1 + AS, (tile - 1) % AS);
      }
      // Warp partials -> shared memory (overwrites the stages).
      // Row pitch D + 8 floats: a warp's fragment stores (8 rows x 4 column
      // pairs) hit distinct banks.
      constexpr int OP = D + 8;
      float* opart = work;                     // [kWarps][16][OP]
      float* mpart = work + kWarps * 16 * OP;  // [kWarps][16]
      float* lpart = mpart + kWarps * 16;
      __syncthreads();
      const int r_lo = lane >> 2;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        const int col = dn * 8 + (lane & 3) * 2;
        *reinterpret_cast<float2*>(opart + (warp * 16 + r_lo) * OP + col) =
            make_float2(oacc[dn][0], oacc[dn][1]);
        *reinterpret_cast<float2*>(opart + (warp * 16 + r_lo + 8) * OP + col) =
            make_float2(oacc[dn][2], oacc[dn][3]);
      }
      if ((lane & 3) == 0) {
        mpart[warp * 16 + r_lo] = m_lo;
        lpart[warp * 16 + r_lo] = l_lo;
        mpart[warp * 16 + r_lo + 8] = m_hi;
        lpart[warp * 16 + r_lo + 8] = l_hi;
      }
      // The receive area shares no bytes with what peers still use (their
      // selection is complete and their own stages lie below it), so only
      // this CTA's partials need a barrier.
      __syncthreads();
      // Per query row: the CTA max, the weights 2^(m_w - max) of the key-group
      // warps and the weighted sum; (max, sum) go straight to the row's owner.
      const int KGW = kWarps / MB;
      float* wts = lpart + kWarps * 16;  // [G][KGW]
      if (tid < G) {
        const int qi = tid, qmb = qi >> 4, r = qi & 15;
        float mx = -INFINITY;
        for (int g = 0; g < KGW; ++g) mx = fmaxf(mx, mpart[(qmb + MB * g) * 16 + r]);
        float l = 0.f;
        for (int g = 0; g < KGW; ++g) {
          const int w = qmb + MB * g;
          const float f = safe_exp2_diff(mpart[w * 16 + r], mx);
          wts[qi * KGW + g] = f;
          l += f * lpart[w * 16 + r];
        }
        const int owner = qi / rpo, ro = qi - owner * rpo;
        float* dst = peer(recv_ml, owner) + (rank * rpo + ro) * 2;
        dst[0] = mx;
        dst[1] = l;
      }
      __syncthreads();
      // CTA partial of row qi, pushed straight to the CTA that finalises it.
      for (int e = tid; e < G * (D / 4); e += kThreads) {
        const int qi = e / (D / 4), col = (e % (D / 4)) * 4;
        const int qmb = qi >> 4, r = qi & 15;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int g = 0; g < KGW; ++g) {
          const float f = wts[qi * KGW + g];
          const float4 v = *reinterpret_cast<const float4*>(opart + ((qmb + MB * g) * 16 + r) * OP + col);
          acc.x += f * v.x; acc.y += f * v.y; acc.z += f * v.z; acc.w += f * v.w;
        }
        const int owner = qi / rpo, ro = qi - owner * rpo;
        *reinterpret_cast<float4*>(peer(recv_o, owner) + (rank * rpo + ro) * D + col) = acc;
      }
    } else {
      // ------------------------------------------------ fp32 FMA path
      float* sS = work;                    // [kMaxQ][33] logits / probabilities
      float* m_run = work + kMaxQ * 33;
      float* l_run = m_run + kMaxQ;
      float* corr_s = l_run + kMaxQ;
      const float* qf = reinterpret_cast<const float*>(qs);
      constexpr int C4 = D / 4;
      constexpr int QG = kThreads / C4;
      constexpr int QPT = kMaxQ / QG;
      float oacc[QPT][4];
#pragma unroll
      for (int i = 0; i < QPT; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[i][e] = 0.f;
      if (tid < kMaxQ) {
        m_run[tid] = -INFINITY;
        l_run[tid] = 0.f;
      }
      __syncthreads();
      for (int tile = 0; tile < ntiles; ++tile) {
        const int stage = tile % AS;
        // Tiles issued before this iteration's refill: 0 .. min(ntiles, AS + tile - 1) - 1.
        cp_async_wait_pending(tile == 0 ? min(ntiles, AS) - 1 : min(ntiles - tile - 1, AS - 2));
        __syncthreads();  // this tile's rows are visible; every warp is done with tile - 1
        // Refill the stage tile - 1 used, while this tile is computed.
        if (tile >= 1 && tile - 1 + AS < ntiles)
          attn_issue<T, D>(p, mode, c, ar, kst, vst, TK, tile - 1 + AS, (tile - 1) % AS);
        const float* kb = reinterpret_cast<const float*>(kst + stage * TK * RB);
        const float* vb = reinterpret_cast<const float*>(vst + stage * TK * RB);
        {
          const int kk = tid & 31, g = tid >> 5;
          const bool v = attn_key_valid(p, mode, c, ar, k0 + tile * TK + kk);
          for (int qi = g; qi < G; qi += 8) {
            float acc = 0.f;
            for (int col = 0; col < D; col += 4) {
              const float4 a = *reinterpret_cast<const float4*>(kb + kk * RF + col);
              const float4 b = *reinterpret_cast<const float4*>(qf + qi * RF + col);
              acc = fmaf(a.x, b.x, acc);
              acc = fmaf(a.y, b.y, acc);
              acc = fmaf(a.z, b.z, acc);
              acc = fmaf(a.w, b.w, acc);
            }
            sS[qi * 33 + kk] = v ? acc * p.scale_log2 : -INFINITY;
          }
        }
        __syncthreads();
        for (int qi = warp; qi < G; qi += kWarps) {
          const float sv = sS[qi * 33 + lane];
          const float mo = m_run[qi];
          const float mn = fmaxf(mo, warp_max(sv));
          const float base = mn == -INFINITY ? 0.f : mn;
          const float pv = fast_exp2(sv - base);
          const float sum = warp_sum(pv);
          sS[qi * 33 + lane] = pv;
          if (lane == 0) {
            const float corr = fast_exp2(mo - base);
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
      }
      __syncthreads();  // the receive area shares no bytes with what peers still use
      const int c4 = tid % C4, qg = tid / C4;
#pragma unroll
      for (int i = 0; i < QPT; ++i) {
        const int qi = qg + QG * i;
        if (qi >= G) continue;
        const int owner = qi / rpo, ro = qi - owner * rpo;
        *reinterpret_cast<float4*>(peer(recv_o, owner) + (rank * rpo + ro) * D + c4 * 4) =
            make_float4(oacc[i][0], oacc[i][1], oacc[i][2], oacc[i][3]);
        if (c4 == 0) {
          float* dst = peer(recv_ml, owner) + (rank * rpo + ro) * 2;
          dst[0] = m_run[qi];
          dst[1] = l_run[qi];
        }
      }
    }
    cluster.sync();
    // Finalise this CTA's query rows [rank * rpo, ...): merge the cs partials,
    // four output columns per thread.
    const int q0 = rank * rpo, q1 = min(G, q0 + rpo);
    for (int e = tid; e < (q1 - q0) * (D / 4); e += kThreads) {
      const int ro = e / (D / 4), col = (e % (D / 4)) * 4;
      float mx = -INFINITY;
      for (int r = 0; r < cs; ++r) mx = fmaxf(mx, recv_ml[(r * rpo + ro) * 2]);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float l = 0.f;
      for (int r = 0; r < cs; ++r) {
        const float f = safe_exp2_diff(recv_ml[(r * rpo + ro) * 2], mx);
        const float4 v = *reinterpret_cast<const float4*>(recv_o + (r * rpo + ro) * D + col);
        acc.x += f * v.x; acc.y += f * v.y; acc.z += f * v.z; acc.w += f * v.w;
        l += f * recv_ml[(r * rpo + ro) * 2 + 1];
      }
      const float inv = 1.f / l;
      const int qi = q0 + ro;
      *reinterpret_cast<float4*>(p.o + (unit * G + qi) * D + col) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      if (col == 0 && p.lse != nullptr) p.lse[unit * G + qi] = (mx + log2f(l)) * kLn2;
    }
  }
  tc_fence_before();
  // Peers may still read or write this CTA's shared memory, unless the attend
  // phase ran: its cluster barrier followed the last such access.
  if (mode & kModeAttend)
    __syncthreads();
  else
    cluster.sync();
  if (use_tmem && warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename T, int D>
cudaError_t launch_typed(int64_t units, const PathParams& prm, size_t smem, cudaStream_t stream) {
  // The constant-folded variants serve bf16 steps with every phase, the
  // all-gather final selection and resident token logits.
  int var = 0;
  if (sizeof(T) == 2 && prm.mode == (kModeScore | kModeFilter | kModeAttend) && prm.gather_all &&
      prm.filter_fast == 1)
    var = prm.fuse_dwt ? 1 : (prm.al != nullptr ? 2 : 0);
  void (*kern)(const PathParams) = path_kernel<T, D, 0>;
  if constexpr (sizeof(T) == 2) {
    if (var == 1) kern = path_kernel<T, D, 1>;
    if (var == 2) kern = path_kernel<T, D, 2>;
  }
  // The constant-folded instantiations take 16 keys per warp per tile: a plan
  // of 32 (four query-row blocks) runs as half-size tiles in twice the
  // stages, the same shared-memory bytes.
  PathParams pk = prm;
  if (var != 0 && pk.G > 32 && pk.tile_keys == 64) {
    pk.tile_keys = 32;
    pk.a_stages = std::min(6, 2 * pk.a_stages);
  }
  cudaError_t e = cudaSuccess;
  if (var == 1) {
    if constexpr (sizeof(T) == 2) e = ensure_max_smem<path_kernel<T, D, 1>>();
  } else if (var == 2) {
    if constexpr (sizeof(T) == 2) e = ensure_max_smem<path_kernel<T, D, 2>>();
  } else {
    e = ensure_max_smem<path_kernel<T, D, 0>>();
  }
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.cs, static_cast<unsigned>(units), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = prm.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, pk);
}

// cuTensorMapEncodeTiled from the driver, looked up once (no link-time
// dependency on the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static std::atomic<void*> cached{nullptr};
  void* f = cached.load(std::memory_order_acquire);
  if (f == nullptr) {
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || f == nullptr) {
      (void)cudaGetLastError();
      return nullptr;
    }
    cached.store(f, std::memory_order_release);
  }
  return reinterpret_cast<EncodeTiledFn>(f);
}

// Tensor map of K_p [units * N_p rows, d columns] (bf16) with a box of 64
// columns x box_rows rows and the 128-byte swizzle of the tensor-core operand
// layout.  Returns false if unavailable.
bool encode_span_map(const LaunchDims& ld, const void* kp, CUtensorMap* map, int box_rows) {
  if (ld.dtype != WF_BF16 || kp == nullptr || box_rows < 8 || box_rows > 256) return false;
  const EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(ld.head_dim),
                              static_cast<cuuint64_t>(ld.units) * ld.n_prompt};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld.head_dim) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kp), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A cached fp32 A_L [U, P, d] as a 2-D tensor for tensor copies of 64-row,
// 32-column boxes with 128-byte swizzle.
bool encode_al_map(const LaunchDims& ld, const float* al, CUtensorMap* map) {
  const EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr || al == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(ld.head_dim),
                              static_cast<cuuint64_t>(ld.units) * (ld.n_prompt >> ld.levels)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld.head_dim) * 4};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kScoreChunk)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(al), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t smem_bytes(const LaunchDims& ld, const PathParams& p) {
  if (ld.dtype == WF_BF16)
    return ld.head_dim == 128 ? PathSmem<__nv_bfloat16, 128>(p).total
                              : PathSmem<__nv_bfloat16, 64>(p).total;
  return ld.head_dim == 128 ? PathSmem<float, 128>(p).total : PathSmem<float, 64>(p).total;
}

int pow2_floor(int x) {
  int p = 1;
  while (p * 2 <= x) p *= 2;
  return p;
}

}  // namespace

int device_sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return 152;  // GB300
  }
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
    (void)cudaGetLastError();
    return 152;
  }
  cached[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Plans a launch of the phases in `mode` (see PathPlan).  k may be null when
// the filter phase is not run (kL and budget come from the arguments).
bool plan_path(const LaunchDims& ld, int mode, const int32_t* k, int k_l, int budget,
               int sm_count, PathPlan* plan) {
  PathParams p = {};
  const bool want_fuse = mode == (kPhaseAll | kPhaseFuseDwt);
  const bool want_al = mode == (kPhaseAll | kPhaseCachedAl) || mode == (kPhaseScore | kPhaseCachedAl);
  mode &= kPhaseAll;
  p.mode = mode;
  p.G = ld.n_gen;
  p.GZ = coarse_logit_pitch(ld.n_gen);
  p.levels = ld.levels;
  p.n_prompt = ld.n_prompt;
  p.P = ld.n_prompt >> ld.levels;
  p.kL = k_l;
  p.budget = budget;
  p.n_keys = budget + ld.n_gen;
  // Preferred cluster: one wave of clusters at one CTA per SM (the largest
  // power of two with units * cs <= SMs), capped by the work each phase can
  // split.  If that does not fit in shared memory, larger clusters (smaller
  // per-CTA slices) are tried before giving up.
  int cs0 = pow2_floor(std::max(1, static_cast<int>(std::min<int64_t>(kMaxCluster, sm_count / std::max<int64_t>(1, ld.units)))));
  auto cluster_ok = [&](int c) {
    if ((mode & kModeScore) && (p.P % c != 0 || p.P / c < 8)) return false;
    if ((mode & kModeFilter) && k_l < c) return false;
    if ((mode & kModeAttend) && p.n_keys < 16 * c) return false;
    return true;
  };
  while (cs0 > 1 && !cluster_ok(cs0)) cs0 /= 2;
  int cs = cs0;
  size_t smem = 0;
  bool t_in_smem = true;
  bool found = false;
  // The fast filter (token logits on tcgen05 through a tensor-copy ring) serves
  // bf16 inputs whose schedule selects only at the token level below L (every
  // level in between keeps all children; the default schedule) with spans of
  // 8..256 rows.
  bool fast_sched = (mode & kModeFilter) && ld.dtype == WF_BF16 && ld.levels >= 3 &&
                    ld.levels <= 8 && k != nullptr;
  if (fast_sched) {
    for (int j = 1; j < ld.levels; ++j)
      if (k[j] < 2 * k[j + 1]) fast_sched = false;
    if (k[0] >= 2 * k[1]) fast_sched = false;
  }
  for (;; cs *= 2) {
    p.cs = cs;
    p.per_cta_p = (mode & kModeScore) ? p.P / cs : 0;
    const int spans_cap = (mode & kModeFilter) ? (k_l + cs - 1) / cs : 0;
    p.rows_cap = spans_cap << ld.levels;
    int sc = 1;
    while (sc < std::max(k_l, 1)) sc <<= 1;
    p.sorted_cap = (mode & kModeFilter) ? sc : 0;
    p.keys_cap = std::max(p.per_cta_p, p.rows_cap);
    p.klist_cap = (mode & kModeAttend) ? (p.n_keys + cs - 1) / cs + 1 : 0;
    if (ld.dtype == WF_BF16) {
      const int mb = ld.n_gen <= 16 ? 1 : (ld.n_gen <= 32 ? 2 : 4);
      p.tile_keys = (mb == 4 ? 32 : 16) * (kWarps / mb);  // 64 keys: 16 or 32 per warp
    } else {
      p.tile_keys = 32;
    }
    // cp.async ring depths: every tile in flight when it fits (at most 6).
    const int f_tiles = (p.rows_cap + kTileRows - 1) / kTileRows;
    const int a_tiles = ((p.n_keys + cs - 1) / cs + p.tile_keys - 1) / p.tile_keys;
    const int f_want = std::max(2, std::min(6, f_tiles));
    const int a_want = std::max(2, std::min(6, a_tiles));
    // Fused step 1 needs one score chunk per CTA and whole spans per stage.
    const int elem = ld.dtype == WF_BF16 ? 2 : 4;
    const bool fuse_try = want_fuse && p.per_cta_p <= kScoreChunk &&
                          (static_cast<int64_t>(elem) * ld.head_dim << ld.levels) <= kFuseStageBytes;
    // Cached A_L staged by bulk copies (bf16 queries; the logits of every
    // position of the CTA resident at once).
    const bool al_try = want_al && ld.dtype == WF_BF16 && p.per_cta_p <= kZRows;
    // Prefer the fused step 1, the gather-all selection and token logits in
    // shared memory, in that order.
    // Fast filter: resident accumulators when every tile has its own columns
    // (ntiles * N <= 512), else four rotating ones; ring of up to 4 tiles.
    const int n_cols = (ld.n_gen + 15) & ~15;
    const int f_ntl = (p.rows_cap + 127) / 128;
    const bool f_res = f_ntl * n_cols <= 512;
    const int f_nb = f_res ? f_ntl : std::min(4, 512 / n_cols);
    const int s_want = std::min(std::min(4, f_ntl), f_nb);
    // The fast filter prefers the all-gather selection, then the deepest
    // tile ring, then the deepest attention ring (the phases share one
    // region, so the two depths are independent); the general path trades
    // ring depth against the all-gather.
    for (int ff = fast_sched ? 1 : 0; ff >= 0 && !found; --ff)
    for (int fz = fuse_try || al_try ? 1 : 0; fz >= 0 && !found; --fz)
    for (int it = 0; it < (ff ? 2 * 4 * 5 : 10) && !found; ++it) {
      int ga, fs, as;
      if (ff) {
        ga = 1 - it / 20;
        fs = std::max(1, s_want - (it % 20) / 5);
        as = std::max(2, a_want - it % 5);
        if (ga && fs < std::min(2, s_want)) continue;  // no all-gather at the cost of a serial ring
      } else {
        ga = 1 - (it & 1);
        fs = std::max(2, f_want - (it >> 1));
        as = std::max(2, a_want - (it >> 1));
      }
      p.filter_fast = ff ? (f_res ? 1 : 2) : 0;
      p.f_nb = ff ? f_nb : 0;
      p.f_stages = fs;
      p.a_stages = as;
      if (ga && (!(mode & kModeFilter) || static_cast<int64_t>(cs) * p.rows_cap > 8192)) continue;
      p.gather_all = ga;
      p.fuse_dwt = fuse_try ? fz : 0;
      p.al_stage = al_try ? fz : 0;
      p.t_ws = nullptr;
      // Every A_L stage resident (no refill latency) if that fits, else a ring of three.
      p.al_ring = (p.per_cta_p + kScoreChunk - 1) / kScoreChunk;
      if (p.al_stage && p.al_ring > kFuseStages && smem_bytes(ld, p) > kMaxSmem) p.al_ring = kFuseStages;
      smem = smem_bytes(ld, p);
      t_in_smem = true;
      if (ff) {
        found = smem <= kMaxSmem;
        continue;
      }
      if ((mode & kModeFilter) && smem > kMaxSmem) {
        p.t_ws = reinterpret_cast<float*>(16);  // placeholder: only its nullness matters here
        smem = smem_bytes(ld, p);
        t_in_smem = false;
      }
      found = smem <= kMaxSmem && (t_in_smem || !fz);  // never fuse at the cost of spilling
    }
    if (found || cs * 2 > kMaxCluster || !cluster_ok(cs * 2)) break;
  }
  plan->cluster = cs;
  plan->smem_bytes = smem;
  plan->t_in_smem = t_in_smem;
  plan->t_bytes = t_in_smem ? 0
                            : sizeof(float) * static_cast<size_t>(ld.units) * cs * p.rows_cap *
                                  ((ld.n_gen + 3) & ~3);  // spilled row pitch
  plan->per_cta_p = p.per_cta_p;
  plan->rows_cap = p.rows_cap;
  plan->sorted_cap = p.sorted_cap;
  plan->keys_cap = p.keys_cap;
  plan->gather_all = p.gather_all;
  plan->klist_cap = p.klist_cap;
  plan->tile_keys = p.tile_keys;
  plan->f_stages = p.f_stages;
  plan->a_stages = p.a_stages;
  plan->fuse_dwt = p.fuse_dwt;
  plan->al_stage = p.al_stage;
  plan->al_ring = p.al_ring;
  plan->filter_fast = p.filter_fast;
  plan->f_nb = p.f_nb;
  plan->mode = mode;
  return smem <= kMaxSmem;
}

cudaError_t launch_path(const LaunchDims& ld, const PathPlan& plan, const PathArgs& a,
                        cudaStream_t stream) {
  PathParams p = {};
  p.q = a.q;
  p.kp = a.kp;
  p.vp = a.vp;
  p.kg = a.kg;
  p.vg = a.vg;
  p.zl = a.zl;
  p.al = a.al;
  p.idx_l_in = a.idx_l_in;
  p.idx_in = a.idx_in;
  p.idx_l_out = a.idx_l_out;
  p.scores_out = a.scores_out;
  p.idx_out = a.idx_out;
  p.o = a.o;
  p.lse = a.lse;
  p.status = a.status;
  p.t_ws = plan.t_in_smem ? nullptr : a.t_ws;
  p.mode = plan.mode;
  p.n_prompt = ld.n_prompt;
  p.G = ld.n_gen;
  p.GZ = coarse_logit_pitch(ld.n_gen);
  p.levels = ld.levels;
  p.P = ld.n_prompt >> ld.levels;
  p.kL = a.k_l;
  p.budget = a.budget;
  p.n_keys = a.budget + ld.n_gen;
  p.cs = plan.cluster;
  p.per_cta_p = plan.per_cta_p;
  p.rows_cap = plan.rows_cap;
  p.sorted_cap = plan.sorted_cap;
  p.keys_cap = plan.keys_cap;
  p.gather_all = plan.gather_all;
  p.klist_cap = plan.klist_cap;
  p.tile_keys = plan.tile_keys;
  p.f_stages = plan.f_stages;
  p.a_stages = plan.a_stages;
  p.fuse_dwt = plan.fuse_dwt;
  p.al_stage = plan.al_stage;
  p.al_ring = plan.al_ring;
  if (plan.al_stage && !encode_al_map(ld, a.al, &p.tmap_al)) return cudaErrorInvalidValue;
  p.inject_polls = plan.fuse_dwt ? consume_wait_injection() : 0u;
  p.filter_fast = plan.filter_fast;
  p.f_nb = plan.f_nb;
  if (plan.filter_fast) {
    // The fast filter's tiles come only through tensor copies.
    if (!encode_span_map(ld, a.kp, &p.tmap_spans, std::min(1 << ld.levels, 128)))
      return cudaErrorNotSupported;
    p.use_tma_spans = 1;
  } else {
    p.use_tma_spans = (plan.mode & kModeFilter) != 0 && ld.levels >= 3 && ld.levels <= 8 &&
                              encode_span_map(ld, a.kp, &p.tmap_spans, 1 << ld.levels)
                          ? 1
                          : 0;
  }
  p.al_scale = static_cast<float>(std::pow(2.0, -0.5 * ld.levels));  // 2^(-L/2)
  for (int j = 0; j <= ld.levels; ++j) {
    p.k[j] = a.k != nullptr ? a.k[j] : 0;
    p.scale[j] = static_cast<float>(std::pow(2.0, -0.5 * j) / std::sqrt(static_cast<double>(ld.head_dim)));
  }
  p.inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(ld.head_dim)));
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(ld.head_dim)));
  if (ld.dtype == WF_BF16) {
    if (ld.head_dim == 128) return launch_typed<__nv_bfloat16, 128>(ld.units, p, plan.smem_bytes, stream);
    return launch_typed<__nv_bfloat16, 64>(ld.units, p, plan.smem_bytes, stream);
  }
  if (ld.head_dim == 128) return launch_typed<float, 128>(ld.units, p, plan.smem_bytes, stream);
  return launch_typed<float, 64>(ld.units, p, plan.smem_bytes, stream);
}

}  // namespace wf
