// Device helpers shared by the WaveFilter kernels (sm_103a).
//
// Contents: 16-byte vector loads with bf16 -> fp32 widening, warp/block scans,
// thread-block-cluster helpers (DSMEM), mbarrier + bulk-copy (TMA engine)
// helpers with bounded waits, and the cluster-wide exact Top-K used by the
// coarse selection and every recursive-filtering level.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wavefilter.h"

namespace wf {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;  // every kernel of this library uses 256-thread CTAs
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
// Bounded waits: an mbarrier that has not completed after this many polls
// sets WF_DEV_WAIT_TIMEOUT and the CTA gives up instead of spinning forever.
constexpr uint32_t kWaitPolls = 1u << 24;

// ---------------------------------------------------------------- status word
__device__ __forceinline__ void raise_flag(int32_t* status, int code) {
  if (status != nullptr) atomicOr(status, code);
}

// ------------------------------------------------------------------ loads
template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kPer16B = 8;
};
template <>
struct Elem<float> {
  static constexpr int kPer16B = 4;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Loads 16 bytes (read-only path) and widens them to fp32.
__device__ __forceinline__ void load16_f32(const __nv_bfloat16* p, float* f) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}
__device__ __forceinline__ void load16_f32(const float* p, float* f) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(p));
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
// Streaming 16-byte load (read-only path, no L1 allocation).  Being volatile,
// consecutive calls are issued in program order, so a run of them keeps that
// many requests in flight before the first result is used.
__device__ __forceinline__ uint4 ldg16_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void widen16(const uint4& v, const __nv_bfloat16*, float* f) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}
__device__ __forceinline__ void widen16(const uint4& v, const float*, float* f) {
  f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}

__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(float x) { return x; }

// 2^x by the hardware approximation (ex2.approx.ftz: relative error below
// 2^-22; results below 2^-126 flush to zero, which only drops softmax terms
// that vanish beside the maximum).  The softmax statistics, scores and
// attention weights of the path all use it.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Inclusive prefix sum over the warp.
__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// Block-wide exclusive scan of one int per thread; returns the exclusive
// prefix and writes the block total to *total.  `scratch` holds kWarps + 1
// ints.  Contains three __syncthreads(), so back-to-back calls may reuse
// the same scratch.
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int incl = warp_incl_scan(v);
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? scratch[lane] : 0;
    const int wi = warp_incl_scan(w);
    if (lane < kWarps) scratch[lane] = wi - w;
    if (lane == kWarps - 1) scratch[kWarps] = wi;
  }
  __syncthreads();
  const int excl = scratch[warp] + incl - v;
  *total = scratch[kWarps];
  __syncthreads();
  return excl;
}

// ------------------------------------------------------------------ shared memory
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier + bulk copy
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase.  Returns false (and raises
// WF_DEV_WAIT_TIMEOUT) if the phase did not complete within `polls` polls
// (kWaitPolls unless a test injects a shorter limit).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  int32_t* status,
                                                  uint32_t polls = kWaitPolls) {
  for (uint32_t i = 0; i < polls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  raise_flag(status, WF_DEV_WAIT_TIMEOUT);
  return false;
}
// Plain arrival (no transaction bytes) on an mbarrier.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Barrier among a subset of the CTA's warps (named barrier `id` >= 1, `count`
// threads, a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// One bulk global -> shared copy through the TMA engine; completion is
// signalled on `bar` as transaction bytes.  dst, src and bytes must be
// multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ cp.async row gathers
// 16-byte asynchronous global -> shared copies (L2 only), grouped and waited
// on with commit/wait groups.  Used for gathers of many small rows, where
// one instruction per thread per 16 bytes keeps the copies in flight without
// per-copy descriptor overhead.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ cluster exchanges
//
// Every exchange between the CTAs of a cluster is push-based: a CTA stores
// its contribution straight into its peers' shared memory (distributed
// shared memory stores do not stall the writer), one cluster barrier
// (release/acquire) makes the data visible, and every CTA then reads its own
// shared memory.  A buffer written by peers is not written again before
// every CTA has passed at least one more cluster barrier after reading it.

template <typename P>
__device__ __forceinline__ P* peer(P* local, int rank) {
  return cg::this_cluster().map_shared_rank(local, rank);
}

// (m, l) softmax-statistics merge in the log2 domain (l = Σ 2^(z - m));
// pairs with m = -inf (empty) are skipped.
__device__ __forceinline__ void merge_ml(float& m, float& l, float m2, float l2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    l = l2;
    return;
  }
  const float mx = fmaxf(m, m2);
  l = l * fast_exp2(m - mx) + l2 * fast_exp2(m2 - mx);
  m = mx;
}

constexpr int kMaxQ = 64;  // maximum queries per unit

// All-reduce of per-query softmax statistics (log2 domain) over the cluster.
// loc_m/loc_l hold this CTA's (max, Σ 2^(z - max)) per query; on return
// gm/ginv hold the cluster-wide max and 1 / sum.  stat_in: [kMaxCluster][2]
// [kMaxQ] floats.  If counts_in is not null, `my_count` is all-gathered into
// counts_in[rank] in the same exchange.  One cluster barrier.
static __device__ __noinline__ void cluster_merge_stats(const float* loc_m, const float* loc_l, int G,
                                           float* stat_in, float* gm, float* ginv,
                                           int my_count = 0, int32_t* counts_in = nullptr) {
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = static_cast<int>(cluster.num_blocks());
  const int me = static_cast<int>(cluster.block_rank());
  for (int e = threadIdx.x; e < G * cs; e += kThreads) {
    const int q = e % G, r = e / G;
    float* dst = peer(stat_in, r) + me * 2 * kMaxQ;
    dst[q] = loc_m[q];
    dst[kMaxQ + q] = loc_l[q];
  }
  if (counts_in != nullptr && threadIdx.x < cs) peer(counts_in, threadIdx.x)[me] = my_count;
  cluster.sync();
  for (int q = threadIdx.x; q < G; q += kThreads) {
    float m = -INFINITY, l = 0.f;
    for (int r = 0; r < cs; ++r) merge_ml(m, l, stat_in[r * 2 * kMaxQ + q], stat_in[r * 2 * kMaxQ + kMaxQ + q]);
    gm[q] = m;
    ginv[q] = 1.f / l;
  }
  __syncthreads();
}

// Split cluster barrier: every thread arrives once early (relaxed, no
// ordering) and waits later, e.g. so that no CTA touches a peer's shared
// memory before every CTA of the cluster has started.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ cluster Top-K
//
// Exact selection of the k largest 32-bit keys spread over the CTAs of a
// cluster.  Candidates live in each CTA's shared memory in ascending
// position order, and every position held by rank r is below every position
// held by rank r+1, so "lower position wins a tie" is "lower rank, then lower
// local index wins".  Keys are the IEEE bit patterns of non-negative floats,
// whose unsigned order equals their numeric order.
//
// Three radix rounds (11, 11, 10 bits, most significant first) find the k-th
// largest key T; every key > T is taken, plus the first (k - #{key > T}) keys
// equal to T in (rank, index) order.  When a round's boundary bin is taken
// whole, T becomes the bin's lowest value minus one with no ties, and the
// remaining rounds are skipped.  Two variants: gather-all (every CTA
// receives every key and selects locally; one cluster barrier) for small
// candidate sets, and distributed (histograms reduce-scattered and
// all-gathered through DSMEM; two barriers per round) for large ones.
struct TopkSmem {
  uint32_t hist[3][2048];          // digit histograms (one per radix round)
  uint32_t region[3][32];          // per-round counts of 32 equal bin ranges
  int32_t cnt_in[kMaxCluster][2];  // distributed: (#> T, #== T) pushed by each rank
  int32_t wcnt[2][kWarps];         // block select: per-warp (#> T, #== T)
  int32_t scan[kWarps + 1];
  int32_t bcast[4];
};

struct TopkResult {
  int local_taken;  // selected candidates in this CTA
  int offset;       // selected candidates in lower ranks
};

// Digit d* of a histogram with #{digit > d*} < need <= #{digit >= d*}.
// Returns d* and stores #{digit > d*} in *above.  Block-wide.
__device__ inline uint32_t find_digit(const uint32_t* total, int nb, int need, TopkSmem& sm,
                                      int* above) {
  const int tid = threadIdx.x;
  const int per = nb / kThreads;
  const int owner = kThreads - 1 - tid;  // thread 0 owns the highest bins
  int mine = 0;
  for (int b = 0; b < per; ++b) mine += static_cast<int>(total[owner * per + b]);
  int tot;
  const int above_owner = block_excl_scan(mine, sm.scan, &tot);
  if (above_owner < need && above_owner + mine >= need) {
    int acc = above_owner;
    for (int b = per - 1; b >= 0; --b) {
      const int c = static_cast<int>(total[owner * per + b]);
      if (acc + c >= need) {
        sm.bcast[0] = owner * per + b;
        sm.bcast[1] = acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
  *above = sm.bcast[1];
  const uint32_t d = static_cast<uint32_t>(sm.bcast[0]);
  __syncthreads();
  return d;
}

__device__ __forceinline__ int round_shift(int round) { return round == 0 ? 21 : (round == 1 ? 10 : 0); }
__device__ __forceinline__ int round_bins(int round) { return round == 2 ? 1024 : 2048; }

// Marks take[i] for local candidates given the threshold, this CTA's tie
// quota; block-wide.
__device__ inline void mark_taken(const uint32_t* keys, int n, uint32_t thr, int quota,
                                  uint8_t* take, TopkSmem& sm) {
  int carry = 0;
  for (int base = 0; base < n; base += kThreads) {
    const int i = base + threadIdx.x;
    const uint32_t key = i < n ? keys[i] : 0u;
    const int is_eq = (i < n) && key == thr;
    int tot;
    const int before = block_excl_scan(is_eq, sm.scan, &tot);
    if (i < n) take[i] = static_cast<uint8_t>(key > thr || (is_eq && carry + before < quota));
    carry += tot;
  }
  __syncthreads();
}

// Distributed variant (any candidate count).
static __device__ __noinline__ TopkResult topk_distributed(const uint32_t* keys, int n, int k, uint8_t* take,
                                              TopkSmem& sm) {
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = static_cast<int>(cluster.num_blocks());
  const int me = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x;
  uint32_t* hist = sm.hist[0];     // local histogram
  uint32_t* total = sm.hist[1];    // cluster-wide histogram
  uint32_t* part_in = sm.hist[2];  // slices pushed by the peers
  uint32_t prefix = 0, pmask = 0;
  int need = k;
#pragma unroll 1
  for (int round = 0; round < 3; ++round) {
    const int shift = round_shift(round), nb = round_bins(round);
    const int sl = nb / cs;  // bins owned by each rank
    for (int b = tid; b < nb; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t key = keys[i];
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    for (int b = tid; b < nb; b += kThreads) peer(part_in, b / sl)[me * sl + (b % sl)] = hist[b];
    cluster.sync();
    for (int e = tid; e < sl * cs; e += kThreads) {
      const int bl = e % sl, r = e / sl;
      uint32_t t = 0;
      for (int src = 0; src < cs; ++src) t += part_in[src * sl + bl];
      peer(total, r)[me * sl + bl] = t;
    }
    cluster.sync();
    int above;
    const uint32_t digit = find_digit(total, nb, need, sm, &above);
    need -= above;
    prefix |= digit << shift;
    pmask |= static_cast<uint32_t>(nb - 1) << shift;
    // Early exit as in block_select_topk (total is the same on every rank).
    if (round < 2 && static_cast<int>(total[digit]) == need && prefix != 0u) {
      prefix -= 1u;
      need = 0;
      break;
    }
  }
  const uint32_t thr = prefix;
  int gt = 0, eq = 0;
  for (int i = tid; i < n; i += kThreads) {
    gt += keys[i] > thr;
    eq += keys[i] == thr;
  }
  int tot_gt, tot_eq;
  (void)block_excl_scan(gt, sm.scan, &tot_gt);
  (void)block_excl_scan(eq, sm.scan, &tot_eq);
  if (tid < cs) {
    int32_t* dst = peer(&sm.cnt_in[0][0], tid) + 2 * me;
    dst[0] = tot_gt;
    dst[1] = tot_eq;
  }
  cluster.sync();
  int quota_me = 0, offset = 0, ties_before = 0;
  for (int r = 0; r < cs; ++r) {
    const int g = sm.cnt_in[r][0], e = sm.cnt_in[r][1];
    int q = need - ties_before;
    q = q < 0 ? 0 : (q > e ? e : q);
    if (r < me) offset += g + q;
    if (r == me) quota_me = q;
    ties_before += e;
  }
  mark_taken(keys, n, thr, quota_me, take, sm);
  return TopkResult{tot_gt + quota_me, offset};
}

// ------------------------------------------------------------------ block Top-K
//
// Block-wide exact Top-k over keys[0, n) in this CTA's shared memory (index
// order is the tie order: lower index wins).  Radix rounds of 11/11/10 bits,
// each histogram in its own pre-zeroed buffer, so a round costs one barrier:
// every warp then finds the round's digit redundantly (vectorised bin sums,
// a warp scan over lanes and a second warp scan inside the boundary lane's
// bins).  Counts of the keys above the threshold and of the ties per 32-key
// sub-chunk, scanned, give every selected key its rank among the selected
// (ascending index), and only the sub-chunks holding slots of the caller's
// range are emitted.  A round whose boundary bin is taken whole ends the
// search early (usually after the second round).
// Digit d of the round with #{digit > d} < need <= #{digit >= d}, found by one
// warp from the 32 range counts (lane 0 = highest range) and then the bins of
// the boundary range (descending, per/32 bins per lane).  Every lane returns
// the digit and #{digit > d}.
__device__ __forceinline__ void warp_find_digit(const uint32_t* h, const uint32_t* region, int nb,
                                                int need, uint32_t* digit, int* above) {
  const int lane = threadIdx.x & 31;
  const int per = nb / 32;  // 64 or 32 bins per range
  const int rc = static_cast<int>(region[31 - lane]);
  const int incl = warp_incl_scan(rc);
  const int before = incl - rc;
  const unsigned owner_mask = __ballot_sync(0xffffffffu, before < need && incl >= need);
  const int owner = __ffs(owner_mask) - 1;
  const int base = __shfl_sync(0xffffffffu, before, owner);
  const int obin0 = (31 - owner) * per;  // lowest bin of the boundary range
  const int w = per / 32;                // 2 or 1
  const int hi_bin = obin0 + per - 1 - lane * w;
  const int c0 = static_cast<int>(h[hi_bin]);
  const int c1 = w > 1 ? static_cast<int>(h[hi_bin - 1]) : 0;
  const int incl2 = warp_incl_scan(c0 + c1);
  const int pre = base + incl2 - (c0 + c1);
  int my_digit = -1, my_above = 0;
  if (pre < need && pre + c0 >= need) {
    my_digit = hi_bin;
    my_above = pre;
  } else if (w > 1 && pre + c0 < need && pre + c0 + c1 >= need) {
    my_digit = hi_bin - 1;
    my_above = pre + c0;
  }
  const unsigned m2 = __ballot_sync(0xffffffffu, my_digit >= 0);
  const int src = __ffs(m2) - 1;
  *digit = static_cast<uint32_t>(__shfl_sync(0xffffffffu, my_digit, src));
  *above = __shfl_sync(0xffffffffu, my_above, src);
}

// Writes out[slot - lo] = i for every selected key i whose rank among the
// selected (ascending index) falls in [lo, hi).
// Zeroes the histograms of block_select_topk (block-wide, no barrier); a
// caller may do this ahead of time, off its critical path.
__device__ __forceinline__ void topk_zero(TopkSmem& sm) {
  for (int b = threadIdx.x; b < 3 * 2048; b += kThreads) (&sm.hist[0][0])[b] = 0;
  if (threadIdx.x < 3 * 32) (&sm.region[0][0])[threadIdx.x] = 0;
}

// `prezeroed`: the histograms were zeroed (topk_zero, followed by a barrier)
// since their last use.  `map` (nullable): out receives map[i] instead of i.
static __device__ __noinline__ void block_select_topk(const uint32_t* keys, int n, int k, int lo_slot,
                                               int hi_slot, int32_t* out, TopkSmem& sm,
                                               bool prezeroed = false,
                                               const int32_t* map = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (!prezeroed) {
    topk_zero(sm);
    __syncthreads();
  }
  uint32_t prefix = 0, pmask = 0;
  int need = k;
#pragma unroll 1
  for (int round = 0; round < 3; ++round) {
    const int shift = round == 0 ? 21 : (round == 1 ? 10 : 0);
    const int nb = round == 2 ? 1024 : 2048;
    uint32_t* h = sm.hist[round];
    const int per = nb / 32;
#pragma unroll 4
    for (int base = 0; base < n; base += kThreads) {  // whole warps iterate together
      const int i = base + tid;
      const uint32_t kv = i < n ? keys[i] : 0u;
      const bool active = i < n && (kv & pmask) == prefix;
      const uint32_t bin = (kv >> shift) & (nb - 1);
      if (active) {
        atomicAdd(&h[bin], 1u);
        atomicAdd(&sm.region[round][bin / per], 1u);
      }
    }
    __syncthreads();
    uint32_t digit;
    int above;
    warp_find_digit(h, sm.region[round], nb, need, &digit, &above);
    need -= above;
    prefix |= digit << shift;
    pmask |= static_cast<uint32_t>(nb - 1) << shift;
    // Early exit: every key of the boundary bin is taken, so the threshold is
    // the bin's lowest value (every key > prefix - 1) and no tie remains.
    // (Same decision in every warp: all read the same histogram.)
    if (round < 2 && static_cast<int>(h[digit]) == need && prefix != 0u) {
      prefix -= 1u;
      need = 0;
      break;
    }
  }
  const uint32_t thr = prefix;
  const int S = (n + 31) >> 5;  // 32-key sub-chunks
  if (S <= kThreads) {
    // Counts of keys above the threshold and of ties per sub-chunk (warp w
    // takes sub-chunks w, w + kWarps, ...), in the spent first histogram;
    // exclusive scans over the sub-chunks give each one its first slot, so
    // only the sub-chunks holding slots of [lo_slot, hi_slot) are emitted,
    // spread over the warps.
    __syncthreads();  // every warp is done reading the histograms
    int32_t* sgt = reinterpret_cast<int32_t*>(sm.hist[0]);
    int32_t* seq = sgt + kThreads;
    int32_t* sslot = seq + kThreads;      // S + 1 entries
    int32_t* stie = sslot + kThreads + 1;
    for (int sc = warp; sc < S; sc += kWarps) {
      const int i = sc * 32 + lane;
      const uint32_t kv = i < n ? keys[i] : 0u;
      const int g = __popc(__ballot_sync(0xffffffffu, i < n && kv > thr));
      const int e = __popc(__ballot_sync(0xffffffffu, i < n && kv == thr));
      if (lane == 0) {
        sgt[sc] = g;
        seq[sc] = e;
      }
    }
    __syncthreads();
    const int g = tid < S ? sgt[tid] : 0, e = tid < S ? seq[tid] : 0;
    int tot_g, tot_e;
    const int gb = block_excl_scan(g, sm.scan, &tot_g);
    const int eb = block_excl_scan(e, sm.scan, &tot_e);
    if (tid < S) {
      sslot[tid] = gb + min(need, eb);  // selected keys before the sub-chunk
      stie[tid] = eb;                   // ties before it
    }
    if (tid == 0) sslot[S] = tot_g + min(need, tot_e);
    __syncthreads();
    for (int sc = warp; sc < S; sc += kWarps) {
      const int s0 = sslot[sc], s1 = sslot[sc + 1];
      if (s1 <= lo_slot || s0 >= hi_slot) continue;  // no slot of the range here
      const int i = sc * 32 + lane;
      const uint32_t kv = i < n ? keys[i] : 0u;
      const unsigned below = (1u << lane) - 1u;
      const unsigned eqm = __ballot_sync(0xffffffffu, i < n && kv == thr);
      const bool tie_taken = (eqm >> lane & 1u) && stie[sc] + __popc(eqm & below) < need;
      const bool taken = (i < n && kv > thr) || tie_taken;
      const unsigned tm = __ballot_sync(0xffffffffu, taken);
      const int my_slot = s0 + __popc(tm & below);
      if (taken && my_slot >= lo_slot && my_slot < hi_slot) out[my_slot - lo_slot] = map ? map[i] : i;
    }
    __syncthreads();
    return;
  }
  // Larger sets: fused compaction, warp w owns keys [lo, hi).
  const int chunk = (((n + kWarps - 1) / kWarps) + 31) & ~31;
  const int lo = min(n, warp * chunk), hi = min(n, lo + chunk);
  int gt = 0, eq = 0;
#pragma unroll 4
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const uint32_t kv = i < hi ? keys[i] : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, i < hi && kv > thr));
    eq += __popc(__ballot_sync(0xffffffffu, i < hi && kv == thr));
  }
  if (lane == 0) {
    sm.wcnt[0][warp] = gt;
    sm.wcnt[1][warp] = eq;
  }
  __syncthreads();
  // Selected keys and ties before this warp's chunk: exclusive scans of the
  // per-warp counts (lane w holds warp w's); the ties taken before a chunk
  // are min(need, ties seen before it).
  int gi = 0, ei = 0;
  if (lane < kWarps) {
    gi = sm.wcnt[0][lane];
    ei = sm.wcnt[1][lane];
  }
  const int gw = gi, ew = ei;
#pragma unroll
  for (int off = 1; off < kWarps; off <<= 1) {
    const int g2 = __shfl_up_sync(0xffffffffu, gi, off), e2 = __shfl_up_sync(0xffffffffu, ei, off);
    if (lane >= off) {
      gi += g2;
      ei += e2;
    }
  }
  const int e_ex = ei - ew;
  int slot = __shfl_sync(0xffffffffu, gi - gw + min(need, e_ex), warp);
  int ties = __shfl_sync(0xffffffffu, e_ex, warp);
#pragma unroll 4
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const uint32_t kv = i < hi ? keys[i] : 0u;
    const unsigned below = (1u << lane) - 1u;
    const unsigned eqm = __ballot_sync(0xffffffffu, i < hi && kv == thr);
    const bool tie_taken = (eqm >> lane & 1u) && ties + __popc(eqm & below) < need;
    const bool taken = (i < hi && kv > thr) || tie_taken;
    const unsigned tm = __ballot_sync(0xffffffffu, taken);
    const int my_slot = slot + __popc(tm & below);
    if (taken && my_slot >= lo_slot && my_slot < hi_slot) out[my_slot - lo_slot] = map ? map[i] : i;
    slot += __popc(tm);
    ties += __popc(eqm);
  }
  __syncthreads();
}

// ------------------------------------------------------------------ coarse logits
//
// z[q] = zscale * Σ_c a[c] * Q[q][c] for one row a of the level-L
// approximation, computed by the C consecutive lanes that hold its channels
// (lane l of the group: channels l*V .. l*V+V-1, fp32) against every query of
// the row's unit.  Each lane forms its channels' partial dot product with all
// queries, then a reduce-scatter over the group (log2 C shuffle rounds, each
// halving the values a lane keeps) leaves lane l the totals of queries
// l*GP/C .. (l+1)*GP/C - 1.  Warp-collective: every lane of the warp calls it
// (groups are C-aligned within the warp); `active` lanes store their queries
// (those below G) to out[q].  GP >= G is a multiple of C.

template <int N, int O>
struct ReduceScatter {
  static __device__ __forceinline__ void run(float* v, int lane) {
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float send = up ? v[i] : v[i + N / 2];
      const float keep = up ? v[i + N / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
    ReduceScatter<N / 2, O / 2>::run(v, lane);
  }
};
template <int N>
struct ReduceScatter<N, 0> {
  static __device__ __forceinline__ void run(float*, int) {}
};

template <typename T, int V, int C, int GP>
__device__ __forceinline__ void emit_coarse_logits(const float* a, bool active, const T* q_unit,
                                                   int D, int G, float zscale, float* out) {
  static_assert(GP % C == 0 && (C & (C - 1)) == 0 && C <= 32, "lane group layout");
  static_assert(V == Elem<T>::kPer16B, "a lane holds one 16-byte chunk of each query row");
  const int lane = threadIdx.x & 31, g = lane & (C - 1);
  float v[GP];
#pragma unroll
  for (int q = 0; q < GP; ++q) {
    float s = 0.f;
    if (active && q < G) {
      float f[V];
      widen16(ldg16(q_unit + static_cast<int64_t>(q) * D + g * V), static_cast<const T*>(nullptr), f);
#pragma unroll
      for (int e = 0; e < V; ++e) s = fmaf(a[e], f[e], s);
    }
    v[q] = s;
  }
  ReduceScatter<GP, C / 2>::run(v, lane);
  constexpr int W = GP / C;  // queries per lane after the reduce-scatter
  if (!active) return;
  const int q0 = g * W;
  if (q0 + W <= G) {
    if constexpr (W == 4) {
      *reinterpret_cast<float4*>(out + q0) =
          make_float4(v[0] * zscale, v[1] * zscale, v[2] * zscale, v[3] * zscale);
    } else if constexpr (W == 2) {
      *reinterpret_cast<float2*>(out + q0) = make_float2(v[0] * zscale, v[1] * zscale);
    } else {
#pragma unroll
      for (int i = 0; i < W; ++i) out[q0 + i] = v[i] * zscale;
    }
  } else {
#pragma unroll
    for (int i = 0; i < W; ++i)
      if (q0 + i < G) out[q0 + i] = v[i] * zscale;
  }
}

// Exclusive prefix over the cluster of one int per CTA (pushed to every
// peer).  Returns the sum over lower ranks; *total gets the cluster sum.
// cnt_in: [kMaxCluster] ints.  Contains one cluster barrier.
__device__ inline int cluster_excl_count(int mine, int32_t* cnt_in, int* total) {
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = static_cast<int>(cluster.num_blocks());
  const int me = static_cast<int>(cluster.block_rank());
  if (threadIdx.x < cs) peer(cnt_in, threadIdx.x)[me] = mine;
  cluster.sync();
  int before = 0, all = 0;
  for (int r = 0; r < cs; ++r) {
    if (r < me) before += cnt_in[r];
    all += cnt_in[r];
  }
  *total = all;
  return before;
}

// Stable compaction of the taken entries of two parallel int arrays.
// Returns the new count.  Block-wide (contains __syncthreads()).
static __device__ __noinline__ int compact2(const int32_t* a_in, const int32_t* b_in, const uint8_t* take,
                               int n, int32_t* a_out, int32_t* b_out, int32_t* scan) {
  int carry = 0;
  for (int base = 0; base < n; base += kThreads) {
    const int i = base + threadIdx.x;
    const int t = i < n ? take[i] : 0;
    int tot;
    const int pos = block_excl_scan(t, scan, &tot);
    if (t) {
      a_out[carry + pos] = a_in[i];
      b_out[carry + pos] = b_in[i];
    }
    carry += tot;
  }
  __syncthreads();
  return carry;
}

}  // namespace wf
