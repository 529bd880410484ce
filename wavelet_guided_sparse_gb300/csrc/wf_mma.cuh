// Warp-level bf16 tensor-core helpers (m16n8k16, fp32 accumulate) and
// ldmatrix shared-memory fragment loads.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "wf_common.cuh"

namespace wf {

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
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D = A(16x16, row) * B(16x8, col) + D; bf16 inputs, fp32 accumulators.
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

// Exact split of an fp32 value into three bf16 parts, hi + mid + lo = x to
// within 2^-24 relative (each part rounds the remainder of the previous).
__device__ __forceinline__ void split3_bf16(float x, float& hi, float& mid, float& lo) {
  hi = __bfloat162float(__float2bfloat16_rn(x));
  const float r1 = x - hi;
  mid = __bfloat162float(__float2bfloat16_rn(r1));
  lo = r1 - mid;
}

// Coarse logits of 16 consecutive rows of the level-L approximation on the
// warp's tensor cores:
//   out[(span0 + r) * GZ + q] = zscale * Σ_k A[r][k] * Q[q][k]
// for rows r in [ra, rb) and queries q < G (one unit's queries, bf16).  A
// rows come as fp32 (rows r < nrows of `a`, `pitch` floats apart; shared or
// global memory); each value is split into three bf16 parts whose products
// with the bf16 queries are exact, accumulated in fp32 by m16n8k16 MMAs.
// The warp covers the query tiles nt0, nt0 + nt_step, ... (8 queries each).
// Warp-collective.
template <int D>
__device__ __forceinline__ void coarse_logits_rows16(const float* a, int pitch, int nrows, int ra,
                                                     int rb, int64_t span0,
                                                     const __nv_bfloat16* q, int G, int GZ,
                                                     float zscale, float* out, int nt0,
                                                     int nt_step) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int NT = (G + 7) >> 3;
  constexpr int kMaxTiles = 8;  // G <= 64
  float c[kMaxTiles][4];
#pragma unroll
  for (int t = 0; t < kMaxTiles; ++t)
#pragma unroll
    for (int e = 0; e < 4; ++e) c[t][e] = 0.f;
  const bool r0ok = gid < nrows, r1ok = gid + 8 < nrows;
#pragma unroll 2
  for (int ks = 0; ks < D / 16; ++ks) {
    const int k0 = ks * 16 + 2 * tig;
    float2 v[4];  // (row gid, k0), (row gid + 8, k0), (row gid, k0 + 8), (row gid + 8, k0 + 8)
    v[0] = r0ok ? *reinterpret_cast<const float2*>(a + gid * pitch + k0) : make_float2(0.f, 0.f);
    v[1] = r1ok ? *reinterpret_cast<const float2*>(a + (gid + 8) * pitch + k0) : make_float2(0.f, 0.f);
    v[2] = r0ok ? *reinterpret_cast<const float2*>(a + gid * pitch + k0 + 8) : make_float2(0.f, 0.f);
    v[3] = r1ok ? *reinterpret_cast<const float2*>(a + (gid + 8) * pitch + k0 + 8) : make_float2(0.f, 0.f);
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
      const int nt = nt0 + t * nt_step;
      if (nt >= NT) break;
      const int qn = nt * 8 + gid;
      uint32_t b[2] = {0u, 0u};
      if (qn < G) {
        const __nv_bfloat16* qr = q + static_cast<int64_t>(qn) * D + k0;
        b[0] = __ldg(reinterpret_cast<const unsigned int*>(qr));
        b[1] = __ldg(reinterpret_cast<const unsigned int*>(qr + 8));
      }
#pragma unroll
      for (int pl = 0; pl < 3; ++pl) mma_bf16(c[t], af[pl], b);
    }
  }
#pragma unroll
  for (int t = 0; t < kMaxTiles; ++t) {
    const int nt = nt0 + t * nt_step;
    if (nt >= NT) break;
    const int col = nt * 8 + 2 * tig;
    if (col >= G) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = gid + 8 * h;
      if (r < ra || r >= rb) continue;
      float* dst = out + (span0 + r) * GZ + col;
      if (col + 1 < G)
        *reinterpret_cast<float2*>(dst) = make_float2(c[t][2 * h] * zscale, c[t][2 * h + 1] * zscale);
      else
        dst[0] = c[t][2 * h] * zscale;
    }
  }
}

// Coarse logits zl[r, q] = zscale Q[unit(r)][q]·A_L[r] of the A_L rows
// [r_begin, r_end) (global, fp32; unit(r) = r / P), by `workers` of the
// block's warps (worker w = this warp's index among them).  bf16 queries: 16
// rows per warp task on the tensor cores (exact three-way split of A_L);
// fp32 queries: lane groups (C lanes per row) with FMAs.
template <typename T, int D>
__device__ __forceinline__ void coarse_logits_range(const float* al, const T* q, float* zl,
                                                    int64_t r_begin, int64_t r_end, int64_t P,
                                                    int G, int GZ, float zscale, int64_t worker,
                                                    int64_t workers) {
  if constexpr (sizeof(T) == 2) {
    for (int64_t r0 = r_begin + worker * 16; r0 < r_end; r0 += workers * 16) {
      const int n = static_cast<int>(r_end - r0 < 16 ? r_end - r0 : 16);
      for (int64_t u = r0 / P; u * P < r0 + n; ++u) {
        const int ra = static_cast<int>(u * P > r0 ? u * P - r0 : 0);
        const int rb = static_cast<int>((u + 1) * P - r0 < n ? (u + 1) * P - r0 : n);
        coarse_logits_rows16<D>(al + r0 * D, D, n, ra, rb, r0,
                                reinterpret_cast<const __nv_bfloat16*>(q) + u * G * D, G, GZ,
                                zscale, zl, 0, 1);
      }
    }
  } else {
    constexpr int V = Elem<T>::kPer16B, C = D / V, RPW = 32 / C;  // rows per warp pass
    const int lane = threadIdx.x & 31, c = lane % C;
    for (int64_t base = r_begin + worker * RPW; base < r_end; base += workers * RPW) {
      const int64_t row = base + lane / C;
      const bool act = row < r_end;
      float a[V];
#pragma unroll
      for (int v = 0; v < V; v += 4) {
        const float4 x = act ? *reinterpret_cast<const float4*>(al + row * D + c * V + v)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        a[v] = x.x; a[v + 1] = x.y; a[v + 2] = x.z; a[v + 3] = x.w;
      }
      const int64_t unit = act ? row / P : 0;
      float* dst = zl + (act ? row : 0) * GZ;
      if (G <= 32)
        emit_coarse_logits<T, V, C, 32>(a, act, q + unit * G * D, D, G, zscale, dst);
      else
        emit_coarse_logits<T, V, C, 64>(a, act, q + unit * G * D, D, G, zscale, dst);
    }
  }
}

}  // namespace wf
