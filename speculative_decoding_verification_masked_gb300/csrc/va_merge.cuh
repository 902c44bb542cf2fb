// The in-kernel split-segment merge shared by the tcgen05 attention kernels
// (cooperative launches): per-segment arrival counters in the workspace, the
// bounded wait for a segment's parts, and the exact log-sum-exp merge of a
// share of its rows (LongSpec 2.C).
#pragma once

#include <math.h>

#include "va_common.cuh"
#include "va_kernels.h"

namespace va {

// Wrapping increments (x = x >= wrap ? 0 : x + 1) of a per-segment merge
// counter: each of the np parts arrives once (release) and leaves once, so the
// counter reads >= np once all have arrived and is back at 0 after the last one
// has left -- no atomic result is waited for.
__device__ __forceinline__ void red_release_inc_gpu(unsigned *ptr, unsigned wrap) {
  asm volatile("red.release.gpu.global.inc.u32 [%0], %1;" ::"l"(ptr), "r"(wrap) : "memory");
}
__device__ __forceinline__ void red_relaxed_inc_gpu(unsigned *ptr, unsigned wrap) {
  asm volatile("red.relaxed.gpu.global.inc.u32 [%0], %1;" ::"l"(ptr), "r"(wrap) : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int *ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

// Exact log-sum-exp merge (LongSpec 2.C) of rows [r0, r1) of a split segment
// of sequence b, kv-head hkv, whose row r is packed query row row_base + r,
// from its np parts at slots slot0..slot0+np-1, by one warp of n_warps: LPR
// lanes per row, each with 128/LPR columns, the lse and output loads of up to
// MB parts in flight at once, a running maximum across batches.
template <int LPR, int MB>
__device__ __forceinline__ void merge_rows_warp(const AttnParams &p, int b, int hkv, int row_base, int slot0, int np,
                                                int r0, int r1, int warp_id, int n_warps, int lane) {
  constexpr int D = 128;
  constexpr int RPW = 32 / LPR;      // rows per warp pass
  constexpr int C4 = D / LPR / 4;    // float4 per lane and part
  const int sub = lane / LPR, li = lane % LPR;
  const int group = p.Hq / p.Hkv;
  const size_t ostride = (size_t)p.rows_pad * D;
  for (int rbase = r0 + warp_id * RPW; rbase < r1; rbase += n_warps * RPW) {
    const int row = rbase + sub;
    const bool act = row < r1;
    const int rr = act ? row : r0;
    const float *l = p.lse_part + (size_t)slot0 * p.rows_pad + rr;
    const float *o = p.o_part + ((size_t)slot0 * p.rows_pad + rr) * D + li * C4 * 4;
    float M = -INFINITY, L = 0.f;
    float4 acc[C4];
#pragma unroll
    for (int c = 0; c < C4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = 0; q0 < np; q0 += MB) {
      float ls[MB];
      float4 v[MB][C4];
#pragma unroll
      for (int j = 0; j < MB; ++j) {
        const bool in = q0 + j < np;
        ls[j] = in ? __ldcg(l + (size_t)(q0 + j) * p.rows_pad) : -INFINITY;  // written by other CTAs: L2
#pragma unroll
        for (int c = 0; c < C4; ++c)
          v[j][c] = in ? __ldcg(reinterpret_cast<const float4 *>(o + (size_t)(q0 + j) * ostride) + c)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float m = M;
#pragma unroll
      for (int j = 0; j < MB; ++j) m = fmaxf(m, ls[j]);
      if (m == -INFINITY) continue;  // no part so far saw a key
      const float a = M == -INFINITY ? 0.f : __expf(M - m);
      L *= a;
#pragma unroll
      for (int c = 0; c < C4; ++c) {
        acc[c].x *= a;
        acc[c].y *= a;
        acc[c].z *= a;
        acc[c].w *= a;
      }
#pragma unroll
      for (int j = 0; j < MB; ++j) {
        const float w = ls[j] == -INFINITY ? 0.f : __expf(ls[j] - m);
        L += w;
#pragma unroll
        for (int c = 0; c < C4; ++c) {
          acc[c].x = fmaf(w, v[j][c].x, acc[c].x);
          acc[c].y = fmaf(w, v[j][c].y, acc[c].y);
          acc[c].z = fmaf(w, v[j][c].z, acc[c].z);
          acc[c].w = fmaf(w, v[j][c].w, acc[c].w);
        }
      }
      M = m;
    }
    if (!act) continue;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int t = (row_base + row) / group, hq = hkv * group + (row_base + row) % group;
    uint2 *dst = reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.out) +
                                           (((size_t)b * p.T + t) * p.Hq + hq) * D + li * C4 * 4);
#pragma unroll
    for (int c = 0; c < C4; ++c)
      dst[c] = make_uint2(pack_bf16(acc[c].x * inv, acc[c].y * inv), pack_bf16(acc[c].z * inv, acc[c].w * inv));
    if (li == 0) p.lse[((size_t)b * p.Hq + hq) * p.T + t] = L > 0.f ? M + __logf(L) : -INFINITY;
  }
}

// Thread 0 of a CTA: wait (bounded) until all np parts of split segment s have
// announced themselves.  False (and VA_ERR_TIMEOUT recorded) when the limit
// ran out; the caller then skips the merge.
__device__ __forceinline__ bool wait_parts_arrived(const AttnParams &p, int s, int np) {
  if (ld_acquire_gpu(&p.merge_cnt[s].x) >= np) return true;
  const uint64_t t0w = globaltimer_ns();
  while (ld_acquire_gpu(&p.merge_cnt[s].x) < np) {
    if (globaltimer_ns() - t0w > p.wait_ns) {
      record_status(p.status, VA_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

}  // namespace va
