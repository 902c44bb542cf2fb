// Verification attention on the 5th-generation tensor cores for segments of
// more than 128 packed query rows with K/V tiles that arrive by TMA -- the
// long-context token-tree workload (a 64-node tree with GQA group 4 gives 256
// rows per kv-head over a 131072-token prefix).  LongSpec 2.C: the unmasked
// prefix and the masked draft block are one stream of key tiles (the draft
// block is the last tile(s) of a segment, the only place the bitmask is
// applied), and the parts of a segment cut over several CTAs are merged
// exactly by their log-sum-exp, here inside the kernel.
//
// Two 128-row M-tiles share every 128-key tile read from HBM:
//   S_i  (128 rows x 128 keys) = Q_i K^T     A = Q_i (smem, K-major), B = K tile (K-major)
//   O_i  (128 rows x 128 d)   += P_i V       A = P_i (TMEM, over S_i), B = V tile (MN-major)
// TMEM (512 columns): O_0 at 0, O_1 at 128, S_0/P_0 at 256, S_1/P_1 at 384.
// P_i is written over S_i (per half of 64 keys, bf16 hi in the half's first 32
// columns and the bf16 residual, when needed, in its next 32), so S_i(t+1) may
// only be issued once PV_i(t) has completed.  A single MMA warp issues, per tile t,
//     PV_0(t), S_0(t+1), PV_1(t), S_1(t+1)
// so while one warpgroup runs the softmax of its M-tile the tensor core works
// on the other's PV and next S: the two softmax warpgroups alternate without
// any barrier between them.  128-key tiles halve the S MMAs and the re-reads
// of Q from shared memory against 64-key tiles.
//
// K and V tiles live in separate two-slot rings: a K slot is released as soon
// as both S MMAs of its tile have read it, early in the tile, so the next K
// tile's load starts one tile ahead and each V tile has two tiles' time to
// land -- about three tiles of loads in flight from 128 KB of ring.
//
// Roles (10 warps, one CTA per SM, cooperative launch):
//   warps 0-3 / 4-7  softmax warpgroup of M-tile 0 / 1: thread = one query row
//                    = one TMEM lane.  Online softmax in log2 units against a
//                    reference maximum that moves only when a score passes it
//                    by more than 2^8 (exact either way); P's bf16 residual is
//                    added where a key of the tile may carry more than 1/16 of
//                    the row's weight so far (a per-tile warpgroup vote; draft
//                    tiles always), so no weight loses more than 2^-8 of itself
//                    where it matters.  Then the epilogue and the merge.
//   warp 8           producer: TMA boxes of K and V (dense: 64 tokens a box;
//                    paged: one box per page) into the two rings
//   warp 9           MMA issuer and TMEM owner
// Every wait is bounded; on timeout the CTA records VA_ERR_TIMEOUT, keeps the
// barrier sequence of all roles, drains and frees TMEM.
#include <cuda.h>
#include <math.h>

#include "va_common.cuh"
#include "va_kernels.h"
#include "va_merge.cuh"
#include "va_pipeline.cuh"
#include "va_rope_fused.cuh"
#include "va_tcgen05.cuh"

namespace va {

constexpr int kTpKeys = 128;  // keys per tile
constexpr int kTpSlots = 2;   // slots of the K ring and of the V ring

struct TpSmem {
  using Geo = StageGeom<__nv_bfloat16, 128, kTpKeys>;  // one K (or V) tile: 2 columns x 128 keys x 128 B
  static constexpr int kQBytes = 2 * 32768;            // 2 M-tiles x [2 columns][128 rows][128 B]
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + kTpSlots * Geo::kTileBytes;
  static constexpr int kBarOff = kVOff + kTpSlots * Geo::kTileBytes;
  // barriers: kfull[2], kempty[2], vfull[2], vempty[2], s_full[2], p_full[2], o_done[2], drain
  static constexpr int kNumBars = 4 * kTpSlots + 3 * 2 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag, merge flag
  static constexpr int kLoFlagOff = kMiscOff + 16;          // int [2]: P residual written, per M-tile
  // then the rotary table of the segment (rope_table_bytes, 0 without
  // positions) and the tile starts of the work plan
  static constexpr int kRopeOff = kLoFlagOff + 16;
  static constexpr int kThreads = 10 * 32;
  static_assert(kKOff % 1024 == 0 && kVOff % 1024 == 0 && Geo::kTileBytes % 1024 == 0, "swizzle atoms");
};

// Offset of chunk c (16 B) of row r in a 128-row, 128B-swizzled pair of columns.
__device__ __forceinline__ uint32_t tp_swz(int r, int c) {
  return (uint32_t)((c >> 3) * (128 * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Producer warp: the K and V boxes of every tile of this CTA, each ring slot
// refilled once the MMAs that read it have completed.
__device__ __forceinline__ void tp_produce(const AttnParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                           const int *tstart, const CtaRange &cr, uint8_t *sK, uint8_t *sV,
                                           uint64_t *kfull, uint64_t *kempty, uint64_t *vfull, uint64_t *vempty,
                                           volatile int *abort_flag) {
  constexpr int TK = kTpKeys;
  constexpr int kTile = TpSmem::Geo::kTileBytes;
  const int lane = threadIdx.x & 31;
  const uint64_t policy = l2_evict_first_policy();
  if (lane == 0) {
    prefetch_tmap(tmk);
    prefetch_tmap(tmv);
  }
  bool ok = true;
  auto wait_slot = [&](uint64_t *bar, uint32_t parity) { role_wait(bar, parity, ok, abort_flag, p.wait_ns, p.status); };
  int it = 0;
  for (int s = cr.s0; s < p.S && tstart[s] < cr.t1; ++s) {
    const Seg g = seg_info(p, s, false);
    const int lt0 = max(tstart[s], cr.t0) - tstart[s];
    const int lt1 = min(tstart[s + 1], cr.t1) - tstart[s];
    for (int lt = lt0; lt < lt1; ++lt, ++it) {
      const int sl = it % kTpSlots;
      const uint32_t ph = (uint32_t)(it / kTpSlots) & 1u;
      const int k0 = lt * TK;
      // boxes of BR rows: dense BR = 64 consecutive tokens (rows past the
      // segment end arrive too and are masked); paged one box per page, boxes
      // starting past the segment end not loaded
      const int BR = p.tma_box;
      const bool paged = p.layout == VA_LAYOUT_PAGED;
      const int nb = paged ? min(TK / BR, (g.nkeys - k0 + BR - 1) / BR) : TK / BR;
      int row = 0;
      if (lane < nb) {
        const int slot = k0 + lane * BR;
        if (paged) {
          int page = __ldg(p.page_table + (size_t)g.b * p.max_pages + (slot >> p.page_shift));
          if (page < 0 || page >= p.num_pages) {
            record_status(p.status, VA_ERR_DEVICE_BOUNDS);
            page = 0;
          }
          row = (page << p.page_shift) + (slot & ((1 << p.page_shift) - 1));
        } else {
          row = g.b * p.len_cap + slot;
        }
      }
      const uint32_t bytes = (uint32_t)(nb * BR * 128 * 2);
      const int off = lane * BR * 128;
      wait_slot(kempty + sl, ph ^ 1u);
      if (ok) {
        if (lane == 0) mbar_arrive_expect_tx(kfull + sl, bytes);
        __syncwarp();
        if (lane < nb) {
          uint8_t *dst = sK + sl * kTile + off;
          tma_load_3d(dst, tmk, 0, g.hkv, row, kfull + sl, policy);
          tma_load_3d(dst + TK * 128, tmk, 64, g.hkv, row, kfull + sl, policy);
        }
      }
      wait_slot(vempty + sl, ph ^ 1u);
      if (ok) {
        if (lane == 0) mbar_arrive_expect_tx(vfull + sl, bytes);
        __syncwarp();
        if (lane < nb) {
          uint8_t *dst = sV + sl * kTile + off;
          tma_load_3d(dst, tmv, 0, g.hkv, row, vfull + sl, policy);
          tma_load_3d(dst + TK * 128, tmv, 64, g.hkv, row, vfull + sl, policy);
        }
      }
    }
  }
  if (!ok) {
    // drain the boxes this warp issued before leaving (bounded)
    for (int j = max(0, it - kTpSlots); j < it; ++j) {
      mbar_wait(kfull + (j % kTpSlots), (uint32_t)(j / kTpSlots) & 1u, p.wait_ns >> 4);
      mbar_wait(vfull + (j % kTpSlots), (uint32_t)(j / kTpSlots) & 1u, p.wait_ns >> 4);
    }
  }
}

template <bool kRope>
__global__ void __launch_bounds__(TpSmem::kThreads, 1)
    verify_attn_tcp_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                           const __grid_constant__ CUtensorMap tmv) {
  using SM = TpSmem;
  using Geo = SM::Geo;
  constexpr int D = 128;
  constexpr int TK = kTpKeys;
  constexpr int NSL = kTpSlots;
  constexpr int kSoft = 256;
  constexpr int kProducerWarp = 8, kMmaWarp = 9;
  constexpr int kBarQ = 1, kBarSoft = 2, kBarEnd = 3, kBarVote = 4;  // kBarVote + M-tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *sQ = smem;
  uint8_t *sK = smem + SM::kKOff;
  uint8_t *sV = smem + SM::kVOff;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kBarOff);
  uint64_t *kfull = bars, *kempty = bars + NSL, *vfull = bars + 2 * NSL, *vempty = bars + 3 * NSL;
  uint64_t *s_full = bars + 4 * NSL;      // [M-tile]
  uint64_t *p_full = bars + 4 * NSL + 2;  // [M-tile]
  uint64_t *o_done = bars + 4 * NSL + 4;  // [M-tile]
  uint64_t *drain = bars + 4 * NSL + 6;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SM::kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM::kMiscOff + 4);
  volatile int *merge_ok = abort_flag + 1;
  volatile int *lo_flag = reinterpret_cast<volatile int *>(smem + SM::kLoFlagOff);
  float2 *rope_tab = reinterpret_cast<float2 *>(smem + SM::kRopeOff);
  int *tstart = reinterpret_cast<int *>(smem + SM::kRopeOff + (kRope ? rope_table_bytes(p) : 0));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = blockIdx.x;

  if (tid == 0) {
    for (int i = 0; i < NSL; ++i) {
      mbar_init(kfull + i, 1);
      mbar_init(kempty + i, 1);
      mbar_init(vfull + i, 1);
      mbar_init(vempty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 128);
      mbar_init(o_done + i, 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  const CtaRange cr = plan_cta<TK>(p, tstart);  // contains __syncthreads
  if (c >= cr.G) return;
  const int t0 = cr.t0, t1 = cr.t1, s0 = cr.s0;

  if (warp == kProducerWarp) {
    tp_produce(p, &tmk, &tmv, tstart, cr, sK, sV, kfull, kempty, vfull, vempty, abort_flag);
    return;
  }

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  named_bar_sync(kBarEnd, kSoft + 32);
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const float cl2 = p.scale * kLog2e;
  const int group = p.Hq / p.Hkv;

  bool ok = true;
  auto wait_ok = [&](uint64_t *bar, uint32_t parity) { role_wait(bar, parity, ok, abort_flag, p.wait_ns, p.status); };

  if (warp == kMmaWarp) {
    // ================================ MMA issuer ================================
    const uint32_t id_s = umma_idesc(128, 128, 0, 0);  // S = Q K^T, both K-major
    const uint32_t id_o = umma_idesc(128, 128, 0, 1);  // O += P V, V MN-major
    // descriptors built once; a K-step, M-tile or slot offset is an add to the
    // start-address field (addresses stay below 256 KB: the field never carries)
    const uint64_t dQ0 = umma_sdesc(smem_u32(sQ), 16, 1024);
    const uint64_t dK0 = umma_sdesc(smem_u32(sK), 16, 1024);
    const uint64_t dV0 = umma_sdesc(smem_u32(sV), TK * 128, 1024);
    constexpr uint64_t kSlotStep = (uint64_t)(Geo::kTileBytes >> 4);
    // the draft keys of tile lt of segment g, rotated in place before any S MMA reads them
    auto rotate_draft = [&](int sl, const Seg &g, int lt) {
      if (kRope && ok && lt * TK + TK > g.n_prefix) {
        const int r0 = max(0, g.n_prefix - lt * TK), r1 = min(TK, g.nkeys - lt * TK);
        rope_rotate_tile_rows<__nv_bfloat16, D, TK>(sK + sl * Geo::kTileBytes, r0, r1, lt * TK + r0 - g.n_prefix,
                                                    rope_tab, lane, 32);
        fence_proxy_async_smem();
      }
      __syncwarp();
    };
    auto issue_s = [&](int i, int sl) {  // S_i = Q_i K^T into TMEM 256 + 128 i
      if (!ok || lane != 0) return;
      tc_fence_after();
      const uint64_t dQ = dQ0 + (uint64_t)(i * (32768 >> 4));
      const uint64_t dK = dK0 + (uint64_t)sl * kSlotStep;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t off = (uint64_t)(((ks >> 2) * (TK * 128) + (ks & 3) * 32) >> 4);  // Q and K: same layout
        umma_ss(tmem + 256 + 128 * i, dQ + off, dK + off, id_s, ks > 0 ? 1u : 0u);
      }
      umma_commit(s_full + i);
    };
    auto issue_pv = [&](int i, int sl, bool first, bool lo) {  // O_i += P_i V (+ residual P_i V)
      if (!ok || lane != 0) return;
      tc_fence_after();
      const uint64_t dV = dV0 + (uint64_t)sl * kSlotStep;
      const uint32_t aP = tmem + 256 + 128 * i;
      // keys 16 kk .. 16 kk + 15: bf16 P at column 64 (kk / 4) + 8 (kk % 4) of
      // S_i, the residual 32 columns further
#pragma unroll
      for (int kk = 0; kk < TK / 16; ++kk) {
        const uint64_t bb = dV + (uint64_t)((kk * 2048) >> 4);
        umma_ts(tmem + 128 * i, aP + 64 * (kk >> 2) + 8 * (kk & 3), bb, id_o, (!first || kk > 0) ? 1u : 0u);
      }
      if (lo) {
#pragma unroll
        for (int kk = 0; kk < TK / 16; ++kk)
          umma_ts(tmem + 128 * i, aP + 64 * (kk >> 2) + 32 + 8 * (kk & 3), dV + (uint64_t)((kk * 2048) >> 4), id_o,
                  1u);
      }
      umma_commit(o_done + i);
    };
    auto commit = [&](uint64_t *bar) {
      if (ok && lane == 0) umma_commit(bar);
    };

    int it = 0, jt = 0;
    for (int s = s0; s < p.S && tstart[s] < t1; ++s) {
      const Seg g = seg_info(p, s, false);
      const int lt0 = max(tstart[s], t0) - tstart[s];
      const int lt1 = min(tstart[s + 1], t1) - tstart[s];
      named_bar_sync(kBarQ, kSoft + 32);  // Q of this segment is in shared memory
      wait_ok(kfull + it % NSL, (uint32_t)(it / NSL) & 1u);
      rotate_draft(it % NSL, g, lt0);
      issue_s(0, it % NSL);
      issue_s(1, it % NSL);
      commit(kempty + it % NSL);  // the K slot is free once both S MMAs have read it
      for (int lt = lt0; lt < lt1; ++lt, ++it, ++jt) {
        const int sl = it % NSL;
        const uint32_t jph = (uint32_t)jt & 1u;
        const bool more = lt + 1 < lt1;
        for (int i = 0; i < 2; ++i) {
          wait_ok(p_full + i, jph);
          // the softmax wrote the P residual of this tile too (set before its
          // arrive on p_full; rewritten only after this PV has completed)
          const bool lo = lo_flag[i] != 0;
          if (i == 0) {
            wait_ok(vfull + sl, (uint32_t)(it / NSL) & 1u);
            if (ok && lt * TK + TK > g.nkeys) {
              // rows past the segment end: whatever the boxes brought (or an
              // unfilled slot) must not meet P = 0 as NaN; zero those V rows
              uint8_t *vt = sV + sl * Geo::kTileBytes;
              for (int e = lane; e < TK * 16; e += 32) {
                const int r = e >> 4;
                if (lt * TK + r >= g.nkeys) *reinterpret_cast<uint4 *>(vt + tp_swz(r, e & 15)) = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
            }
            __syncwarp();
          }
          issue_pv(i, sl, lt == lt0, lo);
          if (i == 1) commit(vempty + sl);
          if (more) {
            wait_ok(o_done + i, jph);  // PV_i(t) has read P_i: S_i(t+1) may overwrite it
            if (i == 0) {
              wait_ok(kfull + (it + 1) % NSL, (uint32_t)((it + 1) / NSL) & 1u);
              rotate_draft((it + 1) % NSL, g, lt + 1);
            }
            issue_s(i, (it + 1) % NSL);
            if (i == 1) commit(kempty + (it + 1) % NSL);
          }
        }
        __syncwarp();
      }
    }
    // drain: every MMA issued has finished before TMEM is released
    if (lane == 0) umma_commit(drain);
    mbar_wait(drain, 0u, p.wait_ns);
    tc_fence_before();
    named_bar_sync(kBarEnd, kSoft + 32);
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    return;
  }

  // ============================ softmax warpgroups ============================
  const int mi = warp >> 2;              // M-tile of this warpgroup
  const int r = (warp & 3) * 32 + lane;  // row in the M-tile = TMEM lane
  const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t tO = tmem + lane_bits + 128 * mi;
  const uint32_t tS = tmem + lane_bits + 256 + 128 * mi;
  int jt = 0;
  int rope_b = -1;  // sequence whose rotary table is in shared memory
  // split segments this CTA holds a part of (at most its first and its last)
  int n_split = 0, ms[2] = {0, 0}, mslot[2] = {0, 0}, mnp[2] = {0, 0}, mpart[2] = {0, 0};
  for (int s = s0; s < p.S && tstart[s] < t1; ++s) {
    const Seg g = seg_info(p, s, false);
    const int lt0 = max(tstart[s], t0) - tstart[s];
    const int lt1 = min(tstart[s + 1], t1) - tstart[s];
    const int first_cta = owner_cta(tstart[s], cr.total, cr.G);
    const int n_parts = owner_cta(tstart[s + 1] - 1, cr.total, cr.G) - first_cta + 1;
    if (lt0 == 0 && tid == 0) p.meta[s] = make_int2(s + first_cta, n_parts);

    // ---- Q of this segment into shared memory (both warpgroups; every S MMA
    // of the previous segment has completed once both have passed here) ----
    named_bar_sync(kBarSoft, kSoft);
    if constexpr (kRope) {
      // rotary table of this sequence's draft tokens (kept while the CTA stays
      // on the sequence), then q rotated on its way in
      if (g.b != rope_b) {
        rope_build_table(p, g.b, rope_tab, tid, kSoft);
        named_bar_sync(kBarSoft, kSoft);
        rope_b = g.b;
      }
      const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q);
      for (int e = tid; e < 2 * 128 * 8; e += kSoft) {
        const int m = e >> 10;
        const int row = (e >> 3) & 127;
        const int ch = e & 7;
        const int rr = g.rb * p.rows_pad + m * 128 + row;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        if (rr < p.R) {
          const int t = rr / group;
          const int hq = g.hkv * group + rr % group;
          const uint4 *src = reinterpret_cast<const uint4 *>(qb + (((size_t)g.b * p.T + t) * p.Hq + hq) * D);
          lo = __ldg(src + ch);
          hi = __ldg(src + ch + 8);
          rope_rotate8_bf16(lo, hi, rope_tab + t * (D / 2) + ch * 8);
        }
        *reinterpret_cast<uint4 *>(sQ + m * 32768 + tp_swz(row, ch)) = lo;
        *reinterpret_cast<uint4 *>(sQ + m * 32768 + tp_swz(row, ch + 8)) = hi;
      }
      fence_proxy_async_smem();
    } else {
      const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q);
      for (int e = tid; e < 2 * 128 * 16; e += kSoft) {
        const int m = e >> 11;
        const int row = (e >> 4) & 127;
        const int ch = e & 15;
        const int rr = g.rb * p.rows_pad + m * 128 + row;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (rr < p.R) {
          const int t = rr / group;
          const int hq = g.hkv * group + rr % group;
          v = __ldg(reinterpret_cast<const uint4 *>(qb + (((size_t)g.b * p.T + t) * p.Hq + hq) * D) + ch);
        }
        *reinterpret_cast<uint4 *>(sQ + m * 32768 + tp_swz(row, ch)) = v;
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    named_bar_arrive(kBarQ, kSoft + 32);

    const int rr = g.rb * p.rows_pad + mi * 128 + r;
    const bool rvalid = rr < p.R;
    const int t = rvalid ? rr / group : 0;
    const int hq = g.hkv * group + (rvalid ? rr % group : 0);
    uint64_t rmask = 0;  // the draft keys this row sees
    if (lt1 * TK > g.n_prefix) {
      uint64_t tl = 0, th = 0;
      if (p.parent != nullptr) warp_tree_rows(p, g.b, tl, th);
      rmask = draft_row(p, g.b, t, tl, th);
    }
    float m_used = -INFINITY;  // reference maximum of the exponentials (raw score units)
    float l = 0.f;

    for (int lt = lt0; lt < lt1; ++lt, ++jt) {
      wait_ok(s_full + mi, (uint32_t)jt & 1u);
      tc_fence_after();
      const int k0 = lt * TK;
      const bool masked = k0 + TK > g.n_prefix;
      // key k0 + j is visible to this row (only draft tiles carry a mask)
      auto visible = [&](int j) {
        const int key = k0 + j;
        bool vis = key < g.nkeys;
        if (vis && key >= g.n_prefix) vis = (rmask >> (key - g.n_prefix)) & 1ull;
        return vis;
      };
      // pass 1: the row's maximum over the tile (all 128 columns in flight at
      // once; the scores are read again chunk by chunk for the exponentials,
      // which keeps the softmax within the registers 10 warps leave a thread)
      float mx;
      {
        uint32_t u[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tS + 32 * q, u[q]);
        tmem_ld_wait();
        if (masked) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (!visible(32 * q + j)) u[q][j] = __float_as_uint(-INFINITY);
        }
        float m8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t *v = &u[q >> 1][(q & 1) * 16];
          float a = fmaxf(fmaxf(__uint_as_float(v[0]), __uint_as_float(v[1])),
                          fmaxf(__uint_as_float(v[2]), __uint_as_float(v[3])));
          float b = fmaxf(fmaxf(__uint_as_float(v[4]), __uint_as_float(v[5])),
                          fmaxf(__uint_as_float(v[6]), __uint_as_float(v[7])));
          float c2 = fmaxf(fmaxf(__uint_as_float(v[8]), __uint_as_float(v[9])),
                           fmaxf(__uint_as_float(v[10]), __uint_as_float(v[11])));
          float d = fmaxf(fmaxf(__uint_as_float(v[12]), __uint_as_float(v[13])),
                          fmaxf(__uint_as_float(v[14]), __uint_as_float(v[15])));
          m8[q] = fmaxf(fmaxf(a, b), fmaxf(c2, d));
        }
        mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      }
      const float m_new = fmaxf(m_used, mx);
      // move the reference only when it grew by more than 2^8 (exact either
      // way); O, which holds every PV up to tile t-1 (S_i(t) was issued only
      // after PV_i(t-1) completed), is rescaled once P is written
      bool rescale = false;
      float alpha = 1.f;
      if (lt == lt0) {
        m_used = m_new;
      } else {
        const bool need = (m_new - m_used) * cl2 > 8.f;
        rescale = __any_sync(0xffffffffu, need);
        if (need) {
          alpha = exp2f((m_used - m_new) * cl2);
          l *= alpha;
          m_used = m_new;
        }
      }
      const float mu = (m_used == -INFINITY) ? 0.f : m_used * cl2;
      // P's residual is needed where the tile's largest weight may exceed 1/16
      // of the row's weight up to and including it: 2^(mx - mu) > (l + 2^(mx - mu)) / 16
      bool lo = masked;
      if (!masked) lo = bar_red_or(kBarVote + mi, 128, ex2_approx(fmaf(mx, cl2, -mu)) * 15.f > l);
      if (r == 0) lo_flag[mi] = lo ? 1 : 0;
      // pass 2: P = 2^(s cl2 - mu) for each half of 64 keys, written over the
      // half's own 64 S columns once both of its chunks are in registers: the
      // bf16 pairs of keys 64h + 32c .. at column 64h + 16c, their residual 32
      // columns further (so no score is overwritten before it is read)
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums: short add chains
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t u[2][32];
        tmem_ld32(tS + 64 * h, u[0]);
        tmem_ld32(tS + 64 * h + 32, u[1]);
        tmem_ld_wait();
#pragma unroll
        for (int cq = 0; cq < 2; ++cq) {
          if (masked) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (!visible(64 * h + 32 * cq + j)) u[cq][j] = __float_as_uint(-INFINITY);
          }
          uint32_t ph[16];
          if (lo) {
            uint32_t pl[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float a = ex2_approx(fmaf(__uint_as_float(u[cq][2 * j]), cl2, -mu));
              const float bq = ex2_approx(fmaf(__uint_as_float(u[cq][2 * j + 1]), cl2, -mu));
              ls4[j & 3] += a + bq;
              split_bf16x2(a, bq, ph[j], pl[j]);
            }
            tmem_st16(tS + 64 * h + 16 * cq, ph);
            tmem_st16(tS + 64 * h + 32 + 16 * cq, pl);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float a = ex2_approx(fmaf(__uint_as_float(u[cq][2 * j]), cl2, -mu));
              const float bq = ex2_approx(fmaf(__uint_as_float(u[cq][2 * j + 1]), cl2, -mu));
              ls4[j & 3] += a + bq;
              ph[j] = pack_bf16(a, bq);
            }
            tmem_st16(tS + 64 * h + 16 * cq, ph);
          }
        }
      }
      l += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
      if (rescale) {
#pragma unroll
        for (int cch = 0; cch < 4; ++cch) {
          uint32_t u[32];
          tmem_ld32(tO + 32 * cch, u);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(__uint_as_float(u[j]) * alpha);
          tmem_st32(tO + 32 * cch, u);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full + mi);
    }

    // ---- epilogue: O / l of this row for this segment part ----
    wait_ok(o_done + mi, (uint32_t)(jt - 1) & 1u);
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_nat = l > 0.f ? (m_used * cl2 + log2f(l)) * kLn2 : -INFINITY;
    const bool write = rvalid && ok;
    const size_t slot = (size_t)(s + c);
#pragma unroll
    for (int cch = 0; cch < 4; ++cch) {
      uint32_t u[32];
      tmem_ld32(tO + 32 * cch, u);
      tmem_ld_wait();
      if (!write) continue;
      if (n_parts == 1) {
        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.out) + (((size_t)g.b * p.T + t) * p.Hq + hq) * D + 32 * cch;
        if (p.out_align16) {
          uint4 *ob = reinterpret_cast<uint4 *>(orow);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            ob[q4] = make_uint4(pack_bf16(__uint_as_float(u[8 * q4 + 0]) * inv, __uint_as_float(u[8 * q4 + 1]) * inv),
                                pack_bf16(__uint_as_float(u[8 * q4 + 2]) * inv, __uint_as_float(u[8 * q4 + 3]) * inv),
                                pack_bf16(__uint_as_float(u[8 * q4 + 4]) * inv, __uint_as_float(u[8 * q4 + 5]) * inv),
                                pack_bf16(__uint_as_float(u[8 * q4 + 6]) * inv, __uint_as_float(u[8 * q4 + 7]) * inv));
        } else {
          uint2 *ob = reinterpret_cast<uint2 *>(orow);
#pragma unroll
          for (int q2 = 0; q2 < 8; ++q2)
            ob[q2] = make_uint2(pack_bf16(__uint_as_float(u[4 * q2 + 0]) * inv, __uint_as_float(u[4 * q2 + 1]) * inv),
                                pack_bf16(__uint_as_float(u[4 * q2 + 2]) * inv, __uint_as_float(u[4 * q2 + 3]) * inv));
        }
      } else {
        float4 *op = reinterpret_cast<float4 *>(p.o_part + (slot * p.rows_pad + mi * 128 + r) * D + 32 * cch);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          op[q4] = make_float4(__uint_as_float(u[4 * q4]) * inv, __uint_as_float(u[4 * q4 + 1]) * inv,
                               __uint_as_float(u[4 * q4 + 2]) * inv, __uint_as_float(u[4 * q4 + 3]) * inv);
      }
    }
    if (write) {
      if (n_parts == 1)
        p.lse[((size_t)g.b * p.Hq + hq) * p.T + t] = lse_nat;
      else
        p.lse_part[slot * p.rows_pad + mi * 128 + r] = lse_nat;
    }
    if (n_parts > 1) {
      // publish the part (always, also after a failed wait, so the counters
      // return to zero): the barrier orders both warpgroups' row and lse
      // stores before thread 0's release increment, which is cumulative
      named_bar_sync(kBarSoft, kSoft);
      if (tid == 0 && c != p.test_drop_part)
        red_release_inc_gpu(reinterpret_cast<unsigned *>(&p.merge_cnt[s].x), 2u * n_parts - 1u);
      if (n_split < 2) {
        ms[n_split] = s;
        mslot[n_split] = s + first_cta;
        mnp[n_split] = n_parts;
        mpart[n_split] = c - first_cta;
        ++n_split;
      }
    }
  }

  // ---- merge of the split segments: once every part of a segment has
  // arrived, each of its CTAs merges an equal share of its rows ----
  for (int k = 0; k < n_split; ++k) {
    const int s = ms[k], np = mnp[k];
    if (tid == 0) *merge_ok = wait_parts_arrived(p, s, np) ? 1 : 0;
    named_bar_sync(kBarSoft, kSoft);  // thread 0's acquire, then the barrier, orders the reads below
    if (*merge_ok) {
      const int rb = s % p.NRB, hkv = (s / p.NRB) % p.Hkv, b = s / (p.NRB * p.Hkv);
      const int nrows = min(p.rows_pad, p.R - rb * p.rows_pad);
      const int r0 = mpart[k] * nrows / np, r1 = (mpart[k] + 1) * nrows / np;
      if (np <= 4)
        merge_rows_warp<8, 4>(p, b, hkv, rb * p.rows_pad, mslot[k], np, r0, r1, warp, 8, lane);
      else
        merge_rows_warp<32, 24>(p, b, hkv, rb * p.rows_pad, mslot[k], np, r0, r1, warp, 8, lane);
    }
    named_bar_sync(kBarSoft, kSoft);
    // leave: np arrivals and np departures wrap the counter back to zero
    if (tid == 0) red_relaxed_inc_gpu(reinterpret_cast<unsigned *>(&p.merge_cnt[s].x), 2u * np - 1u);
  }
  tc_fence_before();
  named_bar_sync(kBarEnd, kSoft + 32);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
size_t attn_tcp_smem_required(const AttnParams &p) {
  return 1024 + (size_t)TpSmem::kRopeOff + (size_t)rope_table_bytes(p) + (size_t)(p.S + 1) * 4;
}

cudaError_t launch_attention_tcp(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                                 cudaStream_t stream) {
  const size_t smem = attn_tcp_smem_required(p);
  auto kern = p.positions != nullptr ? verify_attn_tcp_kernel<true> : verify_attn_tcp_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // cooperative: every CTA is resident, so the wait for a segment's parts ends
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(TpSmem::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tmk, tmv);
}

}  // namespace va
