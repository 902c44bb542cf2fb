// Verification attention on the 5th-generation tensor cores (tcgen05 + TMEM),
// for the case where the packed query rows of one kv-head (GQA group x T draft
// tokens) exceed 64 -- e.g. a 64-node token tree with group 4 gives 256 rows.
// Same method and work plan as verify_attn_kernel (LongSpec 2.C: unmasked
// prefix, masked draft block, exact log-sum-exp merge; stream-K over
// 64-key tiles), but every K/V tile read from HBM now feeds up to 256 query
// rows through UMMA instead of warp-level mma.sync.
//
// Roles (12 warps when the segment has two 128-row M-tiles; one CTA per SM,
// cooperative launch):
//   warps 0-3 / 4-7  softmax warpgroup of M-tile 0 / 1: thread = one query row
//                    = one TMEM lane.  Reads S from TMEM, applies the draft
//                    bitmask, runs the online softmax, writes P (bf16) back
//                    over S, rescales O in TMEM when the row max grows by more
//                    than 2^8, and writes the output row.
//                    A bf16 P keeps each weight only to 2^-8 of itself, which
//                    shows in the output when a few keys carry the weight of a
//                    row (attention sinks).  So the warpgroup votes per tile:
//                    if the largest weight of the tile may be more than 1/16
//                    of some row's weight so far, P's bf16 residual is written
//                    too and its PV issuer multiplies it as well (draft tiles
//                    always).  A key left to the bf16 P then carries at most
//                    1/16 of its row's final weight, and on spread-out rows
//                    only a part's first tiles take the extra MMAs.
//   warp 4*NMT       producer: TMA boxes (dense) / cp.async gathers (paged,
//                    sparse) into a 4-stage ring (3 when shared memory is short)
//   warps 4*NMT+1+i  PV issuer of M-tile i: O_i += P_i V (A = P from TMEM, B =
//                    V as an MN-major operand).  Issuer 0 owns the TMEM
//                    allocation.
//   warp 5*NMT+1     S issuer of every M-tile: S_i = Q_i K^T (M128 N64 K128,
//                    both operands in shared memory, K-major 128B swizzle)
//                    into one of two S/P buffers per M-tile.  S of tile t goes
//                    into the buffer of tile t-2 once PV(t-2), which reads P
//                    from it, has completed (MMAs with different accumulators
//                    are not ordered against each other); with S and PV on
//                    separate warps neither waits behind the other's issue.
// TMEM (512 columns): O_i at 128*i, S/P buffers at 256 + 64*(2*i + b).
// A segment cut over several CTAs leaves one normalised part per CTA; after
// its last tile every CTA of the segment waits (bounded) for all parts and
// merges an equal share of the rows by their log-sum-exp.
// Every wait is bounded; on timeout the CTA records VA_ERR_TIMEOUT, keeps the
// barrier sequence of all roles intact, drains and frees TMEM.
#include <cuda.h>
#include <math.h>

#include "va_common.cuh"
#include "va_kernels.h"
#include "va_merge.cuh"
#include "va_pipeline.cuh"
#include "va_rope_fused.cuh"
#include "va_tcgen05.cuh"

namespace va {

// Stages of the K/V ring: 4 (measured on the tree workload: 3 stages 130.4 us,
// 4 stages 125.5 us, 5 stages 128.6 us), or 3 when the plan's tile starts and
// the rotary table leave no room for the fourth.
constexpr int kTcStagesMin = 3;
constexpr int kTcStagesMax = 4;

// ---------------------------------------------------------------------------
// shared memory plan
// ---------------------------------------------------------------------------
template <int NMT, int NS>
struct TcSmem {
  static constexpr int kQBytes = NMT * 2 * 128 * 128;  // NMT M-tiles x 2 columns x 128 rows x 128 B
  static constexpr int kStageBytes = StageGeom<__nv_bfloat16, 128>::kStageBytes;
  static constexpr int kStagesOff = kQBytes;
  static constexpr int kBarOff = kStagesOff + NS * kStageBytes;
  // barriers: full[NS], empty[NS], s_full[2][2], p_full[2][2], o_done[2][2], drain
  static constexpr int kNumBars = 2 * NS + 4 + 4 + 4 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag, merge flag
  static constexpr int kLoFlagOff = kMiscOff + 16;          // int [2][2]: P residual written, per M-tile and buffer
  // then the rotary table of the segment (rope_table_bytes, 0 without
  // positions) and the tile starts of the work plan
  static constexpr int kRopeOff = kLoFlagOff + 16;
  static constexpr int kThreads = (5 * NMT + 2) * 32;
};

// Offset of chunk c (16 B) of row r in a 128-row, 128B-swizzled Q tile pair.
__device__ __forceinline__ uint32_t swz128(int r, int c) {
  return (uint32_t)((c >> 3) * (128 * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int NMT, bool kTma, bool kRope, int NS>
__global__ void __launch_bounds__(TcSmem<NMT, NS>::kThreads, 1)
    verify_attn_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv) {
  using SM = TcSmem<NMT, NS>;
  using Geo = StageGeom<__nv_bfloat16, 128>;
  constexpr int D = 128;
  constexpr int kSoftThreads = 128 * NMT;
  constexpr int kProducerWarp = 4 * NMT;
  constexpr int kMmaWarp0 = 4 * NMT + 1;  // PV issuer of M-tile i is warp kMmaWarp0 + i
  constexpr int kSWarp = 5 * NMT + 1;     // S issuer of every M-tile
  constexpr int kMmaThreads = 32 * (NMT + 1);
  constexpr int kBarQ = 1, kBarSoft = 2, kBarEnd = 3, kBarVote = 4;  // kBarVote + M-tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *sQ = smem;
  uint8_t *stages = smem + SM::kStagesOff;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kBarOff);
  uint64_t *full = bars;
  uint64_t *empty = bars + NS;
  uint64_t *s_full = bars + 2 * NS;       // [i][b] at 2*i + b, b = tile parity = buffer
  uint64_t *p_full = bars + 2 * NS + 4;   // [i][b]
  uint64_t *o_done = bars + 2 * NS + 8;   // [i][b]
  uint64_t *drain = bars + 2 * NS + 12;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SM::kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM::kMiscOff + 4);
  volatile int *merge_ok = abort_flag + 1;
  float2 *rope_tab = reinterpret_cast<float2 *>(smem + SM::kRopeOff);
  int *tstart = reinterpret_cast<int *>(smem + SM::kRopeOff + (kRope ? rope_table_bytes(p) : 0));
  volatile int *lo_flag = reinterpret_cast<volatile int *>(smem + SM::kLoFlagOff);
  constexpr bool use_tma = kTma;  // tiles by TMA boxes (dense, paged), else cp.async gathers

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = blockIdx.x;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full + i, use_tma ? 1 : 32);
      mbar_init(empty + i, NMT);  // one arrive per M-tile issuer
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 128);
      mbar_init(o_done + i, 1);
    }
    mbar_init(drain, NMT + 1);  // one commit per MMA-issuing warp
    *abort_flag = 0;
    fence_mbar_init();
  }
  const CtaRange cr = plan_cta(p, tstart);  // contains __syncthreads
  if (c >= cr.G) return;
  const int t0 = cr.t0, t1 = cr.t1, s0 = cr.s0;

  if (warp == kProducerWarp) {
    bool pok = true;
    // at most NS-1 tiles in flight, and the second waits for the first: the
    // first tile of every CTA lands sooner when the kernel starts (-1 us)
    produce_tiles<__nv_bfloat16, D, NS, kTK, NS - 1, 1, kTma ? 1 : 0>(p, &tmk, &tmv, tstart, cr, stages, full, empty,
                                                                  abort_flag, use_tma, pok);
    return;
  }

  // TMEM: 512 columns, allocated by the MMA warp
  if (warp == kMmaWarp0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  named_bar_sync(kBarEnd, kSoftThreads + kMmaThreads);
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const float cl2 = p.scale * kLog2e;
  const int group = p.Hq / p.Hkv;

  if (warp >= kMmaWarp0) {
    // ================== MMA issuers: PV of M-tile mi, or S of all ==================
    const bool s_issuer = warp == kSWarp;
    const int mi = s_issuer ? 0 : warp - kMmaWarp0;
    const uint32_t id_s = umma_idesc(128, 64, 0, 0);
    const uint32_t id_o = umma_idesc(128, 128, 0, 1);
    int it = 0, jt = 0;
    bool ok = true;
    auto wait_ok = [&](uint64_t *bar, uint32_t parity) { role_wait(bar, parity, ok, abort_flag, p.wait_ns, p.status); };
    // make stage `st` of tile lt ready for the MMAs: wait for it; on the dense
    // path zero the V rows past the segment end (TMA brought whole boxes)
    auto acquire_stage = [&](int st, uint32_t ph, int lt, const Seg &g) {
      wait_ok(full + st, ph);
      if (ok && use_tma && lt * kTK + kTK > g.nkeys) {
        uint8_t *vt = stages + st * Geo::kStageBytes + Geo::kTileBytes;
        for (int e = lane; e < kTK * Geo::kChunks; e += 32) {
          const int r = e / Geo::kChunks;
          if (lt * kTK + r >= g.nkeys) *reinterpret_cast<uint4 *>(vt + swz(r, e % Geo::kChunks)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
    };
    // Shared-memory descriptors are built once; a K-step or stage offset is an
    // add to the start-address field (addresses stay below 256 KB, so the
    // 14-bit field never carries).
    const uint64_t dQ0 = umma_sdesc(smem_u32(sQ), 16, 1024);
    const uint64_t dK0 = umma_sdesc(smem_u32(stages), 16, 1024);
    const uint64_t dV0 = umma_sdesc(smem_u32(stages) + Geo::kTileBytes, 8192, 1024);
    constexpr uint64_t kStageStep = Geo::kStageBytes >> 4;
    auto issue_s = [&](int i, int b, int st) {  // S_i(b) = Q_i K^T
      if (!ok) return;
      tc_fence_after();
      const uint64_t dK = dK0 + (uint64_t)st * kStageStep;
      const uint32_t dS = tmem + 256 + 64 * (2 * i + b);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t qoff = (uint64_t)(((ks >> 2) * 16384 + (ks & 3) * 32) >> 4);
        const uint64_t koff = (uint64_t)(((ks >> 2) * 8192 + (ks & 3) * 32) >> 4);
        umma_ss_warp(dS, dQ0 + (uint64_t)(i * (32768 >> 4)) + qoff, dK + koff, id_s, ks > 0 ? 1u : 0u);
      }
      umma_commit_warp(s_full + 2 * i + b);
    };
    auto issue_pv = [&](int i, int b, int st, bool first, bool exact) {  // O_i += P_i V
      if (!ok) return;
      tc_fence_after();
      const uint64_t dV = dV0 + (uint64_t)st * kStageStep;
      const uint32_t aP = tmem + 256 + 64 * (2 * i + b);  // P hi; the residual 32 columns on
      const uint32_t dO = tmem + 128 * i;
#pragma unroll
      for (int kk = 0; kk < kTK / 16; ++kk) {
        const uint64_t bb = dV + (uint64_t)((kk * 2048) >> 4);
        umma_ts_warp(dO, aP + kk * 8, bb, id_o, (!first || kk > 0) ? 1u : 0u);
        if (exact) umma_ts_warp(dO, aP + 32 + kk * 8, bb, id_o, 1u);
      }
      umma_commit_warp(o_done + 2 * i + b);
      umma_commit_warp(empty + st);  // this M-tile is done with the K/V stage once these complete
    };

    for (int s = s0; s < p.S && tstart[s] < t1; ++s) {
      const Seg g = seg_info(p, s, false);
      const int lt0 = max(tstart[s], t0) - tstart[s];
      const int lt1 = min(tstart[s + 1], t1) - tstart[s];
      named_bar_sync(kBarQ, kSoftThreads + kMmaThreads);  // Q of this segment is in shared memory
      for (int lt = lt0; lt < lt1; ++lt, ++it, ++jt) {
        const int st = it % NS;
        const int b = jt & 1;
        if (s_issuer) {
          // S(t) of each M-tile into buffer b once PV(t-2) has read P from it
#pragma unroll
          for (int i = 0; i < NMT; ++i) {
            if (jt >= 2) wait_ok(o_done + 2 * i + b, (uint32_t)((jt - 2) >> 1) & 1u);
            if (i == 0) {
              wait_ok(full + st, (uint32_t)(it / NS) & 1u);
              if (kRope && ok && lt * kTK + kTK > g.n_prefix) {
                // the draft keys of this tile, rotated in place before the S MMAs read them
                const int r0 = max(0, g.n_prefix - lt * kTK), r1 = min(kTK, g.nkeys - lt * kTK);
                rope_rotate_tile_rows<__nv_bfloat16, D, kTK>(stages + st * Geo::kStageBytes, r0, r1,
                                                             lt * kTK + r0 - g.n_prefix, rope_tab, lane, 32);
                fence_proxy_async_smem();
                __syncwarp();
              }
            }
            tc_fence_after();
            issue_s(i, b, st);
          }
        } else {
          wait_ok(p_full + 2 * mi + b, (uint32_t)(jt >> 1) & 1u);
          // the softmax wrote the P residual of this tile too (set before its
          // arrive on p_full; rewritten only after this PV has completed)
          const bool exact = lo_flag[2 * mi + b] != 0;
          acquire_stage(st, (uint32_t)(it / NS) & 1u, lt, g);
          issue_pv(mi, b, st, lt == lt0, exact);
        }
        __syncwarp();
      }
    }
    // drain: every MMA the issuers started has finished before TMEM is released
    umma_commit_warp(drain);
    mbar_wait(drain, 0u, p.wait_ns);
    tc_fence_before();
    named_bar_sync(kBarEnd, kSoftThreads + kMmaThreads);
    tc_fence_after();
    if (warp == kMmaWarp0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    return;
  }

  // ============================ softmax warpgroups ============================
  const int mi = warp >> 2;                 // M-tile of this warpgroup
  const int r = (warp & 3) * 32 + lane;     // row in the M-tile = TMEM lane
  const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t tO = tmem + lane_bits + 128 * mi;
  bool ok = true;
  auto wait_ok = [&](uint64_t *bar, uint32_t parity) { role_wait(bar, parity, ok, abort_flag, p.wait_ns, p.status); };
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

    // the draft structure of the part, when it holds draft keys (parents, or
    // the mask words of tokens lane and lane + 32): loaded now, so that the
    // round trip overlaps the one of Q
    const bool has_draft = lt1 * kTK > g.n_prefix;
    DraftPre dpre{-1, -1, 0ull, 0ull};
    if (has_draft) dpre = draft_prefetch(p, g.b);
    // ---- Q of this segment into shared memory (both warpgroups) ----
    named_bar_sync(kBarSoft, kSoftThreads);  // previous segment's MMAs have all completed
    if constexpr (kRope) {
      // rotary table of this sequence's draft tokens (kept while the CTA stays
      // on the sequence), then q rotated on its way in
      if (g.b != rope_b) {
        rope_build_table(p, g.b, rope_tab, tid, kSoftThreads);
        named_bar_sync(kBarSoft, kSoftThreads);
        rope_b = g.b;
      }
      const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q);
      constexpr int kQIt = NMT * 128 * 8 / kSoftThreads;
      uint4 lo[kQIt], hi[kQIt];
#pragma unroll
      for (int u = 0; u < kQIt; ++u) {  // loads first: one round trip
        const int e = tid + u * kSoftThreads;
        const int rr = g.rb * p.rows_pad + (e / (128 * 8)) * 128 + (e / 8) % 128;
        lo[u] = hi[u] = make_uint4(0, 0, 0, 0);
        if (rr < p.R) {
          const int t = rr / group;
          const int hq = g.hkv * group + rr % group;
          const uint4 *src = reinterpret_cast<const uint4 *>(qb + (((size_t)g.b * p.T + t) * p.Hq + hq) * D);
          lo[u] = __ldg(src + e % 8);
          hi[u] = __ldg(src + e % 8 + 8);
        }
      }
#pragma unroll
      for (int u = 0; u < kQIt; ++u) {
        const int e = tid + u * kSoftThreads;
        const int m = e / (128 * 8);
        const int row = (e / 8) % 128;
        const int ch = e % 8;
        const int rr = g.rb * p.rows_pad + m * 128 + row;
        if (rr < p.R) rope_rotate8_bf16(lo[u], hi[u], rope_tab + (rr / group) * (D / 2) + ch * 8);
        *reinterpret_cast<uint4 *>(sQ + m * 32768 + swz128(row, ch)) = lo[u];
        *reinterpret_cast<uint4 *>(sQ + m * 32768 + swz128(row, ch + 8)) = hi[u];
      }
      fence_proxy_async_smem();
    } else {
      // every load of the thread in flight before the first store (one round
      // trip, not one per row chunk)
      const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q);
      constexpr int kQIt = NMT * 128 * 16 / kSoftThreads;
      uint4 v[kQIt];
#pragma unroll
      for (int u = 0; u < kQIt; ++u) {
        const int e = tid + u * kSoftThreads;
        const int m = e / (128 * 16);
        const int row = (e / 16) % 128;
        const int rr = g.rb * p.rows_pad + m * 128 + row;
        v[u] = make_uint4(0, 0, 0, 0);
        if (rr < p.R) {
          const int t = rr / group;
          const int hq = g.hkv * group + rr % group;
          v[u] = __ldg(reinterpret_cast<const uint4 *>(qb + (((size_t)g.b * p.T + t) * p.Hq + hq) * D) + e % 16);
        }
      }
#pragma unroll
      for (int u = 0; u < kQIt; ++u) {
        const int e = tid + u * kSoftThreads;
        *reinterpret_cast<uint4 *>(sQ + (e / (128 * 16)) * 32768 + swz128((e / 16) % 128, e % 16)) = v[u];
      }
      fence_proxy_async_smem();
    }
    named_bar_arrive(kBarQ, kSoftThreads + kMmaThreads);

    const int rr = g.rb * p.rows_pad + mi * 128 + r;
    const bool rvalid = rr < p.R;
    const int t = rvalid ? rr / group : 0;
    const int hq = g.hkv * group + (rvalid ? rr % group : 0);
    uint64_t rmask = 0;  // the draft keys this row sees
    if (has_draft) {
      uint64_t tl, th;
      draft_rows(p, dpre, tl, th);
      const uint64_t a = __shfl_sync(0xffffffffu, tl, t & 31), c2 = __shfl_sync(0xffffffffu, th, t & 31);
      rmask = t < 32 ? a : c2;
    }
    float m_used = -INFINITY;  // reference max of the exponentials (raw score units)
    float l = 0.f;

    for (int lt = lt0; lt < lt1; ++lt, ++jt) {
      const int b = jt & 1;
      const uint32_t tS = tmem + lane_bits + 256 + 64 * (2 * mi + b);
      wait_ok(s_full + 2 * mi + b, (uint32_t)(jt >> 1) & 1u);
      tc_fence_after();
      float sv[64];
      {  // both halves in flight before the one wait
        uint32_t u[32], w[32];
        tmem_ld32(tS, u);
        tmem_ld32(tS + 32, w);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[j] = __uint_as_float(u[j]);
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[32 + j] = __uint_as_float(w[j]);
      }
      const int k0 = lt * kTK;
      const bool masked = k0 + kTK > g.n_prefix;
      if (masked) {
        const uint64_t vis = tile_vis64(k0, g.n_prefix, g.nkeys, rmask);
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (!((vis >> j) & 1ull)) sv[j] = -INFINITY;
      }
      float mx;
      {  // three-input maxima: 32 instructions, short dependency chains
        float m22[22];
#pragma unroll
        for (int q = 0; q < 21; ++q) m22[q] = max3f(sv[3 * q], sv[3 * q + 1], sv[3 * q + 2]);
        m22[21] = sv[63];
        float m8[8];
#pragma unroll
        for (int q = 0; q < 7; ++q) m8[q] = max3f(m22[3 * q], m22[3 * q + 1], m22[3 * q + 2]);
        m8[7] = m22[21];
        mx = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      }
      const float m_new = fmaxf(m_used, mx);
      // move the reference max only when it grew by more than 2^8 (exact either
      // way); O is rescaled below, once P is written and the scores are dead
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
      if (r == 0) lo_flag[2 * mi + b] = lo ? 1 : 0;
      uint32_t ph[32];
      // packed pairs: the scaled argument and the running sums take one
      // instruction per two scores
      const float2 cl2v = make_float2(cl2, cl2), nmu = make_float2(-mu, -mu);
      float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      if (lo) {
        // P as bf16 hi + lo parts (a second set of MMAs adds the lo parts)
        uint32_t pl[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float2 x = fma2(make_float2(sv[2 * j], sv[2 * j + 1]), cl2v, nmu);
          const float a = ex2_approx(x.x), bq = ex2_approx(x.y);
          ls2[j & 1] = add2(ls2[j & 1], make_float2(a, bq));
          split_bf16x2(a, bq, ph[j], pl[j]);
        }
        tmem_st32(tS, ph);
        tmem_st32(tS + 32, pl);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float2 x = fma2(make_float2(sv[2 * j], sv[2 * j + 1]), cl2v, nmu);
          const float a = ex2_approx(x.x), bq = ex2_approx(x.y);
          ls2[j & 1] = add2(ls2[j & 1], make_float2(a, bq));
          ph[j] = pack_bf16(a, bq);
        }
        tmem_st32(tS, ph);
      }
      const float ls = (ls2[0].x + ls2[1].x) + (ls2[0].y + ls2[1].y);
      l += ls;
      if (rescale) {
        // O relative to the new reference before PV(jt) adds to it; O holds
        // every PV up to tile jt-1 once that one has completed
        wait_ok(o_done + 2 * mi + (b ^ 1), (uint32_t)((jt - 1) >> 1) & 1u);
        tc_fence_after();
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
      mbar_arrive(p_full + 2 * mi + b);
    }

    // ---- epilogue: O / l for this segment part (the last two PVs, in order) ----
    if (jt >= 2) wait_ok(o_done + 2 * mi + (jt & 1), (uint32_t)((jt - 2) >> 1) & 1u);
    wait_ok(o_done + 2 * mi + ((jt - 1) & 1), (uint32_t)((jt - 1) >> 1) & 1u);
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_nat = l > 0.f ? (m_used * cl2 + log2f(l)) * kLn2 : -INFINITY;
    const bool write = rvalid && ok;
    const uint32_t wrows = __ballot_sync(0xffffffffu, write);  // rows of this warp that are written
#pragma unroll
    for (int cch = 0; cch < 4; ++cch) {
      uint32_t u[32];
      tmem_ld32(tO + 32 * cch, u);
      tmem_ld_wait();
      if (n_parts == 1) {
        if (!write) continue;
        uint4 *ob = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) +
                                              (((size_t)g.b * p.T + t) * p.Hq + hq) * D + 32 * cch);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 v;
          v.x = pack_bf16(__uint_as_float(u[8 * q4 + 0]) * inv, __uint_as_float(u[8 * q4 + 1]) * inv);
          v.y = pack_bf16(__uint_as_float(u[8 * q4 + 2]) * inv, __uint_as_float(u[8 * q4 + 3]) * inv);
          v.z = pack_bf16(__uint_as_float(u[8 * q4 + 4]) * inv, __uint_as_float(u[8 * q4 + 5]) * inv);
          v.w = pack_bf16(__uint_as_float(u[8 * q4 + 6]) * inv, __uint_as_float(u[8 * q4 + 7]) * inv);
          ob[q4] = v;
        }
      } else {
        // the warp's 32 rows through a 32 x 33 float tile in the Q buffer (its
        // segment's S MMAs are all done): lane j then stores column j of each
        // row, so every store writes 128 contiguous bytes of one row
        float *tr = reinterpret_cast<float *>(sQ) + warp * (32 * 33);
#pragma unroll
        for (int j = 0; j < 32; ++j) tr[lane * 33 + j] = __uint_as_float(u[j]) * inv;
        __syncwarp();
        float *op = p.o_part + ((size_t)(s + c) * p.rows_pad + mi * 128 + (warp & 3) * 32) * D + 32 * cch + lane;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if ((wrows >> i) & 1u) op[(size_t)i * D] = tr[i * 33 + lane];
        __syncwarp();
      }
    }
    if (write) {
      if (n_parts == 1)
        p.lse[((size_t)g.b * p.Hq + hq) * p.T + t] = lse_nat;
      else
        p.lse_part[(size_t)(s + c) * p.rows_pad + mi * 128 + r] = lse_nat;
    }
    if (n_parts > 1) {
      // publish the part (always, also after a failed wait, so the counters
      // return to zero): the barrier orders every warpgroup's row and lse
      // stores before thread 0's release increment, which is cumulative
      named_bar_sync(kBarSoft, kSoftThreads);
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

  // ---- merge of the split segments (LongSpec 2.C): once every part of a
  // segment has arrived, each of its CTAs merges an equal share of its rows ----
  for (int k = 0; k < n_split; ++k) {
    const int s = ms[k], np = mnp[k];
    if (tid == 0) *merge_ok = wait_parts_arrived(p, s, np) ? 1 : 0;
    named_bar_sync(kBarSoft, kSoftThreads);  // thread 0's acquire, then the barrier, orders the reads below
    if (*merge_ok) {
      const int rb = s % p.NRB, hkv = (s / p.NRB) % p.Hkv, b = s / (p.NRB * p.Hkv);
      const int nrows = min(p.rows_pad, p.R - rb * p.rows_pad);
      const int r0 = mpart[k] * nrows / np, r1 = (mpart[k] + 1) * nrows / np;
      if (np <= 4)
        merge_rows_warp<8, 4>(p, b, hkv, rb * p.rows_pad, mslot[k], np, r0, r1, warp, 4 * NMT, lane);
      else
        merge_rows_warp<32, 24>(p, b, hkv, rb * p.rows_pad, mslot[k], np, r0, r1, warp, 4 * NMT, lane);
    }
    named_bar_sync(kBarSoft, kSoftThreads);
    // leave: np arrivals and np departures wrap the counter back to zero
    if (tid == 0) red_relaxed_inc_gpu(reinterpret_cast<unsigned *>(&p.merge_cnt[s].x), 2u * np - 1u);
  }
  tc_fence_before();
  named_bar_sync(kBarEnd, kSoftThreads + kMmaThreads);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int NMT, int NS>
static size_t tc_smem_bytes(const AttnParams &p) {
  return 1024 + (size_t)TcSmem<NMT, NS>::kRopeOff + (size_t)rope_table_bytes(p) + (size_t)(p.S + 1) * 4;
}

constexpr size_t kTcSmemLimit = 232448;  // bytes of dynamic shared memory a CTA may have

// the ring depth an instance gets: the largest that fits the plan
template <int NMT>
static bool tc_deep_ring(const AttnParams &p) {
  return tc_smem_bytes<NMT, kTcStagesMax>(p) <= kTcSmemLimit;
}

size_t attn_tc_smem_required(const AttnParams &p) {
  return p.rows_pad > 128 ? tc_smem_bytes<2, kTcStagesMin>(p) : tc_smem_bytes<1, kTcStagesMin>(p);
}

template <int NMT, bool kTma, bool kRope, int NS>
static cudaError_t launch_tc_ns(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                                cudaStream_t stream) {
  const size_t smem = tc_smem_bytes<NMT, NS>(p);
  auto kern = verify_attn_tc_kernel<NMT, kTma, kRope, NS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // cooperative: every CTA is resident, so the wait for a segment's parts ends
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(TcSmem<NMT, NS>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tmk, tmv);
}

// instances with and without the rotary embedding (code that never runs still
// costs the hot loop), each with the deep ring or the minimum one
template <int NMT, bool kTma>
static cudaError_t launch_tc_t(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                               cudaStream_t stream) {
  if (p.positions != nullptr)
    return tc_deep_ring<NMT>(p)
               ? launch_tc_ns<NMT, kTma, true, kTcStagesMax>(p, tmk, tmv, grid, stream)
               : launch_tc_ns<NMT, kTma, true, kTcStagesMin>(p, tmk, tmv, grid, stream);
  return tc_deep_ring<NMT>(p)
             ? launch_tc_ns<NMT, kTma, false, kTcStagesMax>(p, tmk, tmv, grid, stream)
             : launch_tc_ns<NMT, kTma, false, kTcStagesMin>(p, tmk, tmv, grid, stream);
}

cudaError_t launch_attention_tc(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                                cudaStream_t stream) {
  const bool tma = p.tma_box > 0;
  if (p.rows_pad > 128)
    return tma ? launch_tc_t<2, true>(p, tmk, tmv, grid, stream) : launch_tc_t<2, false>(p, tmk, tmv, grid, stream);
  return tma ? launch_tc_t<1, true>(p, tmk, tmv, grid, stream) : launch_tc_t<1, false>(p, tmk, tmv, grid, stream);
}

}  // namespace va
