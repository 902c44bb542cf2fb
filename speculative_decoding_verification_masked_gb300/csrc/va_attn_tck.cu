// Verification attention on the 5th-generation tensor cores with the KEYS on
// the TMEM lanes, for segments of at most 64 packed query rows (GQA group x T
// draft tokens; a chain of 8 drafts with group 4 gives 32 rows).  One MMA has
// M = 128, so rather than padding 32 query rows to 128 the products are taken
// transposed, with a 128-key tile as the M side:
//
//   S^T (128 keys x NR rows)   = K (128 x d) . Q^T       A = K tile, K-major; B = Q, K-major
//   O^T (128 d x 2NR)         += V^T . [P_hi | P_lo]^T   A = V tile, MN-major; B = P^T, MN-major
//   l   (2NR, every lane)     += 1 (128 x 128) . [P_hi | P_lo]^T   (64 rows only; A = ones in TMEM)
//
// (LongSpec 2.C: the unmasked prefix and the masked draft block are the same
// tile loop, the draft block being the last tiles of a segment; partial
// results of a segment split over CTAs are merged by the exact log-sum-exp
// combine.)  P is split into a bf16 high part and the bf16 rounding of its
// residual, and both are multiplied by ONE MMA whose N covers the two halves:
// the accumulator columns of O_hi and O_lo sit side by side and are added in
// the epilogue.  ~16 bits of every weight survive, so a row whose weight rests
// on a few keys (attention sinks) keeps the exact result to well below the
// bf16 output rounding, at no extra MMA: an MMA of N <= 128 costs the same
// issue time as one of half that width.
//
// Roles (6 warps, 7 when a second producer warp shares a gather; one CTA per
// SM, cooperative launch):
//   warps 0-3  softmax: thread k owns key k of the tile (TMEM lane k) and all
//              NR rows of it.  Scores are taken in log2 units against a
//              per-row reference max that moves only when some score of the
//              tile exceeds it by more than 2^8 (exact either way: the
//              exponentials stay below 2^8 and O, l are rescaled when it
//              moves); whether it must move is one block-wide vote (bar.red),
//              and only then are the row maxima reduced across the 128 keys.
//              P (bf16 hi and lo parts) is written as the MN-major P^T
//              operand over the K tile of the same stage, which the S MMA has
//              finished reading.  In the epilogue thread d owns output column d.
//   warp 4     producer: TMA boxes (dense, paged with pages of 8 rows or more)
//              or cp.async gathers (sparse, small pages) into a 3-stage ring
//              of 128-key K and V tiles (64 KB a stage)
//   warp 5     MMA issuer and TMEM owner: S of tile i+2 is issued as soon as
//              the softmax of tile i has released its S buffer.
// TMEM columns (NC = max(NR, 32)): O^T hi at 0 and lo at NR, S buffers at 2NC
// and 3NC, the ones operand at 4NC, l hi / lo (64 rows) at 5NC and 5NC + NR.
// Every wait is bounded; on timeout the CTA
// records VA_ERR_TIMEOUT, keeps the barrier sequence of all roles, drains and
// frees TMEM.
#include <cuda.h>
#include <math.h>

#include "va_common.cuh"
#include "va_kernels.h"
#include "va_pipeline.cuh"
#include "va_merge.cuh"
#include "va_rope_fused.cuh"
#include "va_tcgen05.cuh"

namespace va {

constexpr int kTkKeys = 128;  // keys per tile
constexpr int kTkStages = 3;
// Warps: 0-3 softmax, 4 producer, 5 MMA issuer, then NR <= 32 adds a second
// producer warp that shares the cp.async gather of the paged / sparse layouts
// (one warp's gather is limited by the copies it can keep in flight).  Seven
// warps leave at most two per SM sub-partition, so 255 registers stay available.
template <int NR, bool kTma>
struct TkCfg {
  static constexpr int kProducers = !kTma && NR <= 32 ? 2 : 1;
  static constexpr int kThreads = (5 + kProducers) * 32;
};

template <int NR>
struct TkSmem {
  using Geo = StageGeom<__nv_bfloat16, 128, kTkKeys>;
  static constexpr int kStageBytes = Geo::kStageBytes;  // 64 KB
  static constexpr int kQOff = kTkStages * kStageBytes;
  static constexpr int kQBytes = 2 * NR * 128;  // two 128-byte columns of NR rows
  static constexpr int kBarOff = kQOff + kQBytes;
  // barriers: full[3], empty[3], s_full[2], p_full[2], o_done[2], drain
  static constexpr int kNumBars = 2 * kTkStages + 7;
  static constexpr int kMiscOff = (kBarOff + kNumBars * 8 + 15) & ~15;  // tmem base, abort flag, merge flag
  static constexpr int kRowMaskOff = kMiscOff + 16;        // u64 [64]: draft visibility rows
  static constexpr int kKeyMaskOff = kRowMaskOff + 512;    // u64 [64]: per draft key, rows that see it
  static constexpr int kRedOff = kKeyMaskOff + 512;        // float4 [NR]: per-warp row maxima
  static constexpr int kRowInvOff = kRedOff + NR * 16;     // float [64]: 1 / l per row (epilogue)
  // then the rotary table of the segment (rope_table_bytes, 0 without
  // positions) and the tile starts of the work plan
  static constexpr int kRopeOff = kRowInvOff + 256;
  static_assert(kQOff % 1024 == 0 && kQBytes % 1024 == 0, "UMMA operands need 1024-byte aligned swizzle atoms");
  static_assert(kBarOff % 8 == 0 && kRowMaskOff % 8 == 0 && kKeyMaskOff % 8 == 0, "8-byte alignment");
  static_assert(kRedOff % 16 == 0, "float4 array needs 16-byte alignment");
  static_assert(kRowInvOff % 16 == 0, "vector loads of the row constants");
  static constexpr int kNC = NR < 32 ? 32 : NR;            // TMEM columns per region
  static constexpr int kTmemCols = NR <= 32 ? 256 : 512;
  // O_hi | O_lo take columns [0, 2NR): within O and the (unused) l region for
  // NR <= 32; for 64 rows l moves past the ones operand
  static constexpr int kLCol = NR <= 32 ? kNC : 5 * kNC;
  static_assert(2 * NR <= 2 * kNC && kLCol + 2 * NR <= kTmemCols, "TMEM plan");
};

// Row-wise block of a warp: v[N] per lane -> lane holds the warp maximum of
// max(N/32, 1) rows (row j + (N/32)*lane for N >= 32, lane / (32/N) below).
template <int N, int O>
struct WarpScatterMax {
  static __device__ __forceinline__ void run(float *v, int lane) {
    if constexpr (O == 0) {
      return;
    } else if constexpr (N >= 2) {
      constexpr int H = N / 2;
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = up ? v[i] : v[i + H];
        const float keep = up ? v[i + H] : v[i];
        v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, O));
      }
      WarpScatterMax<H, O / 2>::run(v, lane);
    } else {
      v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], O));
      WarpScatterMax<1, O / 2>::run(v, lane);
    }
  }
};

// The same reduce-scatter with sums: lane l ends with the warp's sum of the
// rows WarpScatterMax leaves it.
template <int N, int O>
struct WarpScatterSum {
  static __device__ __forceinline__ void run(float *v, int lane) {
    if constexpr (O == 0) {
      return;
    } else if constexpr (N >= 2) {
      constexpr int H = N / 2;
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = up ? v[i] : v[i + H];
        const float keep = up ? v[i + H] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      WarpScatterSum<H, O / 2>::run(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      WarpScatterSum<1, O / 2>::run(v, lane);
    }
  }
};

// NR fp32 columns of this thread's TMEM lane.
template <int NR>
__device__ __forceinline__ void tmem_ld_f(uint32_t taddr, float (&x)[NR]) {
  if constexpr (NR == 8) {
    uint32_t u[8];
    tmem_ld8(taddr, u);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = __uint_as_float(u[j]);
  } else if constexpr (NR == 16) {
    uint32_t u[16];
    tmem_ld16(taddr, u);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = __uint_as_float(u[j]);
  } else {
#pragma unroll
    for (int h = 0; h < NR / 32; ++h) {
      uint32_t u[32];
      tmem_ld32(taddr + 32 * h, u);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) x[32 * h + j] = __uint_as_float(u[j]);
    }
  }
}

// O_hi + O_lo: N fp32 columns at taddr plus the N columns `lo` further on.
template <int N>
__device__ __forceinline__ void tmem_ld_hilo(uint32_t taddr, uint32_t lo, float (&x)[N]) {
  float y[N];
  tmem_ld_f<N>(taddr, x);
  tmem_ld_f<N>(taddr + lo, y);
#pragma unroll
  for (int j = 0; j < N; ++j) x[j] += y[j];
}

// Multiply column j of this lane's NR columns at taddr by a[j].
template <int NR>
__device__ __forceinline__ void tmem_scale_cols(uint32_t taddr, const float *a) {
  if constexpr (NR == 16) {
    uint32_t u[16];
    tmem_ld16(taddr, u);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) u[j] = __float_as_uint(__uint_as_float(u[j]) * a[j]);
    tmem_st16(taddr, u);
  } else {
    // 16 columns at a time, each stored before the next is loaded: this rare
    // path then needs few registers next to the 64-row softmax state
#pragma unroll
    for (int h = 0; h < NR / 16; ++h) {
      uint32_t u[16];
      tmem_ld16(taddr + 16 * h, u);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) u[j] = __float_as_uint(__uint_as_float(u[j]) * a[16 * h + j]);
      tmem_st16(taddr + 16 * h, u);
      tmem_st_wait();
    }
  }
}

template <int NR, bool kTma, bool kRope>
__global__ void __launch_bounds__(TkCfg<NR, kTma>::kThreads, 1)
    verify_attn_tck_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                           const __grid_constant__ CUtensorMap tmv) {
  using SM = TkSmem<NR>;
  using Geo = typename SM::Geo;
  constexpr int D = 128;
  constexpr int TK = kTkKeys;
  constexpr int NS = kTkStages;
  constexpr int NC = SM::kNC;
  constexpr int kSoft = 128;
  // NR <= 32: the row sums l are kept by the softmax threads (each over its own
  // keys, reduced once per segment part) instead of a ones-operand MMA per tile
  constexpr bool kRegL = NR <= 32;
  constexpr int kProducerWarp = 4, kMmaWarp = 5;
  constexpr int kBarQ = 1, kBarRed = 2, kBarSoft = 3, kBarEnd = 4;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *stages = smem;
  uint8_t *sQ = smem + SM::kQOff;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kBarOff);
  uint64_t *full = bars;
  uint64_t *empty = bars + NS;
  uint64_t *s_full = bars + 2 * NS;      // [b]
  uint64_t *p_full = bars + 2 * NS + 2;  // [b]
  uint64_t *o_done = bars + 2 * NS + 4;  // [tile & 1]
  uint64_t *drain = bars + 2 * NS + 6;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SM::kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM::kMiscOff + 4);
  uint64_t *rowmask = reinterpret_cast<uint64_t *>(smem + SM::kRowMaskOff);
  uint64_t *keymask = reinterpret_cast<uint64_t *>(smem + SM::kKeyMaskOff);
  float4 *red = reinterpret_cast<float4 *>(smem + SM::kRedOff);
  float *row_inv = reinterpret_cast<float *>(smem + SM::kRowInvOff);
  float2 *rope_tab = reinterpret_cast<float2 *>(smem + SM::kRopeOff);
  int *tstart = reinterpret_cast<int *>(smem + SM::kRopeOff + (kRope ? rope_table_bytes(p) : 0));
  constexpr bool use_tma = kTma;  // tiles by TMA boxes (dense, paged), else cp.async gathers

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = blockIdx.x;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full + i, use_tma ? 1 : 32 * TkCfg<NR, kTma>::kProducers);
      mbar_init(empty + i, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(p_full + b, kSoft);
    }
    mbar_init(o_done + 0, 1);
    mbar_init(o_done + 1, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  const CtaRange cr = plan_cta<TK>(p, tstart);  // contains __syncthreads
  if (c >= cr.G) return;
  const int t0 = cr.t0, t1 = cr.t1, s0 = cr.s0;

  if (warp == kProducerWarp || warp > kMmaWarp) {
    bool pok = true;
    produce_tiles<__nv_bfloat16, D, NS, TK, 2, TkCfg<NR, kTma>::kProducers, kTma ? 1 : 0>(
        p, &tmk, &tmv, tstart, cr, stages, full, empty, abort_flag, use_tma, pok,
        warp == kProducerWarp ? 0 : warp - kMmaWarp);
    return;
  }

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(SM::kTmemCols)
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
    const uint32_t id_s = umma_idesc(128, NR, 0, 0);
    const uint32_t id_o = umma_idesc(128, 2 * NR, 1, 1);  // N = [P_hi | P_lo]
    const uint32_t id_l = umma_idesc(128, 2 * NR, 0, 1);
    const uint32_t tO = tmem, tL = tmem + SM::kLCol, tOnes = tmem + 4 * NC;
    int it = 0, jt = 0;
    // Shared-memory descriptors are built once; a K-step or stage offset is an
    // add to the start-address field (addresses stay below 256 KB, so the
    // 14-bit field never carries).
    const uint64_t dK0 = umma_sdesc(smem_u32(stages), 16, 1024);                      // K tile, K-major
    const uint64_t dQ0 = umma_sdesc(smem_u32(sQ), 16, 1024);                          // Q, K-major
    const uint64_t dV0 = umma_sdesc(smem_u32(stages) + Geo::kTileBytes, TK * 128, 1024);  // V tile, MN-major
    // P^T over the K tile: per key a 128-byte row of the hi then lo parts (N =
    // 2NR <= 64, one swizzle atom wide), or for 64 rows hi and lo as two atoms
    // 16 KB apart
    const uint64_t dP0 = umma_sdesc(smem_u32(stages), TK * 128, 1024);
    constexpr uint64_t kStageStep = SM::kStageBytes >> 4;
    auto issue_s = [&](int b, int st, const Seg &g, int lt) {  // S^T(b) = K Q^T
      if (kRope && ok && lt * TK + TK > g.n_prefix) {
        // the draft keys of this tile, rotated in place before the MMA reads them
        const int r0 = max(0, g.n_prefix - lt * TK), r1 = min(TK, g.nkeys - lt * TK);
        rope_rotate_tile_rows_bf16_call<D, TK>(stages + st * SM::kStageBytes, r0, r1, lt * TK + r0 - g.n_prefix,
                                               rope_tab, lane, 32);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (!ok) return;
      tc_fence_after();
      const uint64_t dK = dK0 + (uint64_t)st * kStageStep;
      const uint32_t dS = tmem + (2 + b) * NC;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t koff = (uint64_t)(((ks >> 2) * (TK * 128) + (ks & 3) * 32) >> 4);
        const uint64_t qoff = (uint64_t)(((ks >> 2) * (NR * 128) + (ks & 3) * 32) >> 4);
        umma_ss_warp(dS, dK + koff, dQ0 + qoff, id_s, ks > 0 ? 1u : 0u);
      }
      umma_commit_warp(s_full + b);
    };
    auto issue_pv = [&](int st, int b, bool first) {  // [O_hi|O_lo]^T += V^T [P_hi|P_lo]^T
      if (!ok) return;
      tc_fence_after();
      const uint64_t dV = dV0 + (uint64_t)st * kStageStep;
      const uint64_t dP = dP0 + (uint64_t)st * kStageStep;
      const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
      for (int kk = 0; kk < TK / 16; ++kk) {
        const uint64_t off = (uint64_t)((kk * 2048) >> 4);
        const uint32_t acc = kk > 0 ? 1u : acc0;
        umma_ss_warp(tO, dV + off, dP + off, id_o, acc);
        if constexpr (!kRegL) umma_ts_warp(tL, tOnes, dP + off, id_l, acc);
      }
      umma_commit_warp(o_done + b);
      umma_commit_warp(empty + st);  // the stage is free once these MMAs have read it
    };

    for (int s = s0; s < p.S && tstart[s] < t1; ++s) {
      const Seg g = seg_info(p, s, false);
      const int lt0 = max(tstart[s], t0) - tstart[s];
      const int lt1 = min(tstart[s + 1], t1) - tstart[s];
      named_bar_sync(kBarQ, kSoft + 32);  // Q of this segment is in shared memory
      wait_ok(full + it % NS, (uint32_t)(it / NS) & 1u);
      issue_s(jt & 1, it % NS, g, lt0);
      if (lt0 + 1 < lt1) {
        wait_ok(full + (it + 1) % NS, (uint32_t)((it + 1) / NS) & 1u);
        issue_s((jt + 1) & 1, (it + 1) % NS, g, lt0 + 1);
      }
      for (int lt = lt0; lt < lt1; ++lt, ++it, ++jt) {
        const int b = jt & 1;
        wait_ok(p_full + b, (uint32_t)(jt >> 1) & 1u);
        issue_pv(it % NS, b, lt == lt0);
        if (lt + 2 < lt1) {
          wait_ok(full + (it + 2) % NS, (uint32_t)((it + 2) / NS) & 1u);
          issue_s(b, (it + 2) % NS, g, lt + 2);
        }
        __syncwarp();
      }
    }
    // drain: every MMA issued has finished before TMEM is released
    umma_commit_warp(drain);
    mbar_wait(drain, 0u, p.wait_ns);
    tc_fence_before();
    named_bar_sync(kBarEnd, kSoft + 32);
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(SM::kTmemCols)
                 : "memory");
    return;
  }

  // ================================== softmax ==================================
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t tO = tmem + lane_base, tL = tO + SM::kLCol;
  {  // the all-ones A operand of the row-sum MMA: 8 columns of bf16 pairs (1.0, 1.0)
    uint32_t ones[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ones[j] = 0x3F803F80u;
    tmem_st8(tO + 4 * NC, ones);
    tmem_st_wait();
  }
  int it = 0, jt = 0;
  int rope_b = -1;  // sequence whose rotary table is in shared memory
  // split segments this CTA holds a part of (at most its first and its last):
  // merged after its last tile
  int n_split = 0, ms[2] = {0, 0}, mslot[2] = {0, 0}, mnp[2] = {0, 0}, mpart[2] = {0, 0};
  for (int s = s0; s < p.S && tstart[s] < t1; ++s) {
    const Seg g = seg_info(p, s, false);
    const int lt0 = max(tstart[s], t0) - tstart[s];
    const int lt1 = min(tstart[s + 1], t1) - tstart[s];
    const int first_cta = owner_cta(tstart[s], cr.total, cr.G);
    const int n_parts = owner_cta(tstart[s + 1] - 1, cr.total, cr.G) - first_cta + 1;
    if (lt0 == 0 && tid == 0) p.meta[s] = make_int2(s + first_cta, n_parts);

    // ---- Q of this segment into shared memory: [2 columns][NR rows][128 B], 128B swizzle ----
    // (the previous segment's MMAs have completed: its epilogue waited for the last one)
    if constexpr (kRope) {
      // rotary table of this sequence's draft tokens (kept while the CTA stays
      // on the sequence), then q rotated on its way in
      if (g.b != rope_b) {
        rope_build_table(p, g.b, rope_tab, tid, kSoft);
        named_bar_sync(kBarSoft, kSoft);
        rope_b = g.b;
      }
      const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q);
      constexpr int kQIt = (NR * 8 + kSoft - 1) / kSoft;
      uint4 lo[kQIt], hi[kQIt];
#pragma unroll
      for (int u = 0; u < kQIt; ++u) {  // loads first: one round trip
        const int e = tid + u * kSoft;
        const int row = e >> 3;
        lo[u] = hi[u] = make_uint4(0, 0, 0, 0);
        if (e < NR * 8 && row < p.R) {
          const int t = row / group;
          const int hq = g.hkv * group + row % group;
          const uint4 *src = reinterpret_cast<const uint4 *>(qb + (((size_t)g.b * p.T + t) * p.Hq + hq) * D);
          lo[u] = __ldg(src + (e & 7));
          hi[u] = __ldg(src + (e & 7) + 8);
        }
      }
#pragma unroll
      for (int u = 0; u < kQIt; ++u) {
        const int e = tid + u * kSoft;
        if (e >= NR * 8) continue;
        const int row = e >> 3, ch = e & 7;
        if (row < p.R) rope_rotate8_bf16(lo[u], hi[u], rope_tab + (row / group) * (D / 2) + ch * 8);
        *reinterpret_cast<uint4 *>(sQ + row * 128 + ((ch ^ (row & 7)) << 4)) = lo[u];
        *reinterpret_cast<uint4 *>(sQ + NR * 128 + row * 128 + ((ch ^ (row & 7)) << 4)) = hi[u];
      }
      fence_proxy_async_smem();
    } else {
      // every load of the thread in flight before the first store
      const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q);
      constexpr int kQIt = NR * 16 / kSoft;
      uint4 v[kQIt];
#pragma unroll
      for (int u = 0; u < kQIt; ++u) {
        const int e = tid + u * kSoft;
        const int row = e >> 4;
        v[u] = make_uint4(0, 0, 0, 0);
        if (row < p.R) {
          const int t = row / group;
          const int hq = g.hkv * group + row % group;
          v[u] = __ldg(reinterpret_cast<const uint4 *>(qb + (((size_t)g.b * p.T + t) * p.Hq + hq) * D) + (e & 15));
        }
      }
#pragma unroll
      for (int u = 0; u < kQIt; ++u) {
        const int e = tid + u * kSoft;
        const int row = e >> 4, ch = e & 15;
        *reinterpret_cast<uint4 *>(sQ + (ch >> 3) * (NR * 128) + row * 128 + (((ch & 7) ^ (row & 7)) << 4)) = v[u];
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    named_bar_arrive(kBarQ, kSoft + 32);

    // ---- draft visibility, when this part holds draft keys: per draft key
    // dk, the packed rows r = t * group + h of the tokens t that see it.  Up to
    // 32 rows it is built at once, while the part's first tiles are still on
    // their way (chain -1%, sparse attention -3%); the 64-row instance, whose
    // hot loop has no registers to spare, loads the parents now and builds the
    // masks before the first draft tile ----
    DraftPre dpre{-1, -1, 0ull, 0ull};
    const bool has_draft = lt1 * TK > g.n_prefix;
    if (warp == 0 && has_draft) dpre = draft_prefetch(p, g.b);
    bool masks_ready = false;
    auto build_masks = [&]() {
      if (warp == 0) {
        uint64_t lo, hi;
        draft_rows(p, dpre, lo, hi);
        if (lane < p.T) rowmask[lane] = lo;
        if (lane + 32 < p.T) rowmask[lane + 32] = hi;
      }
      named_bar_sync(kBarSoft, kSoft);
      if (tid < p.T) {
        const uint64_t gbits = group >= 64 ? ~0ull : ((1ull << group) - 1);
        uint64_t kmask = 0;
        for (int t = 0; t < p.T; ++t)
          if ((rowmask[t] >> tid) & 1ull) kmask |= gbits << (t * group);
        keymask[tid] = kmask;
      }
      named_bar_sync(kBarSoft, kSoft);
      masks_ready = true;
    };
    if (NR <= 32 && has_draft) build_masks();

    float mu[NR];  // reference max per row, log2 units
#pragma unroll
    for (int r = 0; r < NR; ++r) mu[r] = -INFINITY;
    // (kRegL) sums over this thread's keys of P (the fp32 weights, which the
    // bf16 hi + lo parts the PV MMA multiplies carry to ~2^-16)
    float lsum[kRegL ? NR : 1];
#pragma unroll
    for (int r = 0; r < (kRegL ? NR : 1); ++r) lsum[r] = 0.f;

    for (int lt = lt0; lt < lt1; ++lt, ++it, ++jt) {
      const int b = jt & 1;
      const int st = it % NS;
      const uint32_t tS = tO + (2 + b) * NC;
      const int key = lt * TK + tid;
      const bool masked = lt * TK + TK > g.n_prefix;
      if (NR > 32 && masked && !masks_ready) build_masks();
      uint64_t km = ~0ull;  // rows that see this key
      if (masked) {
        if (key >= g.nkeys) km = 0;
        else if (key >= g.n_prefix) km = keymask[key - g.n_prefix];
      }
      wait_ok(s_full + b, (uint32_t)(jt >> 1) & 1u);
      // PV of tile jt-2 (same o_done barrier): waiting for every PV in order,
      // two tiles late, keeps each barrier at most one phase ahead of its waiter
      if (jt >= 2) wait_ok(o_done + b, (uint32_t)((jt - 2) >> 1) & 1u);
      tc_fence_after();
      float x[NR];  // raw scores of this key, -inf where the row does not see it
      auto load_scores = [&]() {
        tmem_ld_f<NR>(tS, x);
        if (masked) {
#pragma unroll
          for (int r = 0; r < NR; ++r)
            if (!((km >> r) & 1ull)) x[r] = -INFINITY;
        }
      };
      load_scores();
      if (lt == lt0) {
        // first tile of this part: the scores of key 0 are the reference; the
        // vote below moves it to the exact maxima only when some score is more
        // than 2^8 above it (or key 0 is hidden from a row)
        if (tid == 0) {
#pragma unroll
          for (int r = 0; r < NR; ++r) reinterpret_cast<float *>(red)[r] = x[r] * cl2;
        }
        named_bar_sync(kBarRed, kSoft);
#pragma unroll
        for (int r = 0; r < NR; r += 4) {
          const float4 m4 = reinterpret_cast<const float4 *>(red)[r >> 2];
          mu[r] = m4.x;
          mu[r + 1] = m4.y;
          mu[r + 2] = m4.z;
          mu[r + 3] = m4.w;
        }
      }
      float dmax = -INFINITY;  // (NaN where a row has seen nothing yet: ignored by fmaxf)
#pragma unroll
      for (int r = 0; r < NR; ++r) dmax = fmaxf(dmax, fmaf(x[r], cl2, -mu[r]));
      if (bar_red_or(kBarRed, kSoft, dmax > 8.f)) {
        // some score passed its reference by more than 2^8: move the references
        // to the exact row maxima seen so far
        WarpScatterMax<NR, 16>::run(x, lane);
        if constexpr (NR >= 32) {
#pragma unroll
          for (int j = 0; j < NR / 32; ++j) reinterpret_cast<float *>(red)[(j + (NR / 32) * lane) * 4 + warp] = x[j];
        } else {
          if ((lane & (32 / NR - 1)) == 0) reinterpret_cast<float *>(red)[(lane / (32 / NR)) * 4 + warp] = x[0];
        }
        named_bar_sync(kBarRed, kSoft);
        float *alpha = x;  // the scores are reloaded below
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const float4 m4 = red[r];
          const float mnew = fmaxf(mu[r], fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w)) * cl2);
          alpha[r] = mu[r] == -INFINITY ? 0.f : ex2_approx(mu[r] - mnew);
          mu[r] = mnew;
        }
        if constexpr (kRegL) {
#pragma unroll
          for (int r = 0; r < NR; ++r) lsum[r] *= alpha[r];
        }
        if (lt != lt0) {
          wait_ok(o_done + (b ^ 1), (uint32_t)((jt - 1) >> 1) & 1u);  // O and l hold every PV up to tile jt-1
          tc_fence_after();
          tmem_scale_cols<NR>(tO, x);
          tmem_scale_cols<NR>(tO + NR, x);
          if constexpr (!kRegL) {
            tmem_scale_cols<NR>(tL, x);
            tmem_scale_cols<NR>(tL + NR, x);
          }
          tmem_st_wait();
        }
        load_scores();
      }
      // P^T row of this key over the K tile of the stage (the S MMA is done with
      // it): chunk cc of the hi part, and of the lo part NR/8 chunks further
      // (64 rows: in the second swizzle atom, 16 KB further)
      uint8_t *pk = stages + st * SM::kStageBytes;
      const int sw = tid & 7;
      auto put_p = [&](int cc, const uint32_t (&h)[4], const uint32_t (&l)[4]) {
        *reinterpret_cast<uint4 *>(pk + tid * 128 + ((cc ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
        if constexpr (NR <= 32)
          *reinterpret_cast<uint4 *>(pk + tid * 128 + (((cc + NR / 8) ^ sw) << 4)) = make_uint4(l[0], l[1], l[2], l[3]);
        else
          *reinterpret_cast<uint4 *>(pk + TK * 128 + tid * 128 + ((cc ^ sw) << 4)) = make_uint4(l[0], l[1], l[2], l[3]);
      };
      if (masked) {
#pragma unroll
        for (int cc = 0; cc < NR / 8; ++cc) {
          uint32_t h[4], l[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = 8 * cc + 2 * q;
            // a row that has seen no key yet has mu = -inf and only -inf scores: P = 0
            const float2 e = fma2(make_float2(x[r], x[r + 1]), make_float2(cl2, cl2),
                                  make_float2(mu[r] == -INFINITY ? 0.f : -mu[r],
                                              mu[r + 1] == -INFINITY ? 0.f : -mu[r + 1]));
            const float a = ex2_approx(e.x), bq = ex2_approx(e.y);
            split_bf16x2(a, bq, h[q], l[q]);
            if constexpr (kRegL) {
              const float2 s2 = add2(make_float2(lsum[r], lsum[r + 1]), make_float2(a, bq));
              lsum[r] = s2.x;
              lsum[r + 1] = s2.y;
            }
          }
          put_p(cc, h, l);
        }
        if (use_tma && key >= g.nkeys) {
          // rows past the segment end: TMA brought whatever follows; zero V so 0 * V stays 0
          wait_ok(full + st, (uint32_t)(it / NS) & 1u);
          uint8_t *vt = pk + Geo::kTileBytes;
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) *reinterpret_cast<uint4 *>(vt + swz<TK>(tid, ch)) = make_uint4(0, 0, 0, 0);
        }
      } else {
        // every row sees every key of a prefix tile, so mu is finite here
#pragma unroll
        for (int cc = 0; cc < NR / 8; ++cc) {
          uint32_t h[4], l[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = 8 * cc + 2 * q;
            const float2 e = fma2(make_float2(x[r], x[r + 1]), make_float2(cl2, cl2), make_float2(-mu[r], -mu[r + 1]));
            const float a = ex2_approx(e.x), bq = ex2_approx(e.y);
            split_bf16x2(a, bq, h[q], l[q]);
            if constexpr (kRegL) {
              const float2 s2 = add2(make_float2(lsum[r], lsum[r + 1]), make_float2(a, bq));
              lsum[r] = s2.x;
              lsum[r + 1] = s2.y;
            }
          }
          put_p(cc, h, l);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full + b);
    }

    // ---- epilogue: column d = tid of O / l for every row of this segment part ----
    if (jt >= 2) wait_ok(o_done + (jt & 1), (uint32_t)((jt - 2) >> 1) & 1u);
    wait_ok(o_done + ((jt - 1) & 1), (uint32_t)((jt - 1) >> 1) & 1u);
    tc_fence_after();
    constexpr int CH = NR < 32 ? NR : 32;  // columns per TMEM load
    const size_t slot = (size_t)(s + c);
    // per-row constants, once: thread r takes row r (l is the same on every
    // lane); its l and reference max are picked out of the register arrays by
    // predicated selects, so the rows are done by the threads in parallel
    float my_l = 0.f, my_mu = 0.f;
    if constexpr (kRegL) {
      // l: this thread's key sums, reduce-scattered over the warp (lane l gets
      // row l, or l / 2 for 16 rows), then the four warps' sums of each row
      WarpScatterSum<NR, 16>::run(lsum, lane);
      if ((lane & (32 / NR - 1)) == 0) reinterpret_cast<float *>(red)[(lane / (32 / NR)) * 4 + warp] = lsum[0];
      named_bar_sync(kBarSoft, kSoft);
      if (tid < NR) {
        const float4 l4 = red[tid];
        my_l = (l4.x + l4.y) + (l4.z + l4.w);
      }
#pragma unroll
      for (int j = 0; j < NR; ++j) my_mu = tid == j ? mu[j] : my_mu;
    } else {
#pragma unroll
      for (int h = 0; h < NR / CH; ++h) {
        float lv[CH];
        tmem_ld_hilo<CH>(tL + h * CH, NR, lv);
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          my_l = tid == h * CH + j ? lv[j] : my_l;
          my_mu = tid == h * CH + j ? mu[h * CH + j] : my_mu;
        }
      }
    }
    if (tid < p.R) {
      const int r = tid;
      const int t = r / group;
      const int hq = g.hkv * group + r % group;
      const float lse_nat = my_l > 0.f ? (my_mu + __log2f(my_l)) * kLn2 : -INFINITY;
      row_inv[r] = my_l > 0.f ? __fdividef(1.f, my_l) : 0.f;
      if (ok) {
        if (n_parts == 1)
          p.lse[((size_t)g.b * p.Hq + hq) * p.T + t] = lse_nat;
        else
          p.lse_part[slot * p.rows_pad + r] = lse_nat;
      }
    }
    named_bar_sync(kBarSoft, kSoft);
    // column d = tid of O / l for every row, staged row-major in the Q buffer
    // (free: every MMA of this part has completed) and written by bulk copies
    if (n_parts > 1) {
      constexpr int HR = NR / 2;
      if constexpr (NR <= 32) {
        // fp32 part: thread d stores column d of every row straight from TMEM
        // (a warp writes 128 contiguous bytes of a row)
        float *orow = p.o_part + slot * p.rows_pad * D + tid;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float ov[HR];
          tmem_ld_hilo<HR>(tO + half * HR, NR, ov);
          if (ok) {
#pragma unroll
            for (int j = 0; j < HR; j += 4) {
              const float4 inv4 = *reinterpret_cast<const float4 *>(row_inv + half * HR + j);
              orow[(half * HR + j + 0) * D] = ov[j] * inv4.x;
              orow[(half * HR + j + 1) * D] = ov[j + 1] * inv4.y;
              orow[(half * HR + j + 2) * D] = ov[j + 2] * inv4.z;
              orow[(half * HR + j + 3) * D] = ov[j + 3] * inv4.w;
            }
          }
        }
        // publish the part (always, also after a failed wait, so the counters
        // return to zero): the block barrier orders every thread's row and lse
        // stores before thread 0's release increment, which is cumulative
        named_bar_sync(kBarSoft, kSoft);
        if (tid == 0 && c != p.test_drop_part)
          red_release_inc_gpu(reinterpret_cast<unsigned *>(&p.merge_cnt[s].x), 2u * n_parts - 1u);
      } else {
        // 64 rows (registers are short): rows staged row-major in the Q buffer,
        // two halves of NR/2 rows written by bulk copies
        float *stage_f = reinterpret_cast<float *>(sQ);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float ov[HR];
          tmem_ld_hilo<HR>(tO + half * HR, NR, ov);
#pragma unroll
          for (int j = 0; j < HR; j += 4) {
            const float4 inv4 = *reinterpret_cast<const float4 *>(row_inv + half * HR + j);
            stage_f[(j + 0) * D + tid] = ov[j] * inv4.x;
            stage_f[(j + 1) * D + tid] = ov[j + 1] * inv4.y;
            stage_f[(j + 2) * D + tid] = ov[j + 2] * inv4.z;
            stage_f[(j + 3) * D + tid] = ov[j + 3] * inv4.w;
          }
          fence_proxy_async_smem();
          named_bar_sync(kBarSoft, kSoft);
          if (tid == 0 && ok) {
            bulk_store_s2g(p.o_part + (slot * p.rows_pad + half * HR) * D, stage_f, (uint32_t)(HR * D * 4));
            bulk_commit();
            bulk_wait_read_all();
          }
          named_bar_sync(kBarSoft, kSoft);
        }
        // publish (always): the block barrier orders every thread's lse stores
        // before thread 0's release, which follows the landing of the bulk rows
        named_bar_sync(kBarSoft, kSoft);
        if (tid == 0) {
          bulk_wait_all();
          if (c != p.test_drop_part)
            red_release_inc_gpu(reinterpret_cast<unsigned *>(&p.merge_cnt[s].x), 2u * n_parts - 1u);
        }
      }
      if (n_split < 2) {
        ms[n_split] = s;
        mslot[n_split] = s + first_cta;
        mnp[n_split] = n_parts;
        mpart[n_split] = c - first_cta;
        ++n_split;
      }
    } else {
      // final bf16 rows: the group rows of one draft token are contiguous in out
      __nv_bfloat16 *stage_b = reinterpret_cast<__nv_bfloat16 *>(sQ);
#pragma unroll
      for (int h = 0; h < NR / CH; ++h) {
        float ov[CH];
        tmem_ld_hilo<CH>(tO + h * CH, NR, ov);
#pragma unroll
        for (int j = 0; j < CH; j += 4) {
          const float4 inv4 = *reinterpret_cast<const float4 *>(row_inv + h * CH + j);
          stage_b[(h * CH + j + 0) * D + tid] = __float2bfloat16_rn(ov[j] * inv4.x);
          stage_b[(h * CH + j + 1) * D + tid] = __float2bfloat16_rn(ov[j + 1] * inv4.y);
          stage_b[(h * CH + j + 2) * D + tid] = __float2bfloat16_rn(ov[j + 2] * inv4.z);
          stage_b[(h * CH + j + 3) * D + tid] = __float2bfloat16_rn(ov[j + 3] * inv4.w);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(kBarSoft, kSoft);
      if (ok && tid < p.T) {
        const int t = tid;
        __nv_bfloat16 *dst =
            static_cast<__nv_bfloat16 *>(p.out) + (((size_t)g.b * p.T + t) * p.Hq + g.hkv * group) * D;
        const __nv_bfloat16 *src = stage_b + (size_t)t * group * D;
        if (p.out_align16) {
          bulk_store_s2g(dst, src, (uint32_t)(group * D * 2));
          bulk_commit();
          bulk_wait_read_all();
        } else {
          for (int e = 0; e < group * D; ++e) dst[e] = src[e];
        }
      }
      named_bar_sync(kBarSoft, kSoft);
    }
  }
  // the output and part rows written by bulk copies have landed
  bulk_wait_all();

  // ---- merge of the split segments: once every part of a segment has
  // arrived, each of its CTAs merges an equal share of its rows ----
  volatile int *merge_ok = abort_flag + 1;
  for (int k = 0; k < n_split; ++k) {
    const int s = ms[k], np = mnp[k];
    if (tid == 0) *merge_ok = wait_parts_arrived(p, s, np) ? 1 : 0;
    named_bar_sync(kBarSoft, kSoft);  // thread 0's acquire, then the barrier, orders the reads below
    if (*merge_ok) {
      const int r0 = mpart[k] * p.R / np, r1 = (mpart[k] + 1) * p.R / np;
      if (np <= 4)
        merge_rows_warp<8, 4>(p, s / p.Hkv, s % p.Hkv, 0, mslot[k], np, r0, r1, warp, 4, lane);
      else
        merge_rows_warp<32, 24>(p, s / p.Hkv, s % p.Hkv, 0, mslot[k], np, r0, r1, warp, 4, lane);
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
template <int NR>
static size_t tck_smem_bytes(const AttnParams &p) {
  return 1024 + (size_t)TkSmem<NR>::kRopeOff + (size_t)rope_table_bytes(p) + (size_t)(p.S + 1) * 4;
}

// A kernel instance with the rotary embedding and one without: code that never
// runs still costs the hot loop registers and schedule.

size_t attn_tck_smem_required(const AttnParams &p) {
  return p.rows_pad <= 16 ? tck_smem_bytes<16>(p) : p.rows_pad <= 32 ? tck_smem_bytes<32>(p) : tck_smem_bytes<64>(p);
}

template <int NR, bool kTma>
static cudaError_t launch_tck_t(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                                cudaStream_t stream) {
  const size_t smem = tck_smem_bytes<NR>(p);
  auto kern = p.positions != nullptr ? verify_attn_tck_kernel<NR, kTma, true> : verify_attn_tck_kernel<NR, kTma, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // cooperative: every CTA is resident, so the wait for a segment's parts ends
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(TkCfg<NR, kTma>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tmk, tmv);
}

cudaError_t launch_attention_tck(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                                 cudaStream_t stream) {
  const bool tma = p.tma_box > 0;
  if (p.rows_pad <= 16)
    return tma ? launch_tck_t<16, true>(p, tmk, tmv, grid, stream) : launch_tck_t<16, false>(p, tmk, tmv, grid, stream);
  if (p.rows_pad <= 32)
    return tma ? launch_tck_t<32, true>(p, tmk, tmv, grid, stream) : launch_tck_t<32, false>(p, tmk, tmv, grid, stream);
  return tma ? launch_tck_t<64, true>(p, tmk, tmv, grid, stream) : launch_tck_t<64, false>(p, tmk, tmv, grid, stream);
}

}  // namespace va
