// Verification attention kernels (LongSpec section 2.C, "Hybrid Tree
// Attention": divide-and-aggregate with an exact log-sum-exp merge).
//
// Work decomposition.  A *segment* is one (sequence b, kv-head, block of up to
// 64 packed query rows).  Its packed rows are the GQA group times the T draft
// tokens (row r = t * group + head-in-group), so every key tile read from HBM
// serves group*T query rows at once.  The segment's key stream is the prefix
// (dense slots 0..L_b-1, paged slots through the block table, or the verify
// index list) followed by the T draft keys at slots L_b..L_b+T-1.  The prefix
// keys are unmasked (the cache part of the split); the draft keys are masked
// by the draft bitmask (the speculative part).  All segments' 64-key tiles are
// laid end to end and the persistent grid takes equal contiguous ranges of
// that list (stream-K), so ragged lengths balance to within one tile.  A
// segment covered by one CTA is finalised in place; a segment cut across CTAs
// leaves one normalised partial (o, lse) per CTA, merged exactly by the
// combine kernel (programmatic dependent launch).
//
// CTA roles.  One producer warp fills a ring of shared-memory stages (one
// 64-key K tile + V tile each, 128-byte-swizzled rows).  Dense caches are read
// with tiled TMA boxes (cp.async.bulk.tensor, 64 tokens x 64 dims per box,
// completing on an mbarrier); paged and sparse caches, whose rows are scattered,
// are gathered with 16-byte cp.async copies that zero-fill rows past the
// segment end.  Both write the same swizzled layout, so the consumers do not
// depend on the layout.  Four consumer warps compute S = Q K^T and
// O += P V on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate),
// run the online softmax with quad shuffles and evaluate the draft bitmask in
// registers.  fp32 inputs use a SIMT FMA consumer instead (no TF32).
//
// Every wait is bounded: on timeout the CTA records VA_ERR_TIMEOUT in the
// workspace status word, stops issuing work, drains its own copies and exits.
#include <cuda.h>
#include <math.h>

#include <type_traits>

#include "va_common.cuh"
#include "va_kernels.h"
#include "va_pipeline.cuh"
#include "va_rope_fused.cuh"

namespace va {

constexpr int kNWC = 4;  // consumer warps
constexpr int kThreads = (kNWC + 1) * 32;

// CPS = CTAs resident per SM: 2 when a consumer warp's state is small enough
// (at most 32 packed rows), so two CTAs interleave their latency-bound warps;
// each then keeps a shorter ring (the SM as a whole still has 128 KB in flight).
template <typename Tin, int D, int CPS = 1>
struct Cfg : StageGeom<Tin, D> {
  using G = StageGeom<Tin, D>;
  static constexpr int kStages = CPS == 2 ? (G::kStageBytes <= 16384 ? 4 : 2) : ((G::kStageBytes <= 16384) ? 8 : 5);
  static constexpr bool kF32 = std::is_same<Tin, float>::value;
  static constexpr int kMergeBytes = kF32 ? 128 * (64 + 2) * 4 : kNWC * 16 * (D * 4 + 8);
};


// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <typename Tin, int D, int RG, int CPS, bool kRope>
__global__ void __launch_bounds__(kThreads, CPS)
    verify_attn_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv) {
  using C = Cfg<Tin, D, CPS>;
  constexpr int NS = C::kStages;
  constexpr int KW = C::kF32 ? 2 : kNWC / RG;  // key-split warps per row group
  constexpr int RPS = C::kF32 ? 64 : 16 * RG;  // packed rows per segment
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle pattern repeats every 1024 bytes: stages start 1024-aligned
  uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  uint8_t *stages = smem;
  float *merge = reinterpret_cast<float *>(smem + NS * C::kStageBytes);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * C::kStageBytes + C::kMergeBytes);
  uint64_t *empty = full + NS;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + NS);
  int *tstart = reinterpret_cast<int *>(empty + NS) + 4;
  // the rotary table of the segment (when positions are given), after the plan
  float2 *rope_tab = reinterpret_cast<float2 *>(tstart + ((p.S + 1 + 3) & ~3));
  constexpr int kBarRope = 2;  // consumer warps only
  const bool use_tma = p.tma_box > 0;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = blockIdx.x;
  const int S = p.S;

  // let the combine kernel get resident early; it waits for our completion
  pdl_launch_dependents();

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full + i, use_tma ? 1 : 32);  // TMA: one expect_tx arrive; cp.async: one per producer lane
      mbar_init(empty + i, kNWC);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // ---- plan: tiles per segment, exclusive scan, this CTA's tile range ----
  const CtaRange cr = plan_cta(p, tstart);
  if (c >= cr.G) return;
  const long long total = cr.total;
  const int G = cr.G;
  const int t0 = cr.t0, t1 = cr.t1, s0 = cr.s0;

  if (warp == kNWC) {
    bool pok = true;
    produce_tiles<Tin, D, NS>(p, &tmk, &tmv, tstart, cr, stages, full, empty, abort_flag, use_tma, pok);
    return;
  }

  // ============================ consumer warps ============================
  const float cl2 = p.scale * kLog2e;  // scores are kept raw; exp2 takes scale*log2(e)
  const int group = p.Hq / p.Hkv;
  int it = 0;
  bool ok = true;
  int rope_b = -1;  // sequence whose rotary table is in shared memory

  for (int s = s0; s < S && tstart[s] < t1; ++s) {
    const Seg g = seg_info(p, s, false);
    const int lt0 = max(tstart[s], t0) - tstart[s];
    const int lt1 = min(tstart[s + 1], t1) - tstart[s];
    const int first_cta = owner_cta(tstart[s], total, G);
    const int n_parts = owner_cta(tstart[s + 1] - 1, total, G) - first_cta + 1;
    if (lt0 == 0 && tid == 0) {
      p.meta[s] = make_int2(s + first_cta, n_parts);
      if (n_parts > 1)  // one entry per split segment
        p.split_list[atomicAdd(p.split_count, 1)] = make_int4(s, s + first_cta, n_parts, 0);
    }
    const bool has_draft = lt1 * kTK > g.n_prefix;
    uint64_t tl = 0, th = 0;
    if (has_draft && p.parent != nullptr) warp_tree_rows(p, g.b, tl, th);
    if (kRope && g.b != rope_b) {
      // rotary table of this sequence's draft tokens, kept while the CTA stays
      // on the sequence (the previous segment's readers are past the barrier first)
      named_bar_sync(kBarRope, kNWC * 32);
      rope_build_table(p, g.b, rope_tab, tid, kNWC * 32);
      named_bar_sync(kBarRope, kNWC * 32);
      rope_b = g.b;
    }
    // the draft keys of tile lt, rotated in place by the consumer warps together
    // before any of them reads the tile
    auto rotate_draft = [&](int lt, int st) {
      if (!kRope || lt * kTK + kTK <= g.n_prefix) return;
      named_bar_sync(kBarRope, kNWC * 32);
      const int r0 = max(0, g.n_prefix - lt * kTK), r1 = min(kTK, g.nkeys - lt * kTK);
      rope_rotate_tile_rows<Tin, D, kTK>(stages + st * C::kStageBytes, r0, r1, lt * kTK + r0 - g.n_prefix, rope_tab,
                                         tid, kNWC * 32);
      named_bar_sync(kBarRope, kNWC * 32);
    };

    if constexpr (!C::kF32) {
      // ------------------------- bf16 tensor-core path -------------------------
      const int rg = warp / KW;
      const int kw = warp % KW;
      constexpr int NK = kTK / KW;  // keys per warp per tile
      constexpr int NT = NK / 8;
      const int gq = lane >> 2, tq = lane & 3;
      // this thread's two rows (gq, gq+8 of the warp's 16-row group)
      int rr[2], trow[2];
      bool rvalid[2];
      uint64_t rmask[2] = {0, 0};
      uint32_t qa[D / 16][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        rr[h] = g.rb * RPS + rg * 16 + gq + 8 * h;
        rvalid[h] = rr[h] < p.R;
        trow[h] = rvalid[h] ? rr[h] / group : 0;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint64_t m = has_draft ? draft_row(p, g.b, trow[h], tl, th) : 0ull;
        rmask[h] = m;
      }
      {
        const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q);
        const uint32_t *qrow[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int hq = g.hkv * group + (rvalid[h] ? rr[h] % group : 0);
          qrow[h] = reinterpret_cast<const uint32_t *>(qb + (((size_t)g.b * p.T + trow[h]) * p.Hq + hq) * D);
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          qa[ks][0] = rvalid[0] ? __ldg(qrow[0] + ks * 8 + tq) : 0u;
          qa[ks][1] = rvalid[1] ? __ldg(qrow[1] + ks * 8 + tq) : 0u;
          qa[ks][2] = rvalid[0] ? __ldg(qrow[0] + ks * 8 + 4 + tq) : 0u;
          qa[ks][3] = rvalid[1] ? __ldg(qrow[1] + ks * 8 + 4 + tq) : 0u;
        }
        if constexpr (kRope) {
          // each fragment register holds columns e, e+1 of one row; its partners
          // e + D/2, e+1 + D/2 sit in the fragment D/32 k-steps further
#pragma unroll
          for (int ks = 0; ks < D / 32; ++ks)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int h = j & 1;
              const int e = ks * 16 + (j >> 1) * 8 + 2 * tq;
              const float2 *cs = rope_tab + trow[h] * (D / 2) + e;
              const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qa[ks][j]));
              const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qa[ks + D / 32][j]));
              qa[ks][j] = pack_bf16(x.x * cs[0].x - y.x * cs[0].y, x.y * cs[1].x - y.y * cs[1].y);
              qa[ks + D / 32][j] = pack_bf16(y.x * cs[0].x + x.x * cs[0].y, y.y * cs[1].x + x.y * cs[1].y);
            }
        }
      }
      float o[D / 8][4];
#pragma unroll
      for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      float mrow[2] = {-INFINITY, -INFINITY};
      float lrow[2] = {0.f, 0.f};

      for (int lt = lt0; lt < lt1; ++lt, ++it) {
        const int st = it % NS;
        const uint32_t ph = (uint32_t)(it / NS) & 1u;
        role_wait(full + st, ph, ok, abort_flag, p.wait_ns, p.status);
        rotate_draft(lt, st);
        if (ok) {
          const uint32_t ks_addr = smem_u32(stages + st * C::kStageBytes);
          const uint32_t vs_addr = ks_addr + C::kTileBytes;
          const int kb = kw * NK;
          if (use_tma && lt * kTK + kTK > g.nkeys) {
            // TMA brought whole 64-token boxes: V rows past the segment end may hold
            // any bytes of the cache, so zero them (P is exactly 0 there, but 0*NaN is not)
            uint8_t *vt = stages + st * C::kStageBytes + C::kTileBytes;
            for (int e = lane; e < NK * C::kChunks; e += 32) {
              const int r = kb + e / C::kChunks;
              if (lt * kTK + r >= g.nkeys) *reinterpret_cast<uint4 *>(vt + swz(r, e % C::kChunks)) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          float sacc[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
          for (int j = 0; j < D / 32; ++j) {
            uint32_t bf[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              ldsm_x4(ks_addr + swz(kb + nt * 8 + (lane & 7), 4 * j + (lane >> 3)), bf[nt][0], bf[nt][1], bf[nt][2],
                      bf[nt][3]);
            // independent accumulators back to back; the dependent k-step follows
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16(sacc[nt], qa[2 * j], bf[nt][0], bf[nt][1]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16(sacc[nt], qa[2 * j + 1], bf[nt][2], bf[nt][3]);
          }
          // mask: keys past the segment end, and draft keys the row may not see
          const int tile_k = lt * kTK + kb;
          if (lt * kTK + kTK > g.n_prefix) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int key = tile_k + nt * 8 + 2 * tq + (e & 1);
                bool vis = key < g.nkeys;
                if (vis && key >= g.n_prefix) vis = (rmask[e >> 1] >> (key - g.n_prefix)) & 1ull;
                if (!vis) sacc[nt][e] = -INFINITY;
              }
            }
          }
          // online softmax (scores raw; exponent base 2 with scale folded in)
          float mx[2] = {mrow[0], mrow[1]};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mx[0] = fmaxf(mx[0], fmaxf(sacc[nt][0], sacc[nt][1]));
            mx[1] = fmaxf(mx[1], fmaxf(sacc[nt][2], sacc[nt][3]));
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
          }
          float alpha[2], mu[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            alpha[h] = (mx[h] == -INFINITY) ? 1.f : exp2f((mrow[h] - mx[h]) * cl2);
            mu[h] = (mx[h] == -INFINITY) ? 0.f : mx[h] * cl2;
            mrow[h] = mx[h];
          }
          float ls[2] = {0.f, 0.f};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float pv = ex2_approx(fmaf(sacc[nt][e], cl2, -mu[e >> 1]));
              sacc[nt][e] = pv;
              ls[e >> 1] += pv;
            }
          }
          lrow[0] = lrow[0] * alpha[0] + ls[0];
          lrow[1] = lrow[1] * alpha[1] + ls[1];
#pragma unroll
          for (int i = 0; i < D / 8; ++i) {
            o[i][0] *= alpha[0];
            o[i][1] *= alpha[0];
            o[i][2] *= alpha[1];
            o[i][3] *= alpha[1];
          }
          // O += P V with P split into bf16 hi + lo parts, so ~16 bits of every
          // weight survive: one bf16 P alone keeps a weight only to 2^-8 of
          // itself, which shows in the output when a few keys carry a row's
          // weight (attention sinks, or a draft tile where few keys are visible).
          constexpr bool exact_p = true;
#pragma unroll
          for (int kk = 0; kk < NK / 16; ++kk) {
            uint32_t a[4], al[4];
            split_bf16x2(sacc[2 * kk][0], sacc[2 * kk][1], a[0], al[0]);
            split_bf16x2(sacc[2 * kk][2], sacc[2 * kk][3], a[1], al[1]);
            split_bf16x2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1], a[2], al[2]);
            split_bf16x2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3], a[3], al[3]);
#pragma unroll
            for (int dh = 0; dh < D / 64; ++dh) {  // 4 x 16 columns of d per batch
              uint32_t bv[4][4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int dn = dh * 4 + i;
                ldsm_x4_t(vs_addr + swz(kb + 16 * kk + 8 * ((lane >> 3) & 1) + (lane & 7), 2 * dn + (lane >> 4)),
                          bv[i][0], bv[i][1], bv[i][2], bv[i][3]);
              }
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                mma_bf16(o[2 * (dh * 4 + i)], a, bv[i][0], bv[i][1]);
                mma_bf16(o[2 * (dh * 4 + i) + 1], a, bv[i][2], bv[i][3]);
              }
              if (exact_p) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  mma_bf16(o[2 * (dh * 4 + i)], al, bv[i][0], bv[i][1]);
                  mma_bf16(o[2 * (dh * 4 + i) + 1], al, bv[i][2], bv[i][3]);
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + st);
      }
      // ---- per-warp state -> shared memory ----
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
        lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
      }
      float *om = merge + (size_t)warp * 16 * D;
      float *ml = merge + (size_t)kNWC * 16 * D + warp * 32;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        *reinterpret_cast<float2 *>(om + gq * D + i * 8 + 2 * tq) = make_float2(o[i][0], o[i][1]);
        *reinterpret_cast<float2 *>(om + (gq + 8) * D + i * 8 + 2 * tq) = make_float2(o[i][2], o[i][3]);
      }
      if (tq == 0) {
        ml[2 * gq] = mrow[0];
        ml[2 * gq + 1] = lrow[0];
        ml[2 * (gq + 8)] = mrow[1];
        ml[2 * (gq + 8) + 1] = lrow[1];
      }
      named_bar_sync(1, kNWC * 32);
      // ---- merge the KW key-split warps of each row group; write out ----
      const int ctid = tid;  // 0..127
      constexpr int CH = 4;  // elements per thread-step
      for (int e = ctid * CH; e < RPS * D; e += kNWC * 32 * CH) {
        const int row = e / D;
        const int d = e % D;
        const int rgi = row / 16, r16 = row % 16;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < KW; ++w) {
          const float *mlw = merge + (size_t)kNWC * 16 * D + (rgi * KW + w) * 32;
          M = fmaxf(M, mlw[2 * r16]);
        }
        float Lsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < KW; ++w) {
          const int ww = rgi * KW + w;
          const float *mlw = merge + (size_t)kNWC * 16 * D + ww * 32;
          const float mw = mlw[2 * r16];
          const float sc = (M == -INFINITY || mw == -INFINITY) ? 0.f : exp2f((mw - M) * cl2);
          Lsum += sc * mlw[2 * r16 + 1];
          const float4 ov = *reinterpret_cast<const float4 *>(merge + (size_t)ww * 16 * D + r16 * D + d);
          acc.x += sc * ov.x;
          acc.y += sc * ov.y;
          acc.z += sc * ov.z;
          acc.w += sc * ov.w;
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        const float lse_nat = Lsum > 0.f ? (M * cl2 + log2f(Lsum)) * kLn2 : -INFINITY;
        const int rrow = g.rb * RPS + row;
        if (rrow >= p.R || !ok) continue;
        if (n_parts == 1) {
          const int t = rrow / group;
          const int hq = g.hkv * group + rrow % group;
          __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(p.out) + (((size_t)g.b * p.T + t) * p.Hq + hq) * D + d;
          uint2 pk;
          pk.x = pack_bf16(acc.x, acc.y);
          pk.y = pack_bf16(acc.z, acc.w);
          *reinterpret_cast<uint2 *>(ob) = pk;
          if (d == 0) p.lse[((size_t)g.b * p.Hq + hq) * p.T + t] = lse_nat;
        } else {
          const int slot = s + c;
          *reinterpret_cast<float4 *>(p.o_part + ((size_t)slot * p.rows_pad + row) * D + d) = acc;
          if (d == 0) p.lse_part[(size_t)slot * p.rows_pad + row] = lse_nat;
        }
      }
      named_bar_sync(1, kNWC * 32);
    } else {
      // ------------------------------ fp32 SIMT path ------------------------------
      // thread = (row r in 0..63, key half); D == 64
      const int r = tid & 63;
      const int half = tid >> 6;
      const int rrow = g.rb * RPS + r;
      const bool rv = rrow < p.R;
      const int t = rv ? rrow / group : 0;
      const int hq = g.hkv * group + (rv ? rrow % group : 0);
      uint64_t rmask = 0;
      {
        // every lane of the warp computes its own row's visibility (shuffles need the full warp)
        const uint64_t m = has_draft ? draft_row(p, g.b, t, tl, th) : 0ull;
        rmask = m;
      }
      float qv[64];
      {
        const float4 *qr = reinterpret_cast<const float4 *>(static_cast<const float *>(p.q) +
                                                            (((size_t)g.b * p.T + t) * p.Hq + hq) * 64);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 v4 = rv ? __ldg(qr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          qv[4 * i] = v4.x;
          qv[4 * i + 1] = v4.y;
          qv[4 * i + 2] = v4.z;
          qv[4 * i + 3] = v4.w;
        }
        if constexpr (kRope) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float2 cs = rope_tab[t * 32 + i];
            const float x = qv[i], y = qv[i + 32];
            qv[i] = x * cs.x - y * cs.y;
            qv[i + 32] = y * cs.x + x * cs.y;
          }
        }
      }
      float o[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) o[i] = 0.f;
      float m = -INFINITY, l = 0.f;
      for (int lt = lt0; lt < lt1; ++lt, ++it) {
        const int st = it % NS;
        const uint32_t ph = (uint32_t)(it / NS) & 1u;
        role_wait(full + st, ph, ok, abort_flag, p.wait_ns, p.status);
        rotate_draft(lt, st);
        if (ok) {
          const uint8_t *kt = stages + st * C::kStageBytes;
          uint8_t *vt = stages + st * C::kStageBytes + C::kTileBytes;
          if (use_tma && lt * kTK + kTK > g.nkeys) {
            // zero V rows past the segment end (see the bf16 path); this warp's key half only
            for (int e = lane; e < 32 * C::kChunks; e += 32) {
              const int r = half * 32 + e / C::kChunks;
              if (lt * kTK + r >= g.nkeys) *reinterpret_cast<uint4 *>(vt + swz(r, e % C::kChunks)) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          float sc[32];
#pragma unroll 4
          for (int kk = 0; kk < 32; ++kk) {
            const int kr = half * 32 + kk;
            float a = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float4 k4 = *reinterpret_cast<const float4 *>(kt + swz(kr, i));
              a = fmaf(qv[4 * i], k4.x, a);
              a = fmaf(qv[4 * i + 1], k4.y, a);
              a = fmaf(qv[4 * i + 2], k4.z, a);
              a = fmaf(qv[4 * i + 3], k4.w, a);
            }
            const int key = lt * kTK + half * 32 + kk;
            bool vis = key < g.nkeys;
            if (vis && key >= g.n_prefix) vis = (rmask >> (key - g.n_prefix)) & 1ull;
            sc[kk] = vis ? a : -INFINITY;
          }
          float mx = m;
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) mx = fmaxf(mx, sc[kk]);
          const float alpha = (mx == -INFINITY) ? 1.f : exp2f((m - mx) * cl2);
          const float mu = (mx == -INFINITY) ? 0.f : mx * cl2;
          m = mx;
          float ls = 0.f;
#pragma unroll
          for (int i = 0; i < 64; ++i) o[i] *= alpha;
#pragma unroll 4
          for (int kk = 0; kk < 32; ++kk) {
            const float pv = exp2f(fmaf(sc[kk], cl2, -mu));
            ls += pv;
            const int vrow = half * 32 + kk;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float4 v4 = *reinterpret_cast<const float4 *>(vt + swz(vrow, i));
              o[4 * i] = fmaf(pv, v4.x, o[4 * i]);
              o[4 * i + 1] = fmaf(pv, v4.y, o[4 * i + 1]);
              o[4 * i + 2] = fmaf(pv, v4.z, o[4 * i + 2]);
              o[4 * i + 3] = fmaf(pv, v4.w, o[4 * i + 3]);
            }
          }
          l = l * alpha + ls;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + st);
      }
      // merge the two key halves of each row through shared memory
      float *mine = merge + (size_t)tid * 66;
#pragma unroll
      for (int i = 0; i < 64; ++i) mine[i] = o[i];
      mine[64] = m;
      mine[65] = l;
      named_bar_sync(1, kNWC * 32);
      const float *a0 = merge + (size_t)r * 66;
      const float *a1 = merge + (size_t)(r + 64) * 66;
      const float M = fmaxf(a0[64], a1[64]);
      const float w0 = (M == -INFINITY || a0[64] == -INFINITY) ? 0.f : exp2f((a0[64] - M) * cl2);
      const float w1 = (M == -INFINITY || a1[64] == -INFINITY) ? 0.f : exp2f((a1[64] - M) * cl2);
      const float Lsum = w0 * a0[65] + w1 * a1[65];
      const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
      const float lse_nat = Lsum > 0.f ? (M * cl2 + log2f(Lsum)) * kLn2 : -INFINITY;
      if (rv && ok) {
        if (n_parts == 1) {
          float *ob = static_cast<float *>(p.out) + (((size_t)g.b * p.T + t) * p.Hq + hq) * 64;
          for (int d = half * 32; d < half * 32 + 32; ++d) ob[d] = (w0 * a0[d] + w1 * a1[d]) * inv;
          if (half == 0) p.lse[((size_t)g.b * p.Hq + hq) * p.T + t] = lse_nat;
        } else {
          const int slot = s + c;
          float *op = p.o_part + ((size_t)slot * p.rows_pad + r) * 64;
          for (int d = half * 32; d < half * 32 + 32; ++d) op[d] = (w0 * a0[d] + w1 * a1[d]) * inv;
          if (half == 0) p.lse_part[(size_t)slot * p.rows_pad + r] = lse_nat;
        }
      }
      named_bar_sync(1, kNWC * 32);
    }
  }
}

// ---------------------------------------------------------------------------
// log-sum-exp combine (LongSpec 2.C): out = sum_s exp(lse_s - lse) o_s
// ---------------------------------------------------------------------------
template <typename OutT>
__device__ __forceinline__ void store_out(OutT *dst, float v);
template <>
__device__ __forceinline__ void store_out<float>(float *dst, float v) { *dst = v; }
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16 *dst, float v) {
  *dst = __float2bfloat16_rn(v);
}

// Merge the parts of one row with a block of 128 threads.  Thread (g, c) holds
// the four columns [4c, 4c + 4) of the parts s = g (mod PG), PG = 128 / (D / 4),
// in registers; the first batch of those loads is issued together with the
// loads of the parts' lse, so a merge of up to PG * kCombineBatch parts costs
// one round trip to L2.  The part weights e^(lse_s - M) go to shared memory.
constexpr int kMaxCombineParts = 1024;
constexpr int kCombineBatch = 16;

template <typename OutT>
__device__ __forceinline__ void combine_row(int n_parts, int D, const float *o, size_t o_stride, const float *l,
                                            size_t l_stride, OutT *out, float *lse_out) {
  __shared__ float w[kMaxCombineParts];
  __shared__ float red_m[4], red_s[4];
  __shared__ float4 accs[128];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = D >> 2;     // float4 columns of a row
  const int PG = 128 / q;   // part groups
  const int c = tid % q, g = tid / q;
  float mloc = -INFINITY;
  for (int s = tid; s < n_parts; s += 128) {
    const float ls = __ldg(l + (size_t)s * l_stride);
    w[s] = ls;
    mloc = fmaxf(mloc, ls);
  }
  float4 v[kCombineBatch];
#pragma unroll
  for (int j = 0; j < kCombineBatch; ++j) {
    const int s = g + j * PG;
    v[j] = s < n_parts ? __ldg(reinterpret_cast<const float4 *>(o + (size_t)s * o_stride) + c)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int off = 16; off > 0; off >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, off));
  if (lane == 0) red_m[warp] = mloc;
  __syncthreads();
  const float M = fmaxf(fmaxf(red_m[0], red_m[1]), fmaxf(red_m[2], red_m[3]));
  float sloc = 0.f;
  for (int s = tid; s < n_parts; s += 128) {
    const float ls = w[s];
    const float e = (M == -INFINITY || ls == -INFINITY) ? 0.f : __expf(ls - M);
    w[s] = e;
    sloc += e;
  }
  for (int off = 16; off > 0; off >>= 1) sloc += __shfl_xor_sync(0xffffffffu, sloc, off);
  if (lane == 0) red_s[warp] = sloc;
  __syncthreads();
  const float Lsum = (red_s[0] + red_s[1]) + (red_s[2] + red_s[3]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kCombineBatch; ++j) {
    const int s = g + j * PG;
    const float ws = s < n_parts ? w[s] : 0.f;
    acc.x = fmaf(ws, v[j].x, acc.x);
    acc.y = fmaf(ws, v[j].y, acc.y);
    acc.z = fmaf(ws, v[j].z, acc.z);
    acc.w = fmaf(ws, v[j].w, acc.w);
  }
  for (int base = PG * kCombineBatch; base < n_parts; base += PG * kCombineBatch) {
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) {
      const int s = base + g + j * PG;
      v[j] = s < n_parts ? __ldg(reinterpret_cast<const float4 *>(o + (size_t)s * o_stride) + c)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) {
      const int s = base + g + j * PG;
      const float ws = s < n_parts ? w[s] : 0.f;
      acc.x = fmaf(ws, v[j].x, acc.x);
      acc.y = fmaf(ws, v[j].y, acc.y);
      acc.z = fmaf(ws, v[j].z, acc.z);
      acc.w = fmaf(ws, v[j].w, acc.w);
    }
  }
  accs[tid] = acc;
  __syncthreads();
  if (tid < D) {
    const int cc = tid >> 2, k = tid & 3;
    float r = 0.f;
    for (int gg = 0; gg < PG; ++gg) {
      const float4 a = accs[gg * q + cc];
      r += k == 0 ? a.x : k == 1 ? a.y : k == 2 ? a.z : a.w;
    }
    store_out<OutT>(out + tid, Lsum > 0.f ? r / Lsum : 0.f);
    if (tid == 0 && lse_out != nullptr) *lse_out = Lsum > 0.f ? M + __logf(Lsum) : -INFINITY;
  }
}

// Merge of the segments the attention grid cut over several CTAs (their list
// is in the workspace).  A block of 128 threads holds 128 / (D/4) row slots;
// a slot of D/4 lanes merges one packed row, each lane four columns.  The lse
// and output loads of up to kSplitBatch parts are issued together and merged
// with a running maximum (exact for any number of parts), so a row costs one
// round trip per batch.  Blocks stride over (listed segment, row) items; the
// last block to take a ticket resets the list for the next call.
constexpr int kSplitBatch = 24;

template <typename OutT>
__device__ __forceinline__ void merge_split_row(const AttnParams &p, int4 e, int row, int li) {
  const int s = e.x, P = e.z;
  const int D = p.D;
  const int rb = s % p.NRB;
  const int hkv = (s / p.NRB) % p.Hkv;
  const int b = s / (p.NRB * p.Hkv);
  const int rr = rb * p.rows_pad + row;
  const int group = p.Hq / p.Hkv;
  const int t = rr / group;
  const int hq = hkv * group + rr % group;
  const size_t ostride = (size_t)p.rows_pad * D;
  const float *o = p.o_part + ((size_t)e.y * p.rows_pad + row) * D + 4 * li;
  const float *l = p.lse_part + (size_t)e.y * p.rows_pad + row;
  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < P; s0 += kSplitBatch) {
    float ls[kSplitBatch];
    float4 v[kSplitBatch];
#pragma unroll
    for (int j = 0; j < kSplitBatch; ++j) {
      const bool in = s0 + j < P;
      ls[j] = in ? __ldg(l + (size_t)(s0 + j) * p.rows_pad) : -INFINITY;
      v[j] = in ? __ldg(reinterpret_cast<const float4 *>(o + (size_t)(s0 + j) * ostride))
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float m = M;
#pragma unroll
    for (int j = 0; j < kSplitBatch; ++j) m = fmaxf(m, ls[j]);
    if (m == -INFINITY) continue;  // no part so far saw a key
    const float a = M == -INFINITY ? 0.f : __expf(M - m);
    L *= a;
    acc.x *= a;
    acc.y *= a;
    acc.z *= a;
    acc.w *= a;
#pragma unroll
    for (int j = 0; j < kSplitBatch; ++j) {
      const float w = ls[j] == -INFINITY ? 0.f : __expf(ls[j] - m);
      L += w;
      acc.x = fmaf(w, v[j].x, acc.x);
      acc.y = fmaf(w, v[j].y, acc.y);
      acc.z = fmaf(w, v[j].z, acc.z);
      acc.w = fmaf(w, v[j].w, acc.w);
    }
    M = m;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  OutT *out = static_cast<OutT *>(p.out) + (((size_t)b * p.T + t) * p.Hq + hq) * D + 4 * li;
  store_out<OutT>(out + 0, acc.x * inv);
  store_out<OutT>(out + 1, acc.y * inv);
  store_out<OutT>(out + 2, acc.z * inv);
  store_out<OutT>(out + 3, acc.w * inv);
  if (li == 0) p.lse[((size_t)b * p.Hq + hq) * p.T + t] = L > 0.f ? M + __logf(L) : -INFINITY;
}

template <typename OutT>
__global__ void __launch_bounds__(128) combine_segments_kernel(const AttnParams p) {
  __shared__ int s_count;
  const int lpr = p.D / 4;    // lanes per row
  const int spb = 128 / lpr;  // row slots per block
  const int slot = threadIdx.x / lpr, li = threadIdx.x % lpr;
  const long long it0 = (long long)blockIdx.x * spb + slot;
  // wait until every CTA of the attention grid has finished and flushed
  pdl_wait_primary();
  // the first item's list entry is read before the list length is known
  // (the grid never indexes past the list's capacity)
  int4 e0 = p.split_list[it0 / p.rows_pad];
  int ticket = 0;
  if (threadIdx.x == 0) {
    const int c = *reinterpret_cast<volatile int *>(p.split_count);
    s_count = c;
    ticket = atomicAdd(p.split_done, c >= 0 ? 1 : 2);  // taken after the length was read
  }
  __syncthreads();
  const long long items = (long long)s_count * p.rows_pad;
  for (long long it = it0; it < items; it += (long long)gridDim.x * spb) {
    const int4 e = it == it0 ? e0 : p.split_list[it / p.rows_pad];
    const int row = (int)(it % p.rows_pad);
    if ((e.x % p.NRB) * p.rows_pad + row >= p.R) continue;  // padding row of the last row block
    merge_split_row<OutT>(p, e, row, li);
  }
  // every block took its ticket after reading the length: the last one resets the list
  if (threadIdx.x == 0 && ticket == (int)gridDim.x - 1) {
    *p.split_count = 0;
    *p.split_done = 0;
  }
}

template <typename OutT>
__global__ void __launch_bounds__(128) combine_generic_kernel(int n_rows, int n_parts, int D, const float *o_parts,
                                                              const float *lse_parts, OutT *out, float *lse) {
  const int r = blockIdx.x;
  if (r >= n_rows) return;
  combine_row<OutT>(n_parts, D, o_parts + (size_t)r * D, (size_t)n_rows * D, lse_parts + r, (size_t)n_rows,
                    out + (size_t)r * D, lse != nullptr ? lse + r : nullptr);
}

// ---------------------------------------------------------------------------
// host-side launch helpers
// ---------------------------------------------------------------------------
template <typename Tin, int D, int RG, int CPS>
static size_t attn_smem_bytes(const AttnParams &p) {
  using C = Cfg<Tin, D, CPS>;
  return 1024 + (size_t)C::kStages * C::kStageBytes + C::kMergeBytes + 2 * C::kStages * 8 + 16 +
         (size_t)((p.S + 1 + 3) & ~3) * 4 + (size_t)rope_table_bytes(p);
}

template <typename Tin, int D, int RG, int CPS = 1>
static cudaError_t launch_attn_t(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                                 cudaStream_t stream) {
  const size_t smem = attn_smem_bytes<Tin, D, RG, CPS>(p);
  // instances with and without the rotary embedding (code that never runs
  // still costs the hot loop)
  auto kern = p.positions != nullptr ? verify_attn_kernel<Tin, D, RG, CPS, true> : verify_attn_kernel<Tin, D, RG, CPS, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(p, tmk, tmv);
  return cudaGetLastError();
}

size_t attn_smem_required(const AttnParams &p) {
  if (p.use_tc == 3) return attn_tcp_smem_required(p);
  if (p.use_tc == 1) return attn_tc_smem_required(p);
  if (p.use_tc == 2) return attn_tck_smem_required(p);
  if (p.dtype == VA_DTYPE_FP32) return attn_smem_bytes<float, 64, 4, 1>(p);
  if (p.cps == 2) return p.D == 64 ? attn_smem_bytes<__nv_bfloat16, 64, 2, 2>(p) : attn_smem_bytes<__nv_bfloat16, 128, 2, 2>(p);
  if (p.D == 64) return attn_smem_bytes<__nv_bfloat16, 64, 4, 1>(p);
  return attn_smem_bytes<__nv_bfloat16, 128, 4, 1>(p);
}

cudaError_t launch_attention(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                             cudaStream_t stream) {
  cudaError_t e;
  if (p.use_tc == 1) {
    return launch_attention_tc(p, tmk, tmv, grid, stream);  // merges its split segments itself
  } else if (p.use_tc == 2) {
    return launch_attention_tck(p, tmk, tmv, grid, stream);  // merges its split segments itself
  } else if (p.use_tc == 3) {
    return launch_attention_tcp(p, tmk, tmv, grid, stream);  // merges its split segments itself
  } else if (p.dtype == VA_DTYPE_FP32) {
    e = launch_attn_t<float, 64, 4>(p, tmk, tmv, grid, stream);
  } else if (p.D == 64) {
    e = p.RG == 1 ? launch_attn_t<__nv_bfloat16, 64, 1, 2>(p, tmk, tmv, grid, stream)
        : p.RG == 2 ? launch_attn_t<__nv_bfloat16, 64, 2, 2>(p, tmk, tmv, grid, stream)
                    : launch_attn_t<__nv_bfloat16, 64, 4, 1>(p, tmk, tmv, grid, stream);
  } else {
    e = p.RG == 1 ? launch_attn_t<__nv_bfloat16, 128, 1, 2>(p, tmk, tmv, grid, stream)
        : p.RG == 2 ? launch_attn_t<__nv_bfloat16, 128, 2, 2>(p, tmk, tmv, grid, stream)
                    : launch_attn_t<__nv_bfloat16, 128, 4, 1>(p, tmk, tmv, grid, stream);
  }
  if (e != cudaSuccess) return e;

  // combine, chained by programmatic dependent launch
  // at most one split segment per CTA boundary: min(S, grid) segments of R rows
  const int spb = 128 / (p.D / 4);
  const long long max_items = (long long)min(p.S, grid) * p.rows_pad;
  long long blocks = (max_items + spb - 1) / spb;
  const long long cap = 4ll * (grid < 1 ? 1 : grid);
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(blocks < 1 ? 1 : blocks));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.dtype == VA_DTYPE_FP32)
    e = cudaLaunchKernelEx(&cfg, combine_segments_kernel<float>, p);
  else
    e = cudaLaunchKernelEx(&cfg, combine_segments_kernel<__nv_bfloat16>, p);
  return e;
}

cudaError_t launch_combine_generic(int n_rows, int n_parts, int D, const float *o_parts, const float *lse_parts,
                                   va_dtype out_dtype, void *out, float *lse, cudaStream_t stream) {
  const dim3 grid((unsigned)n_rows);
  if (out_dtype == VA_DTYPE_FP32)
    combine_generic_kernel<float><<<grid, 128, 0, stream>>>(n_rows, n_parts, D, o_parts, lse_parts,
                                                            static_cast<float *>(out), lse);
  else
    combine_generic_kernel<__nv_bfloat16><<<grid, 128, 0, stream>>>(
        n_rows, n_parts, D, o_parts, lse_parts, static_cast<__nv_bfloat16 *>(out), lse);
  return cudaGetLastError();
}

}  // namespace va
