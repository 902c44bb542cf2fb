// Pipeline pieces shared by the verification-attention kernels: the
// stream-K work plan over (sequence, kv-head, row-block) segments, the draft
// visibility rows, key-row addressing for the dense / paged / sparse layouts,
// and the producer warp that fills the shared-memory stage ring with TMA boxes
// (dense) or 16-byte cp.async gathers (paged, sparse).
#pragma once

#include <cuda.h>

#include "va_common.cuh"
#include "va_kernels.h"

namespace va {

constexpr int kTK = 64;  // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Geometry of one stage of the ring: a TK-key K tile and V tile, each split in
// 128-byte columns of TK swizzled rows.
template <typename Tin, int D, int TK = kTK>
struct StageGeom {
  static constexpr int kRowBytes = D * (int)sizeof(Tin);  // 128 or 256
  static constexpr int kChunks = kRowBytes / 16;          // 16-byte chunks per row
  static constexpr int kHalves = kRowBytes / 128;         // 128-byte swizzle columns per row
  static constexpr int kTileBytes = kHalves * TK * 128;   // one TK-key tile of K (or V)
  static constexpr int kStageBytes = 2 * kTileBytes;      // K tile + V tile
};

// Byte offset of 16-byte chunk c of key row r inside a TK-row tile: rows are
// split in 128-byte columns (c / 8) of TK rows each, and inside a column the
// chunk index is XORed with r % 8 -- the TMA 128-byte swizzle, which also makes
// every 8-row ldmatrix conflict-free.
template <int TK = kTK>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)((c >> 3) * (TK * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------------------
// segment geometry
// ---------------------------------------------------------------------------
struct Seg {
  int b, hkv, rb;
  int L;         // committed prefix length of the sequence
  int n_prefix;  // prefix keys of this segment (L, or the verify-set size)
  int nkeys;     // n_prefix + T
};

__device__ __forceinline__ Seg seg_info(const AttnParams &p, int s, bool record) {
  Seg g;
  g.rb = s % p.NRB;
  g.hkv = (s / p.NRB) % p.Hkv;
  g.b = s / (p.NRB * p.Hkv);
  int L = __ldg(p.seqlens + g.b);
  if (L < 0 || L > p.len_cap - p.T) {
    if (record) record_status(p.status, VA_ERR_DEVICE_BOUNDS);
    L = L < 0 ? 0 : p.len_cap - p.T;
  }
  g.L = L;
  if (p.layout == VA_LAYOUT_SPARSE) {
    int n = __ldg(p.n_indices + g.b * p.Hkv + g.hkv);
    if (n < 0 || n > p.max_indices) {
      if (record) record_status(p.status, VA_ERR_DEVICE_BOUNDS);
      n = n < 0 ? 0 : p.max_indices;
    }
    g.n_prefix = n;
  } else {
    g.n_prefix = L;
  }
  g.nkeys = g.n_prefix + p.T;
  return g;
}

// Exclusive scan of a[0..n) in place by one full warp; a[n] receives the total.
__device__ __forceinline__ void warp_scan_inplace(int *a, int n) {
  const int lane = threadIdx.x & 31;
  const int per = (n + 31) / 32;
  const int lo = lane * per;
  const int hi = min(n, lo + per);
  int sum = 0;
  for (int i = lo; i < hi; ++i) sum += a[i];
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - sum;
  for (int i = lo; i < hi; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
  if (lane == 31) a[n] = incl;
}

// CTA that owns tile t when `total` tiles are cut into G near-equal ranges
// [c*total/G, (c+1)*total/G).
__device__ __forceinline__ int owner_cta(long long t, long long total, int G) {
  return (int)(((t + 1) * (long long)G - 1) / total);
}

// ---------------------------------------------------------------------------
// draft visibility of one draft token t as a 64-bit row (bit j = draft key j)
// ---------------------------------------------------------------------------
// Ancestor-or-self rows for t = lane and t = lane + 32 from the parents of
// those nodes (p_lo, p_hi; -1 past T), walked by the whole warp with shuffles
// (LongSpec 1.3 / 2.C: a tree node sees its path).
__device__ __forceinline__ void warp_tree_walk(const AttnParams &p, int p_lo, int p_hi, uint64_t &row_lo,
                                               uint64_t &row_hi) {
  const int lane = threadIdx.x & 31;
  const int T = p.T;
  // a parent that breaks -1 <= parent[i] < i ends the path at that node
  if (p_lo < -1 || p_lo >= lane) {
    if (lane < T) record_status(p.status, VA_ERR_DEVICE_BOUNDS);
    p_lo = -1;
  }
  if (p_hi < -1 || p_hi >= lane + 32) {
    if (lane + 32 < T) record_status(p.status, VA_ERR_DEVICE_BOUNDS);
    p_hi = -1;
  }
  int c0 = lane < T ? lane : -1;
  int c1 = lane + 32 < T ? lane + 32 : -1;
  uint64_t r0 = 0, r1 = 0;
  for (int step = 0; step < T; ++step) {
    if (c0 >= 0) r0 |= 1ull << c0;
    if (c1 >= 0) r1 |= 1ull << c1;
    const int a0 = __shfl_sync(0xffffffffu, p_lo, c0 & 31);
    const int b0 = __shfl_sync(0xffffffffu, p_hi, c0 & 31);
    const int a1 = __shfl_sync(0xffffffffu, p_lo, c1 & 31);
    const int b1 = __shfl_sync(0xffffffffu, p_hi, c1 & 31);
    c0 = c0 < 0 ? -1 : (c0 < 32 ? a0 : b0);
    c1 = c1 < 0 ? -1 : (c1 < 32 ? a1 : b1);
    if (!__any_sync(0xffffffffu, (c0 >= 0) || (c1 >= 0))) break;
  }
  row_lo = r0;
  row_hi = r1;
}

__device__ __forceinline__ void warp_tree_rows(const AttnParams &p, int b, uint64_t &row_lo, uint64_t &row_hi) {
  const int lane = threadIdx.x & 31;
  const int32_t *par = p.parent + (size_t)b * p.T;
  const int p_lo = lane < p.T ? __ldg(par + lane) : -1;
  const int p_hi = lane + 32 < p.T ? __ldg(par + lane + 32) : -1;
  warp_tree_walk(p, p_lo, p_hi, row_lo, row_hi);
}

// The draft structure of sequence b for rows t = lane and lane + 32, loaded
// ahead of use (parents, or the rows of an explicit bitmask).
struct DraftPre {
  int p_lo, p_hi;
  uint64_t w_lo, w_hi;
};

__device__ __forceinline__ DraftPre draft_prefetch(const AttnParams &p, int b) {
  const int lane = threadIdx.x & 31;
  DraftPre d;
  d.p_lo = d.p_hi = -1;
  d.w_lo = d.w_hi = 0;
  if (p.parent != nullptr) {
    const int32_t *par = p.parent + (size_t)b * p.T;
    if (lane < p.T) d.p_lo = __ldg(par + lane);
    if (lane + 32 < p.T) d.p_hi = __ldg(par + lane + 32);
  } else if (p.mask != nullptr) {
    const uint32_t *w = p.mask + (size_t)b * p.T * p.mask_words;
    if (lane < p.T) {
      d.w_lo = __ldg(w + (size_t)lane * p.mask_words);
      if (p.mask_words > 1) d.w_lo |= (uint64_t)__ldg(w + (size_t)lane * p.mask_words + 1) << 32;
    }
    if (lane + 32 < p.T) {
      d.w_hi = __ldg(w + (size_t)(lane + 32) * p.mask_words);
      if (p.mask_words > 1) d.w_hi |= (uint64_t)__ldg(w + (size_t)(lane + 32) * p.mask_words + 1) << 32;
    }
  }
  return d;
}

// Visibility rows of draft tokens t = lane and lane + 32 (whole warp).
__device__ __forceinline__ void draft_rows(const AttnParams &p, const DraftPre &d, uint64_t &row_lo,
                                           uint64_t &row_hi) {
  const int lane = threadIdx.x & 31;
  if (p.parent != nullptr) {
    warp_tree_walk(p, d.p_lo, d.p_hi, row_lo, row_hi);
  } else if (p.mask != nullptr) {
    row_lo = d.w_lo;
    row_hi = d.w_hi;
  } else {  // causal chain
    row_lo = (2ull << lane) - 1;
    row_hi = lane + 32 >= 63 ? ~0ull : ((2ull << (lane + 32)) - 1);
  }
}

// Visibility row of draft token t for sequence b.  Must be called by a full
// warp (the tree walk uses shuffles); tl/th are the warp's tree rows (only
// read when a parent array is given).
__device__ __forceinline__ uint64_t draft_row(const AttnParams &p, int b, int t, uint64_t tl, uint64_t th) {
  if (p.parent != nullptr) {
    const uint64_t a = __shfl_sync(0xffffffffu, tl, t & 31);
    const uint64_t c = __shfl_sync(0xffffffffu, th, t & 31);
    return t < 32 ? a : c;
  }
  if (p.mask != nullptr) {
    const uint32_t *w = p.mask + ((size_t)b * p.T + t) * p.mask_words;
    uint64_t r = __ldg(w);
    if (p.mask_words > 1) r |= (uint64_t)__ldg(w + 1) << 32;
    return r;
  }
  return t >= 63 ? ~0ull : ((2ull << t) - 1);  // causal chain
}

// Visibility of the 64 keys k0 .. k0 + 63 for one row as a word: bit j is set
// when key k0 + j exists (below nkeys) and is a prefix key or a draft key whose
// bit the row's draft mask rmask has.  Built once per tile so that the
// per-key tests are bit tests at fixed positions (a per-key shift by a
// key-dependent amount kept the loop over the scores from being unrolled).
__device__ __forceinline__ uint64_t tile_vis64(int k0, int n_prefix, int nkeys, uint64_t rmask) {
  const int off = n_prefix - k0;  // position of the first draft key in the tile
  uint64_t vis = off >= 64 ? ~0ull : (off <= 0 ? 0ull : (1ull << off) - 1ull);
  if (off < 64) vis |= off >= 0 ? (rmask << off) : (-off >= 64 ? 0ull : rmask >> (-off));
  const int nv = nkeys - k0;  // keys of the tile that exist
  if (nv < 64) vis &= nv <= 0 ? 0ull : (1ull << nv) - 1ull;
  return vis;
}

// ---------------------------------------------------------------------------
// producer: one warp moves K/V rows of each tile with bulk copies
// ---------------------------------------------------------------------------
template <typename Tin, int D>
__device__ __forceinline__ const Tin *key_row(const AttnParams &p, const Seg &g, int k, const Tin *base) {
  // segment-local key k -> cache row
  if (p.layout == VA_LAYOUT_PAGED) {
    const int slot = k;  // logical slot: prefix 0..L-1, draft L..L+T-1
    int page = __ldg(p.page_table + (size_t)g.b * p.max_pages + (slot >> p.page_shift));
    if (page < 0 || page >= p.num_pages) {
      record_status(p.status, VA_ERR_DEVICE_BOUNDS);
      page = 0;
    }
    const size_t row = ((size_t)page << p.page_shift) + (slot & ((1 << p.page_shift) - 1));
    return base + (row * p.Hkv + g.hkv) * D;
  }
  int pos;
  if (p.layout == VA_LAYOUT_SPARSE && k < g.n_prefix) {
    pos = __ldg(p.indices + ((size_t)g.b * p.Hkv + g.hkv) * p.max_indices + k);
    if (pos < 0 || pos >= g.L) {
      record_status(p.status, VA_ERR_DEVICE_BOUNDS);
      pos = 0;
    }
  } else {
    pos = g.L + (k - g.n_prefix);  // dense: n_prefix == L, so pos == k
  }
  return base + (((size_t)g.b * p.len_cap + pos) * p.Hkv + g.hkv) * D;
}


// ---------------------------------------------------------------------------
// the CTA's share of the work list
// ---------------------------------------------------------------------------
struct CtaRange {
  long long total;  // tiles of all segments
  int G;            // CTAs the list is cut over (<= total)
  int t0, t1;       // this CTA's tiles [t0, t1)
  int s0;           // first segment touching t0
};

// Tiles of TK keys per segment, their exclusive scan into tstart[0..S], and
// this CTA's range.  Called by every thread of the block (contains __syncthreads).
template <int TK = kTK>
__device__ __forceinline__ CtaRange plan_cta(const AttnParams &p, int *tstart) {
  for (int s = threadIdx.x; s < p.S; s += blockDim.x) {
    const Seg g = seg_info(p, s, true);
    tstart[s] = (g.nkeys + TK - 1) / TK;
  }
  __syncthreads();
  if ((threadIdx.x >> 5) == 0) warp_scan_inplace(tstart, p.S);
  __syncthreads();
  CtaRange r;
  r.total = tstart[p.S];
  // the list is cut over G <= total CTAs, so every CTA (and every part of a
  // segment) owns at least one tile; surplus CTAs of the grid have no work
  r.G = (int)min((long long)gridDim.x, r.total);
  const int c = blockIdx.x;
  r.t0 = r.t1 = 0;
  r.s0 = 0;
  if (c < r.G) {
    r.t0 = (int)(((long long)c * r.total) / r.G);
    r.t1 = (int)(((long long)(c + 1) * r.total) / r.G);
    int lo = 0, hi = p.S - 1;  // first segment whose tile range reaches past t0
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (tstart[mid + 1] > r.t0) hi = mid; else lo = mid + 1;
    }
    r.s0 = lo;
  }
  return r;
}

// ---------------------------------------------------------------------------
// producer warp: fill the stage ring for this CTA's tiles
// ---------------------------------------------------------------------------
// full[st] completes when stage st holds the tile (TMA: one expect_tx arrive
// plus the box bytes; cp.async: one arrive per lane); empty[st] is completed by
// the consumers when they are done with it.  Returns the tiles issued.
// At most MAXF tiles are in flight (issued, not landed): tile j is issued
// once tile j - MAXF has landed, and with a cap the second tile waits for the
// first, so at the start of the kernel the first tile of every CTA does not
// share the memory system with the rest of the ring.
//
// NPW warps may share the gather (warp pw takes the row sets j = pw mod NPW,
// and full[] then counts 32 * NPW arrivals); only warp 0 issues TMA boxes.
// PATH fixes the way tiles arrive at compile time (1 = TMA boxes only, 0 =
// cp.async gather only; -1 = chosen by use_tma): a kernel built for one way
// carries none of the other's code, which measurably slows the warps that
// share the kernel.
template <typename Tin, int D, int NS, int TK = kTK, int MAXF = NS, int NPW = 1, int PATH = -1>
__device__ __forceinline__ int produce_tiles(const AttnParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                             const int *tstart, const CtaRange &cr, uint8_t *stages,
                                             uint64_t *full, uint64_t *empty, volatile int *abort_flag,
                                             bool use_tma, bool &ok, int pw = 0) {
  using C = StageGeom<Tin, D, TK>;
  constexpr int kRowSets = TK / 32; // key rows per lane in the gather
  static_assert(kRowSets % NPW == 0, "row sets split evenly over the producer warps");
  const int lane = threadIdx.x & 31;
  if constexpr (PATH >= 0) use_tma = PATH == 1;
  if (use_tma && pw != 0) return 0;
  const uint64_t policy = l2_evict_first_policy();
  const Tin *kbase = static_cast<const Tin *>(p.k);
  const uintptr_t vdelta = reinterpret_cast<uintptr_t>(p.v) - reinterpret_cast<uintptr_t>(p.k);
  if (use_tma && lane == 0) {
    prefetch_tmap(tmk);
    prefetch_tmap(tmv);
  }
  // gather: the row addresses of the tile being issued; those of the next
  // tile are loaded before this tile's copies are issued, so their latency
  // hides behind the copies
  const Tin *rows[kRowSets];
  auto load_rows = [&](const Seg &gg, int ltt, const Tin **dst) {
#pragma unroll
    for (int j = 0; j < kRowSets; ++j) {
      if (j % NPW != pw) continue;
      const int k = ltt * TK + lane + 32 * j;
      dst[j] = k < gg.nkeys ? key_row<Tin, D>(p, gg, k, kbase) : kbase;
    }
  };
  if (!use_tma && cr.s0 < p.S && tstart[cr.s0] < cr.t1)
    load_rows(seg_info(p, cr.s0, false), max(tstart[cr.s0], cr.t0) - tstart[cr.s0], rows);
  int it = 0;
  for (int s = cr.s0; s < p.S && tstart[s] < cr.t1; ++s) {
    const Seg g = seg_info(p, s, false);
    const int lt0 = max(tstart[s], cr.t0) - tstart[s];
    const int lt1 = min(tstart[s + 1], cr.t1) - tstart[s];
    for (int lt = lt0; lt < lt1; ++lt, ++it) {
      const int st = it % NS;
      const uint32_t ph = (uint32_t)(it / NS) & 1u;
      role_wait(empty + st, ph ^ 1u, ok, abort_flag, p.wait_ns, p.status);
      // (with a cap, the second tile also waits for the first, which then lands sooner)
      const int gate = it >= MAXF ? it - MAXF : (it == 1 ? 0 : -1);
      if (MAXF < NS && ok && gate >= 0 &&
          !mbar_wait(full + gate % NS, (uint32_t)(gate / NS) & 1u, p.wait_ns)) {
        record_status(p.status, VA_ERR_TIMEOUT);
        *abort_flag = 1;
        ok = false;
      }
      if (!ok) continue;
      uint8_t *kdst = stages + st * C::kStageBytes;
      uint8_t *vdst = kdst + C::kTileBytes;
      const int k0 = lt * TK;
      if (use_tma) {
        // TMA boxes of BR rows x one kv-head x 128 bytes of the head dimension.
        // Dense: BR = 64 consecutive tokens; rows past the segment end arrive
        // too (other tokens or zero fill) and are masked.  Paged: one box per
        // page (BR = page size, at most 64), so a box never crosses a page;
        // boxes that start past the segment end are not loaded (their page
        // entries need not exist) and the rows they would fill are masked.
        const int BR = p.tma_box;
        const int nbox = TK / BR;  // boxes per 128-byte column (at most 16)
        const bool paged = p.layout == VA_LAYOUT_PAGED;
        const int nb = paged ? min(nbox, (g.nkeys - k0 + BR - 1) / BR) : nbox;
        if (lane == 0) mbar_arrive_expect_tx(full + st, (uint32_t)(nb * BR * 128 * C::kHalves * 2));
        __syncwarp();
        if (lane < nb) {
          const int slot = k0 + lane * BR;
          int row;
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
          const int off = lane * BR * 128;
#pragma unroll
          for (int h = 0; h < C::kHalves; ++h) {
            tma_load_3d(kdst + h * TK * 128 + off, tmk, h * (128 / (int)sizeof(Tin)), g.hkv, row, full + st, policy);
            tma_load_3d(vdst + h * TK * 128 + off, tmv, h * (128 / (int)sizeof(Tin)), g.hkv, row, full + st, policy);
          }
        }
      } else {
        // paged (pages below 8 rows) / sparse: gather rows with 16-byte
        // copies, rows past the end zero-filled.  Lane l resolves rows l + 32j;
        // a pass copies RPP rows, each row's address shuffled from its lane.
        const Tin *nrows[kRowSets];
        bool has_next = true;
        if (lt + 1 < lt1) {
          load_rows(g, lt + 1, nrows);
        } else if (s + 1 < p.S && tstart[s + 1] < cr.t1) {
          load_rows(seg_info(p, s + 1, false), max(tstart[s + 1], cr.t0) - tstart[s + 1], nrows);
        } else {
          has_next = false;
        }
        constexpr int CPR = C::kChunks;  // lanes per row
        constexpr int RPP = 32 / CPR;    // rows per pass
        const int cc = lane % CPR;
        const int rsub = lane / CPR;
        const int nvalid = g.nkeys - k0;
#pragma unroll
        for (int j = 0; j < kRowSets; ++j) {
          if (j % NPW != pw) continue;
#pragma unroll
          for (int i = 0; i < 32 / RPP; ++i) {
            const int rl = i * RPP + rsub;
            const uintptr_t a = (uintptr_t)__shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(rows[j]), rl);
            const int r = 32 * j + rl;
            const uintptr_t src = a + (uintptr_t)cc * 16u;
            const uint32_t n = r < nvalid ? 16u : 0u;
            const uint32_t off = swz<TK>(r, cc);
            cp_async_16(kdst + off, reinterpret_cast<const void *>(src), n);
            cp_async_16(vdst + off, reinterpret_cast<const void *>(src + vdelta), n);
          }
        }
        cp_async_mbar_arrive(full + st);
        if (has_next) {
#pragma unroll
          for (int j = 0; j < kRowSets; ++j) rows[j] = nrows[j];
        }
      }
    }
  }
  if (!ok) {
    // drain the copies this warp issued before leaving (bounded)
    if (use_tma) {
      for (int j = max(0, it - NS); j < it; ++j) mbar_wait(full + (j % NS), (uint32_t)(j / NS) & 1u, p.wait_ns >> 4);
    } else {
      cp_async_wait_all();
    }
  }
  return it;
}

}  // namespace va
