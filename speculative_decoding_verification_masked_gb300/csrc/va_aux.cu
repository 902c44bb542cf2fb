// Auxiliary kernels of the verification path:
//  * tree_mask_kernel   -- ancestor-or-self bitmask of token trees
//                          (LongSpec 1.3 / 2.C: each branch attends to its path)
//  * build_index_kernel -- fixed-size verify index set (Dustin section 1)
//  * wait_selftest_kernel -- exercises the bounded-wait error path
#include "va_common.cuh"
#include "va_kernels.h"

namespace va {

// ---------------------------------------------------------------------------
// tree -> bitmask
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(64) tree_mask_kernel(int T, const int32_t *parent, uint32_t *mask, int *status) {
  __shared__ int par[64];
  const int b = blockIdx.x;
  const int t = threadIdx.x;
  if (t < T) {
    int pp = __ldg(parent + (size_t)b * T + t);
    if (pp < -1 || pp >= t) {  // the path is cut at a node whose parent is not earlier
      record_status(status, VA_ERR_DEVICE_BOUNDS);
      pp = -1;
    }
    par[t] = pp;
  }
  __syncthreads();
  if (t >= T) return;
  uint64_t row = 0;
  for (int j = t; j >= 0; j = par[j]) row |= 1ull << j;  // par[j] < j: ends within T steps
  const int W = (T + 31) / 32;
  uint32_t *dst = mask + ((size_t)b * T + t) * W;
  dst[0] = (uint32_t)row;
  if (W > 1) dst[1] = (uint32_t)(row >> 32);
}

cudaError_t launch_tree_mask(int B, int T, const int32_t *parent, uint32_t *mask, int *status, cudaStream_t stream) {
  tree_mask_kernel<<<B, 64, 0, stream>>>(T, parent, mask, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// verify index set (Dustin section 1): sinks + recent window + top-m of the
// draft signal + top of the target signal, sorted ascending.
//
// One CTA per (sequence, kv-head).  The chosen set lives in a bitmap over
// positions, so the output comes out sorted by a prefix count over bitmap
// words.  Each top-k is an exact radix select on order-preserving 32-bit keys
// (digits of 11, 11 and 10 bits, most significant first); keys equal to the
// threshold are taken in increasing position order, which is the tie rule.
// ---------------------------------------------------------------------------
constexpr int kIdxThreads = 1024;
constexpr int kIdxMaxL = 131072;
constexpr int kIdxBitmapWords = kIdxMaxL / 32 + 4;
constexpr int kIdxCacheKeys = 36864;  // keys held in shared memory when L fits
constexpr int kIdxLoads = 16;         // score loads in flight per thread while caching
constexpr int kIdxBins = 2048;        // bins of one radix digit (11 bits)
constexpr int kIdxCopies = 8;         // histogram copies, each shared by 4 warps
constexpr int kIdxCandCap = (kIdxCopies - 1) * kIdxBins;  // candidate keys held behind one histogram
constexpr int kIdxFastCap = 4096;     // candidates of the sampled-threshold select

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 ranks with +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct IdxSmem {
  uint32_t *bitmap;
  uint32_t *hist;  // kIdxCopies histograms of kIdxBins bins
  int *scratch;
  uint32_t *keys;
};

// Block-wide exclusive scan of one int per thread (1024 threads); returns the
// thread's exclusive prefix and the block total.
__device__ __forceinline__ int block_exclusive_scan(int v, int *scratch, int &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int wv = scratch[lane];
    int wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    scratch[32 + lane] = wi - wv;  // exclusive warp offsets
    if (lane == 31) scratch[31] = wi;  // total (slot 31 is no longer needed)
  }
  __syncthreads();
  const int res = scratch[32 + warp] + incl - v;
  total = scratch[31];
  __syncthreads();
  return res;
}

// Keys still to be added to the chosen set: every key k != 0 with
// (k & pmask) >= prefix.  A select whose threshold bucket is taken whole
// leaves this pending; the next fill of the key cache (or the final pass)
// applies it while it reads the old keys.
struct Take {
  uint32_t prefix, pmask;
  bool active;
};

__device__ __forceinline__ bool take_key(uint32_t key, const Take &t) {
  return t.active && key != 0u && (key & t.pmask) >= t.prefix;
}

// Digits of the radix select: bits 31-21, 20-10 and 9-0.  Eleven bits in the
// first digit already split the exponent and the top mantissa bits, so
// continuous scores are usually resolved after two digits.
__device__ __forceinline__ int digit_shift(int d) { return d == 0 ? 21 : d == 1 ? 10 : 0; }
__device__ __forceinline__ int digit_bits(int d) { return d == 2 ? 10 : 11; }

__device__ __forceinline__ void hist_zero(const IdxSmem &sm) {
  for (int j = threadIdx.x; j < kIdxCopies * kIdxBins; j += kIdxThreads) sm.hist[j] = 0;
}

// The bucket of a digit of `bits` bits (at most 11) that holds the kk-th
// largest counted key: thread t owns the 1 or 2 bins just below bin
// nb - 1 - per * t (bins scanned from the top).  Sets scratch[64] = bin,
// [65] = rank inside it, [66] = bucket taken whole.
__device__ __forceinline__ void find_bucket(int bits, int kk, const IdxSmem &sm, int copies) {
  const int nb = 1 << bits;
  const int per = nb > kIdxThreads ? nb / kIdxThreads : 1;  // 2 or 1
  const int tid = threadIdx.x;
  int c[2] = {0, 0};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    if (j < per && tid * per + j < nb) {
      const int bin = nb - 1 - (tid * per + j);
      for (int h = 0; h < copies; ++h) c[j] += (int)sm.hist[h * kIdxBins + bin];
    }
  }
  int tot;
  int run = block_exclusive_scan(c[0] + c[1], sm.scratch, tot);
  if (run < kk && kk <= run + c[0] + c[1]) {
    for (int j = 0; j < per; ++j) {
      if (run + c[j] >= kk) {
        sm.scratch[64] = nb - 1 - (tid * per + j);
        sm.scratch[65] = kk - run;
        sm.scratch[66] = (run + c[j] == kk) ? 1 : 0;
        break;
      }
      run += c[j];
    }
  }
  __syncthreads();
}

// Select the k largest keys among positions [0, L) not yet in the bitmap (nor
// in `prev`, still pending) and return them as a pending Take -- or add them
// to the bitmap now when the key cache is not used or ties decide.
// k must not exceed the number of such positions.
//
// Radix select, most significant digit first.  After each digit the bucket
// holding the k-th largest key is known together with how many keys above it
// are already certain.  If that bucket holds exactly the keys still needed,
// every key at or above it is taken.  Otherwise the search narrows to the
// bucket; if keys equal to the final threshold still outnumber the quota,
// they are taken in increasing position order (the tie rule).
__device__ Take select_top(const float *src, int L, int k, const IdxSmem &sm, const Take prev) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t *myhist = sm.hist + kIdxBins * (warp % kIdxCopies);
  const bool cached = L <= kIdxCacheKeys;
  auto excluded = [&](int i) -> bool { return (sm.bitmap[i >> 5] >> (i & 31)) & 1u; };
  hist_zero(sm);
  __syncthreads();
  if (cached) {
    // fill the key cache, kIdxLoads loads in flight per thread; apply the
    // pending take of the previous select; histogram of the first digit
    for (int base = 0; base < L; base += kIdxThreads * kIdxLoads) {
      float v[kIdxLoads];
#pragma unroll
      for (int u = 0; u < kIdxLoads; ++u) {
        const int i = base + u * kIdxThreads + tid;
        v[u] = i < L ? __ldg(src + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kIdxLoads; ++u) {
        const int i = base + u * kIdxThreads + tid;
        if (base + u * kIdxThreads >= L) break;  // uniform over the block
        bool ex = false, took = false;
        if (i < L) {
          took = take_key(sm.keys[i], prev);
          ex = took || excluded(i);
        }
        const uint32_t word = __ballot_sync(0xffffffffu, took);
        if (lane == 0 && word != 0u) sm.bitmap[((base + u * kIdxThreads) >> 5) + warp] |= word;
        if (i < L) {
          const uint32_t key = ex ? 0u : order_key(v[u]);
          sm.keys[i] = key;
          if (key != 0u) atomicAdd(myhist + (key >> 21), 1u);
        }
      }
    }
  } else {
    for (int i = tid; i < L; i += kIdxThreads) {
      if (!excluded(i)) atomicAdd(myhist + (order_key(__ldg(src + i)) >> 21), 1u);
    }
  }
  __syncthreads();
  if (k <= 0) return Take{0u, 0u, false};
  auto key_at = [&](int i) -> uint32_t {
    if (cached) return sm.keys[i];
    return excluded(i) ? 0u : order_key(__ldg(src + i));
  };

  uint32_t prefix = 0, pmask = 0;
  int kk = k;
  bool exact_bucket = false;
  // after the first digit the keys of its chosen bucket are copied to a
  // candidate list (behind the first histogram), and the later digits count
  // those only, with one histogram; a bucket larger than the list keeps the
  // full passes
  uint32_t *cand = sm.hist + kIdxBins;
  int ncand = -1;
  for (int d = 0; d < 3; ++d) {
    const int shift = digit_shift(d), bits = digit_bits(d);
    if (d > 0 && ncand >= 0) {
      for (int j = tid; j < kIdxBins; j += kIdxThreads) sm.hist[j] = 0;
      __syncthreads();
      for (int e = tid; e < ncand; e += kIdxThreads) {
        const uint32_t key = cand[e];
        if ((key & pmask) == prefix) atomicAdd(sm.hist + ((key >> shift) & ((1u << bits) - 1u)), 1u);
      }
      __syncthreads();
    } else if (d > 0) {
      hist_zero(sm);
      __syncthreads();
      for (int base = 0; base < L; base += kIdxThreads * 4) {
        uint32_t kv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = base + u * kIdxThreads + tid;
          kv[u] = i < L ? key_at(i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (kv[u] != 0u && (kv[u] & pmask) == prefix) atomicAdd(myhist + ((kv[u] >> shift) & ((1u << bits) - 1u)), 1u);
      }
      __syncthreads();
    }
    find_bucket(bits, kk, sm, ncand >= 0 ? 1 : kIdxCopies);
    prefix |= (uint32_t)sm.scratch[64] << shift;
    pmask |= ((1u << bits) - 1u) << shift;
    kk = sm.scratch[65];
    exact_bucket = sm.scratch[66] != 0;
    __syncthreads();
    if (exact_bucket) break;
    if (d == 0 && cached) {
      // candidate list: warp-aggregated appends of the keys in the bucket
      if (tid == 0) sm.scratch[67] = 0;
      __syncthreads();
      for (int base = 0; base < L; base += kIdxThreads) {
        const int i = base + tid;
        const uint32_t key = i < L ? sm.keys[i] : 0u;
        const bool in = key != 0u && (key & pmask) == prefix;
        const uint32_t m = __ballot_sync(0xffffffffu, in);
        int at = 0;
        if (lane == 0 && m != 0u) at = atomicAdd(&sm.scratch[67], __popc(m));
        at = __shfl_sync(0xffffffffu, at, 0) + __popc(m & ((1u << lane) - 1u));
        if (in && at < kIdxCandCap) cand[at] = key;
      }
      __syncthreads();
      const int n = sm.scratch[67];
      ncand = n <= kIdxCandCap ? n : -1;
      __syncthreads();
    }
  }
  if (exact_bucket) {
    const Take t{prefix, pmask, true};
    if (cached) return t;  // applied by the next pass over the key cache
    for (int base = 0; base < L; base += kIdxThreads) {
      const int i = base + tid;
      const bool take = i < L && take_key(key_at(i), t);
      const uint32_t word = __ballot_sync(0xffffffffu, take);
      if (lane == 0 && word != 0u) sm.bitmap[(base >> 5) + warp] |= word;
    }
    __syncthreads();
    return Take{0u, 0u, false};
  }
  // ties at the full 32-bit threshold exceed the quota: above-threshold keys plus
  // the first kk equal keys in position order
  int taken_eq = 0;
  for (int base = 0; base < L; base += kIdxThreads) {
    const int i = base + tid;
    uint32_t key = 0;
    if (i < L) key = key_at(i);
    const bool gt = i < L && key != 0u && key > prefix;
    const bool eq = i < L && key == prefix;
    int tot;
    const int before = block_exclusive_scan(eq ? 1 : 0, sm.scratch, tot);
    const bool take = gt || (eq && taken_eq + before < kk);
    const uint32_t word = __ballot_sync(0xffffffffu, take);
    if (lane == 0 && word != 0u) sm.bitmap[(base >> 5) + warp] |= word;
    taken_eq += tot;
  }
  __syncthreads();
  return Take{0u, 0u, false};
}

// Mark in the bitmap every key of the key cache that a pending Take selects.
__device__ void apply_take(const IdxSmem &sm, int L, const Take &t) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int base = 0; base < L; base += kIdxThreads) {
    const int i = base + tid;
    const bool take = i < L && take_key(sm.keys[i], t);
    const uint32_t word = __ballot_sync(0xffffffffu, take);
    if (lane == 0 && word != 0u) sm.bitmap[(base >> 5) + warp] |= word;
  }
  __syncthreads();
}

// Top k of src over the positions not yet in the bitmap, added to the bitmap,
// in one pass over the scores where it can: a threshold from a sorted sample
// of 1024 positions (chosen so that about 2 k eligible keys reach it), the
// keys at or above it collected with their positions, and the radix select
// run over those candidates only.  Every key of the top k is at or above the
// threshold whenever at least k candidates reach it, so the result is exact.
// Keys equal to the final threshold beyond the quota are taken in position
// order (the tie rule).  Returns false -- having changed nothing -- when fewer
// than k keys reach the sampled threshold, when a warp collects more than its
// share of the candidate space, or when more than 32 keys tie at the final
// threshold; select_top then does the work.
constexpr int kIdxWarpCand = kIdxFastCap / (kIdxThreads / 32);  // candidate slots per warp
__device__ bool select_top_fast(const float *src, int L, int k, const IdxSmem &sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto excluded = [&](int i) -> bool { return (sm.bitmap[i >> 5] >> (i & 31)) & 1u; };
  uint32_t *ckey = sm.keys;                                      // [warp][kIdxWarpCand]
  int *cpos = reinterpret_cast<int *>(sm.keys + kIdxFastCap);    // [warp][kIdxWarpCand]
  int *wcount = sm.scratch + 72;                                 // [32]
  uint32_t thr = 1u;  // the smallest counted key: every eligible key
  const long long q = ((long long)k * 2048 + L - 1) / L + 8;  // sample rank of ~2 k keys
  if (L > kIdxFastCap && q < kIdxThreads) {
    // bitonic sort of the 1024 sample keys, largest first: exchanges between
    // lanes by shuffles, between warps through two alternating arrays
    const int ps = (int)(((long long)tid * L) >> 10);
    uint32_t x = excluded(ps) ? 0u : order_key(__ldg(src + ps));
    uint32_t *buf[2] = {sm.hist, sm.hist + kIdxThreads};
    int pb = 0;
    for (int kb = 2; kb <= kIdxThreads; kb <<= 1) {
      for (int j = kb >> 1; j > 0; j >>= 1) {
        uint32_t y;
        if (j < 32) {
          y = __shfl_xor_sync(0xffffffffu, x, j);
        } else {
          buf[pb][tid] = x;
          __syncthreads();
          y = buf[pb][tid ^ j];
          pb ^= 1;
        }
        const bool keep_max = ((tid & kb) == 0) == ((tid & j) == 0);
        x = keep_max ? max(x, y) : min(x, y);
      }
    }
    if (tid == q - 1) sm.scratch[70] = (int)x;
    __syncthreads();
    thr = (uint32_t)sm.scratch[70];
    __syncthreads();
    if (thr == 0u) return false;
  }
  // one pass: the eligible keys at or above the threshold, with their
  // positions, each warp into its own slots (no shared counter); four
  // consecutive scores a load where the row is 16-byte aligned
  int cw = 0;
  uint32_t kmax = 0u;
  uint32_t *wk = ckey + warp * kIdxWarpCand;
  int *wp = cpos + warp * kIdxWarpCand;
  // the float whose key is thr: !(f < thr_f) holds for every f whose key is
  // at least thr (and for NaN, which the exact key test then settles)
  const float thr_f = __uint_as_float((thr & 0x80000000u) ? (thr & 0x7fffffffu) : ~thr);
  auto offer = [&](int i, float f) {
    bool in = i < L && !(f < thr_f);
    uint32_t key = 0u;
    if (in) {
      key = order_key(f);
      in = key != 0u && key >= thr && !excluded(i);
    }
    const uint32_t m = __ballot_sync(0xffffffffu, in);
    if (in) {
      const int at = cw + __popc(m & ((1u << lane) - 1u));
      kmax = max(kmax, key);
      if (at < kIdxWarpCand) {
        wk[at] = key;
        wp[at] = i;
      }
    }
    cw += __popc(m);
  };
  if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
    constexpr int kV = 8;  // float4 loads in flight per thread
    for (int base = 0; base < L; base += kIdxThreads * 4 * kV) {
      float4 v[kV];
#pragma unroll
      for (int u = 0; u < kV; ++u) {
        const int i = base + 4 * (u * kIdxThreads + tid);
        v[u] = i + 3 < L ? __ldg(reinterpret_cast<const float4 *>(src + i))
                         : make_float4(i < L ? __ldg(src + i) : 0.f, i + 1 < L ? __ldg(src + i + 1) : 0.f,
                                       i + 2 < L ? __ldg(src + i + 2) : 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kV; ++u) {
        if (base + 4 * u * kIdxThreads >= L) break;  // uniform over the block
        const int i = base + 4 * (u * kIdxThreads + tid);
        offer(i, v[u].x);
        offer(i + 1, v[u].y);
        offer(i + 2, v[u].z);
        offer(i + 3, v[u].w);
      }
    }
  } else {
    for (int base = 0; base < L; base += kIdxThreads * kIdxLoads) {
      float v[kIdxLoads];
#pragma unroll
      for (int u = 0; u < kIdxLoads; ++u) {
        const int i = base + u * kIdxThreads + tid;
        v[u] = i < L ? __ldg(src + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kIdxLoads; ++u) {
        if (base + u * kIdxThreads >= L) break;  // uniform over the block
        offer(base + u * kIdxThreads + tid, v[u]);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  if (tid == 0) sm.scratch[71] = 0;
  __syncthreads();
  if (lane == 0) atomicMax(reinterpret_cast<unsigned *>(&sm.scratch[71]), kmax);
  if (lane == 0) wcount[warp] = cw;
  __syncthreads();
  int n = 0;
  bool over = false;
#pragma unroll 4
  for (int w = 0; w < kIdxThreads / 32; ++w) {
    n += wcount[w];
    over = over || wcount[w] > kIdxWarpCand;
  }
  if (over || n < k) return false;
  // radix select among the candidates: every candidate lies in [thr, max],
  // so the bits those two share are fixed and the digits (11 bits at a time)
  // start below them, where the candidates differ
  kmax = (uint32_t)sm.scratch[71];
  const int common = kmax == thr ? 32 : __clz(kmax ^ thr);
  uint32_t pmask = common == 0 ? 0u : (common == 32 ? 0xFFFFFFFFu : ~((1u << (32 - common)) - 1u));
  uint32_t prefix = thr & pmask;
  int kk = k;
  bool exact = false;
  int below = 32 - common;
  if (below == 0) exact = n == k;  // every candidate equal
  while (below > 0 && !exact) {
    const int bits = below < 11 ? below : 11;
    below -= bits;
    const int shift = below;
    for (int j = tid; j < kIdxBins; j += kIdxThreads) sm.hist[j] = 0;
    __syncthreads();
    for (int e = tid; e < kIdxFastCap; e += kIdxThreads) {
      if ((e % kIdxWarpCand) >= wcount[e / kIdxWarpCand]) continue;
      const uint32_t key = ckey[e];
      if ((key & pmask) == prefix) atomicAdd(sm.hist + ((key >> shift) & ((1u << bits) - 1u)), 1u);
    }
    __syncthreads();
    find_bucket(bits, kk, sm, 1);
    prefix |= (uint32_t)sm.scratch[64] << shift;
    pmask |= ((1u << bits) - 1u) << shift;
    kk = sm.scratch[65];
    exact = sm.scratch[66] != 0;
    __syncthreads();
  }
  if (!exact) {
    // keys equal to the full threshold (prefix) outnumber the kk still to
    // take: the kk of them at the smallest positions (the tie rule); up to 32
    // are ranked by one warp, more are left to select_top
    if (tid == 0) sm.scratch[69] = 0;
    __syncthreads();
    int *tpos = reinterpret_cast<int *>(sm.hist);
    for (int e = tid; e < kIdxFastCap; e += kIdxThreads) {
      if ((e % kIdxWarpCand) >= wcount[e / kIdxWarpCand] || ckey[e] != prefix) continue;
      const int at = atomicAdd(&sm.scratch[69], 1);
      if (at < 32) tpos[at] = cpos[e];
    }
    __syncthreads();
    const int ct = sm.scratch[69];
    if (ct > 32) return false;
    if (warp == 0) {
      const int mine = lane < ct ? tpos[lane] : 0x7fffffff;
      int rank = 0;
#pragma unroll
      for (int o = 0; o < 32; ++o) rank += __shfl_sync(0xffffffffu, mine, o) < mine ? 1 : 0;
      if (lane < ct && rank < kk) atomicOr(&sm.bitmap[mine >> 5], 1u << (mine & 31));
    }
  }
  // every key above the threshold bucket (and the bucket itself when it is
  // taken whole)
  for (int e = tid; e < kIdxFastCap; e += kIdxThreads) {
    if ((e % kIdxWarpCand) >= wcount[e / kIdxWarpCand]) continue;
    const uint32_t key = ckey[e] & pmask;
    if (exact ? key >= prefix : key > prefix) {
      const int i = cpos[e];
      atomicOr(&sm.bitmap[i >> 5], 1u << (i & 31));
    }
  }
  __syncthreads();
  return true;
}

struct IndexParams {
  int B, Hkv;
  const int32_t *seqlens;
  const float *sd, *st;
  int stride, n_sink, window, m_draft, budget;
  int32_t *indices, *n_indices;
  int *status;
  int radix_only;  // skip the sampled-threshold select (test hook)
};

__global__ void __launch_bounds__(kIdxThreads) build_index_kernel(const IndexParams p) {
  extern __shared__ __align__(16) uint32_t ism[];
  IdxSmem sm;
  sm.bitmap = ism;
  sm.hist = ism + kIdxBitmapWords;
  sm.scratch = reinterpret_cast<int *>(sm.hist + kIdxCopies * kIdxBins);
  sm.keys = reinterpret_cast<uint32_t *>(sm.scratch + 128);
  const int tid = threadIdx.x;
  const int b = blockIdx.x / p.Hkv;
  const int h = blockIdx.x % p.Hkv;
  int L = __ldg(p.seqlens + b);
  const int cap = min(p.stride, kIdxMaxL);
  if (L < 0 || L > cap) {
    record_status(p.status, VA_ERR_DEVICE_BOUNDS);
    L = L < 0 ? 0 : cap;
  }
  const size_t row = ((size_t)b * p.Hkv + h);
  {
    // both score rows are read in full below: start bringing them into L2 now
    const float *sd = p.sd + row * p.stride, *st = p.st + row * p.stride;
    for (int j = tid; 32 * j < L; j += kIdxThreads) {
      asm volatile("prefetch.global.L2 [%0];" ::"l"(sd + 32 * j));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(st + 32 * j));
    }
  }
  const int nwords = (L + 31) / 32;
  // fixed part: sinks [0, a) and window [wlo, L)
  const int a = min(p.n_sink, L);
  const int wlo = max(0, L - p.window);
  for (int w = tid; w < nwords; w += kIdxThreads) {
    uint32_t bits = 0;
    for (int j = 0; j < 32; ++j) {
      const int i = 32 * w + j;
      if (i < L && (i < a || i >= wlo)) bits |= 1u << j;
    }
    sm.bitmap[w] = bits;
  }
  __syncthreads();
  const int fixed = a + (L - wlo) - max(0, a - wlo);
  const int room = max(0, p.budget - fixed);
  const int ncand = L - fixed;
  const int m1 = max(0, min(min(p.m_draft, room), ncand));
  const int m2 = max(0, min(room - m1, ncand - m1));
  const Take none{0u, 0u, false};
  const bool fast = p.radix_only == 0;
  if (m1 > 0 && !(fast && select_top_fast(p.sd + row * p.stride, L, m1, sm))) {
    const Take t = select_top(p.sd + row * p.stride, L, m1, sm, none);
    if (t.active) apply_take(sm, L, t);
  }
  if (m2 > 0 && !(fast && select_top_fast(p.st + row * p.stride, L, m2, sm))) {
    const Take t = select_top(p.st + row * p.stride, L, m2, sm, none);
    if (t.active) apply_take(sm, L, t);
  }

  // bitmap -> ascending positions
  int32_t *out = p.indices + row * p.budget;
  int written = 0;
  for (int base = 0; base < nwords; base += kIdxThreads) {
    const int w = base + tid;
    const uint32_t bits = w < nwords ? sm.bitmap[w] : 0u;
    int tot;
    int off = written + block_exclusive_scan(__popc(bits), sm.scratch, tot);
    uint32_t rem = bits;
    while (rem) {
      const int j = __ffs(rem) - 1;
      rem &= rem - 1;
      if (off < p.budget) out[off] = 32 * w + j;
      ++off;
    }
    written += tot;
  }
  const int n = min(written, p.budget);
  for (int i = n + tid; i < p.budget; i += kIdxThreads) out[i] = -1;
  if (tid == 0) p.n_indices[row] = n;
}

size_t build_index_smem_bytes() {
  return sizeof(uint32_t) * (kIdxBitmapWords + kIdxCopies * kIdxBins + 128 + kIdxCacheKeys);
}

cudaError_t launch_build_index(int B, int Hkv, const int32_t *seqlens, const float *score_draft,
                               const float *score_target, int score_stride, int n_sink, int window, int m_draft,
                               int budget, int32_t *indices, int32_t *n_indices, int *status, bool radix_only,
                               cudaStream_t stream) {
  IndexParams p;
  p.B = B;
  p.Hkv = Hkv;
  p.seqlens = seqlens;
  p.sd = score_draft;
  p.st = score_target;
  p.stride = score_stride;
  p.n_sink = n_sink;
  p.window = window;
  p.m_draft = m_draft;
  p.budget = budget;
  p.indices = indices;
  p.n_indices = n_indices;
  p.status = status;
  p.radix_only = radix_only ? 1 : 0;
  const size_t smem = build_index_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(build_index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  build_index_kernel<<<B * Hkv, kIdxThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// validation mode of the sparse call: every verify set strictly increasing
// inside [0, L_b) (a set, in the form the index builder writes)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) validate_index_kernel(int Hkv, const int32_t *seqlens, const int32_t *indices,
                                                            const int32_t *n_indices, int max_indices, int len_cap,
                                                            int T, int *status) {
  const int row = blockIdx.x;
  const int b = row / Hkv;
  const int L = min(max(__ldg(seqlens + b), 0), max(len_cap - T, 0));
  const int n = __ldg(n_indices + row);
  if (n < 0 || n > max_indices) {
    if (threadIdx.x == 0) record_status(status, VA_ERR_DEVICE_BOUNDS);
    return;
  }
  const int32_t *idx = indices + (size_t)row * max_indices;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int v = __ldg(idx + j);
    if (v < 0 || v >= L) record_status(status, VA_ERR_DEVICE_BOUNDS);
    else if (j + 1 < n && __ldg(idx + j + 1) <= v) record_status(status, VA_ERR_DEVICE_INVALID);
  }
}

cudaError_t launch_validate_index(int B, int Hkv, const int32_t *seqlens, const int32_t *indices,
                                  const int32_t *n_indices, int max_indices, int len_cap, int T, int *status,
                                  cudaStream_t stream) {
  validate_index_kernel<<<B * Hkv, 256, 0, stream>>>(Hkv, seqlens, indices, n_indices, max_indices, len_cap, T,
                                                     status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// bounded-wait self test: waits on an mbarrier nothing will ever complete;
// the wait must give up after wait_ns and record VA_ERR_TIMEOUT.
// ---------------------------------------------------------------------------
__global__ void wait_selftest_kernel(int *status, uint64_t wait_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0u, wait_ns)) record_status(status, VA_ERR_TIMEOUT);
}

cudaError_t launch_wait_selftest(int *status, uint64_t wait_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, wait_ns);
  return cudaGetLastError();
}

}  // namespace va
