// Importance of the committed positions from a few query heads: the scoring
// pass that feeds the verify-set builder (Dustin, section 1: the target
// model's attention scores are one signal of the global importance map;
// section 2: that estimate runs on a few semantic retrieval heads only).
//
// For sequence b with L committed keys, each listed query head h and draft
// token t, p[h,t] is the attention distribution of q[b,t,h] over the L keys
// of kv-head h / group; the importance of position j is the sum of p[h,t][j]
// over the listed heads and tokens.  It is one map per sequence, written to
// every kv-head row of the output so that the per-(sequence, kv-head) index
// builder takes it unchanged.
//
// Two launches:
//  * head_logits_kernel -- one 4-warp CTA per (128-key chunk, sequence,
//    unit); a unit is up to 8 query rows of one kv-head.  Six CTAs share an
//    SM (80 registers a thread), so that enough K rows are in flight to keep
//    HBM busy without a shared-memory stage.  Each warp scores its 32
//    keys against the unit's rows on the tensor cores: S^T = K Q^T by
//    mma.sync m16n8k16 with 16 keys on the M side, the unit's rows on N and
//    the head dimension as K.  Every K row of the listed kv-heads is read
//    once from HBM (streaming loads).  The scores (base-2 units) go to
//    scratch, and per chunk and row the maximum and the sum of 2^(s - max).
//  * head_score_kernel -- one CTA per (1024-key chunk, sequence), chained by
//    programmatic dependent launch: loads the first rows' scores, merges the
//    chunk partials of every row into its log-sum-exp, then sums
//    2^(s - lse) over the rows for four keys per thread and writes the sums
//    to the Hkv rows of the output.
// Operand layout: a lane loads 16-byte runs of its K rows and of its Q row at
// the same head dimensions (8 * (lane % 4) + 32 j) and hands the four words
// of a run to the fragment slots of two consecutive K-steps.  Both operands
// are permuted along the head dimension in the same way, so every product
// q_d k_d enters the dot product exactly once.
#include <math.h>

#include "va_common.cuh"
#include "va_score.h"

namespace va {

size_t score_scratch_bytes(int B, int R, int max_cache_len) {
  const size_t n_chunks = ((size_t)max_cache_len + kScoreChunk - 1) / kScoreChunk;
  const size_t lpad = n_chunks * kScoreChunk;
  return align256(sizeof(float) * (size_t)B * R * lpad) + align256(sizeof(float2) * (size_t)B * n_chunks * R);
}

// Committed length of sequence b, clamped to what the cache and the output
// rows hold; an out-of-range value is recorded once.
__device__ __forceinline__ int score_len(const ScoreParams &p, int b, bool report) {
  int L = __ldg(p.seqlens + b);
  const int cap = min(p.max_cache_len, p.score_stride);
  if (L < 0 || L > cap) {
    if (report) record_status(p.status, VA_ERR_DEVICE_BOUNDS);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

__device__ __forceinline__ uint32_t word(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__global__ void __launch_bounds__(128, 6) head_logits_kernel(const ScoreParams p) {
  __shared__ float2 wpart[4][kScoreUnitRows];
  const int c = blockIdx.x, b = blockIdx.y;
  const int L = score_len(p, b, c == 0 && threadIdx.x == 0);
  const int k0 = c * kScoreChunk;
  if (k0 >= L) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, qd = lane & 3;
  const int kb = k0 + warp * 32;
  // the reduction grid may be scheduled once every CTA here has started
  // (it waits for this grid's completion before reading anything)
  pdl_launch_dependents();
  const int u = blockIdx.z;
  const int kvh = p.unit_kvh[u], row0 = p.unit_row0[u], nrow = p.unit_n[u];
  // B operand: query row g of the unit at dims 8 qd + 32 j .. +7
  uint4 wq[4];
  if (g < nrow) {
    const int r = row0 + g;
    const uint4 *qr = reinterpret_cast<const uint4 *>(
                          p.q + (((size_t)b * p.T + p.row_t[r]) * p.Hq + p.row_head[r]) * 128) + qd;
#pragma unroll
    for (int j = 0; j < 4; ++j) wq[j] = __ldg(qr + 4 * j);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) wq[j] = make_uint4(0, 0, 0, 0);
  }
  // A operand: keys kb + 16 s + 8 hf + g at the same dims (zero past L)
  uint4 wk[2][2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int key = kb + 16 * s + 8 * hf + g;
      if (key < L) {
        const uint4 *kr = reinterpret_cast<const uint4 *>(
                              p.k + (((size_t)b * p.max_cache_len + key) * p.Hkv + kvh) * 128) + qd;
#pragma unroll
        for (int j = 0; j < 4; ++j) wk[s][hf][j] = __ldcs(kr + 4 * j);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) wk[s][hf][j] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  float acc[2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    acc[s][0] = acc[s][1] = acc[s][2] = acc[s][3] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint32_t a[4] = {word(wk[s][0][j], 2 * h2), word(wk[s][1][j], 2 * h2),
                               word(wk[s][0][j], 2 * h2 + 1), word(wk[s][1][j], 2 * h2 + 1)};
        mma_bf16(acc[s], a, word(wq[j], 2 * h2), word(wq[j], 2 * h2 + 1));
      }
    }
  }
  // acc[s][2 hf + e] = score of key kb + 16 s + 8 hf + g against unit row 2 qd + e
  float x[2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int key = kb + 16 * s + 8 * (i >> 1) + g;
      x[s][i] = key < L ? acc[s][i] * p.scale_log2 : -INFINITY;
    }
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int rl = 2 * qd + e;
    if (rl < nrow) {
      float *lr = p.logits + ((size_t)b * p.R + row0 + rl) * p.lpad;
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int key = kb + 16 * s + 8 * hf + g;
          if (key < L) lr[key] = x[s][2 * hf + e];
        }
    }
    // maximum and sum of 2^(s - max) of row rl over the warp's 32 keys
    // (lanes with the same qd hold the same two rows)
    float m = fmaxf(fmaxf(x[0][e], x[0][2 + e]), fmaxf(x[1][e], x[1][2 + e]));
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float sum = 0.f;
    if (m != -INFINITY)
      sum = (ex2_approx(x[0][e] - m) + ex2_approx(x[0][2 + e] - m)) +
            (ex2_approx(x[1][e] - m) + ex2_approx(x[1][2 + e] - m));
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (g == 0) wpart[warp][rl] = make_float2(m, sum);
  }
  __syncthreads();
  if (threadIdx.x < nrow) {
    const int rl = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, wpart[w][rl].x);
    float S = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float2 v = wpart[w][rl];
      if (v.x != -INFINITY) S += v.y * ex2_approx(v.x - M);
    }
    p.part[((size_t)b * p.n_chunks + c) * p.R + row0 + rl] = make_float2(M, S);
  }
}

__global__ void __launch_bounds__(256) head_score_kernel(const ScoreParams p) {
  __shared__ float lse2[kScoreMaxRows];
  const int c = blockIdx.x, b = blockIdx.y;
  const int L = score_len(p, b, false);
  const int j0 = c * kScoreChunk2;
  if (j0 >= L) return;
  pdl_wait_primary();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = j0 + 4 * threadIdx.x;
  const bool act = j < L;
  const float *lb = p.logits + (size_t)b * p.R * p.lpad + (act ? j : j0);
  constexpr int PF = 8;  // rows whose scores are loaded while the partials are merged
  float4 xs[PF];
#pragma unroll
  for (int i = 0; i < PF; ++i)
    xs[i] = i < p.R ? __ldcg(reinterpret_cast<const float4 *>(lb + (size_t)i * p.lpad)) : make_float4(0.f, 0.f, 0.f, 0.f);
  const int nchk = (L + kScoreChunk - 1) / kScoreChunk;
  for (int r = warp; r < p.R; r += 8) {
    const float2 *pr = p.part + (size_t)b * p.n_chunks * p.R + r;
    float m = -INFINITY, s = 0.f;
    for (int i0 = lane; i0 < nchk; i0 += 128) {
      float2 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + 32 * u;
        v[u] = i < nchk ? __ldcg(pr + (size_t)i * p.R) : make_float2(-INFINITY, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (v[u].x == -INFINITY) continue;
        if (v[u].x > m) {
          s = s * ex2_approx(m - v[u].x) + v[u].y;
          m = v[u].x;
        } else {
          s += v[u].y * ex2_approx(v[u].x - m);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
      const float M = fmaxf(m, m2);
      s = (m == -INFINITY ? 0.f : s * ex2_approx(m - M)) + (m2 == -INFINITY ? 0.f : s2 * ex2_approx(m2 - M));
      m = M;
    }
    if (lane == 0) lse2[r] = m + log2f(s);
  }
  __syncthreads();
  if (!act) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < PF; ++i) {
    if (i < p.R) {
      const float l = lse2[i];
      acc.x += ex2_approx(xs[i].x - l);
      acc.y += ex2_approx(xs[i].y - l);
      acc.z += ex2_approx(xs[i].z - l);
      acc.w += ex2_approx(xs[i].w - l);
    }
  }
  for (int r = PF; r < p.R; r += 4) {
    float4 x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      x[i] = r + i < p.R ? __ldcg(reinterpret_cast<const float4 *>(lb + (size_t)(r + i) * p.lpad))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (r + i < p.R) {
        const float l = lse2[r + i];
        acc.x += ex2_approx(x[i].x - l);
        acc.y += ex2_approx(x[i].y - l);
        acc.z += ex2_approx(x[i].z - l);
        acc.w += ex2_approx(x[i].w - l);
      }
    }
  }
  const int n = min(4, L - j);
  for (int h = 0; h < p.Hkv; ++h) {
    float *dst = p.score + ((size_t)b * p.Hkv + h) * p.score_stride + j;
    if (n == 4 && p.score_vec4) {
      *reinterpret_cast<float4 *>(dst) = acc;
    } else {
      dst[0] = acc.x;
      if (n > 1) dst[1] = acc.y;
      if (n > 2) dst[2] = acc.z;
      if (n > 3) dst[3] = acc.w;
    }
  }
}

cudaError_t launch_head_importance(const ScoreParams &p, cudaStream_t stream) {
  head_logits_kernel<<<dim3((unsigned)p.n_chunks, (unsigned)p.B, (unsigned)p.n_units), 128, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned n2 = (unsigned)((p.max_cache_len + kScoreChunk2 - 1) / kScoreChunk2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n2, (unsigned)p.B);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, head_score_kernel, p);
}

}  // namespace va
