// After verification: greedy acceptance over the token trees and the commit
// of the accepted draft rows into the KV cache (Dustin, section 1 step 5:
// accepted tokens join the cache and rejected ones are dropped; HiSpec,
// section 2: the entries of rejected tokens are removed before the next
// phase, and the output equals the target model's own greedy decoding).
//
//  * accept_greedy_kernel -- one 64-thread block per sequence: a node is
//    accepted when every node on its root path carries the target's greedy
//    token after its predecessor; the deepest accepted path (smallest end
//    node on ties) is written out with the bonus token after it.
//  * commit_kv_kernel -- one block per (sequence, kv-head, K or V): the rows
//    of the accepted nodes are first read into shared memory and only then
//    written to the slots right after the prefix, so the in-place move never
//    reads a row it has already overwritten.
#include "va_common.cuh"
#include "va_kernels.h"
#include "va_commit.h"

namespace va {

__global__ void __launch_bounds__(64) accept_greedy_kernel(int T, const int32_t *parent, const int32_t *draft,
                                                           const int32_t *target_next, int32_t *path,
                                                           int32_t *n_accept, int32_t *bonus, int *status) {
  __shared__ int par[64];
  __shared__ int match[64];
  __shared__ unsigned long long best;  // (depth << 32) | (63 - end node); 0 = nothing accepted
  const int b = blockIdx.x;
  const int t = threadIdx.x;
  const int32_t *tn = target_next + (size_t)b * (T + 1);
  if (t == 0) best = 0ull;
  if (t < T) {
    int p = __ldg(parent + (size_t)b * T + t);
    bool m = false;
    if (p < -1 || p >= t) {
      // not an earlier node: recorded, and the node is rejected (its row of
      // the walk is cut there, so every walk ends)
      record_status(status, VA_ERR_DEVICE_BOUNDS);
      p = -1;
    } else {
      m = __ldg(draft + (size_t)b * T + t) == __ldg(tn + p + 1);
    }
    par[t] = p;
    match[t] = m ? 1 : 0;
  }
  __syncthreads();
  if (t < T) {
    bool acc = true;
    int depth = 0;
    for (int j = t; j >= 0; j = par[j]) {  // par[j] < j: at most T steps
      acc = acc && match[j] != 0;
      ++depth;
    }
    if (acc) atomicMax(&best, ((unsigned long long)depth << 32) | (unsigned long long)(63 - t));
  }
  __syncthreads();
  const unsigned long long k = best;
  const int n = (int)(k >> 32);
  const int end = 63 - (int)(k & 0xffffffffull);
  if (t < T) {
    int node = -1;
    if (t < n) {  // the path's node at depth t: n - 1 - t steps up from the end
      node = end;
      for (int i = 0; i < n - 1 - t; ++i) node = par[node];
    }
    path[(size_t)b * T + t] = node;
  }
  if (t == 0) {
    n_accept[b] = n;
    bonus[b] = n > 0 ? __ldg(tn + end + 1) : __ldg(tn);
  }
}

cudaError_t launch_accept_greedy(int B, int T, const int32_t *parent, const int32_t *draft,
                                 const int32_t *target_next, int32_t *path, int32_t *n_accept, int32_t *bonus,
                                 int *status, cudaStream_t stream) {
  accept_greedy_kernel<<<B, 64, 0, stream>>>(T, parent, draft, target_next, path, n_accept, bonus, status);
  return cudaGetLastError();
}

// Address of (sequence b, logical slot, kv-head h) in a dense or paged cache;
// nullptr when a page entry is out of range (recorded).
__device__ __forceinline__ uint8_t *commit_row(const CommitParams &p, uint8_t *base, int b, int slot, int h) {
  size_t row;
  if (p.page_table != nullptr) {
    const int page = __ldg(p.page_table + (size_t)b * p.max_pages + (slot >> p.page_shift));
    if (page < 0 || page >= p.num_pages) {
      record_status(p.status, VA_ERR_DEVICE_BOUNDS);
      return nullptr;
    }
    row = ((size_t)page << p.page_shift) + (size_t)(slot & ((1 << p.page_shift) - 1));
  } else {
    row = (size_t)b * p.len_cap + slot;
  }
  return base + (row * p.Hkv + h) * (size_t)p.row_bytes;
}

__global__ void __launch_bounds__(128) commit_kv_kernel(const CommitParams p) {
  extern __shared__ uint4 rows[];  // [a][row_bytes / 16]
  __shared__ int src[64];
  const int b = blockIdx.x, h = blockIdx.y;
  uint8_t *base = static_cast<uint8_t *>(blockIdx.z == 0 ? p.k : p.v);
  const int tid = threadIdx.x;
  const int L = __ldg(p.seqlens + b);
  const int a = __ldg(p.n_accept + b);
  const bool first = h == 0 && blockIdx.z == 0;
  if (L < 0 || L > p.len_cap - p.T || a < 0 || a > p.T) {
    if (first && tid == 0) record_status(p.status, VA_ERR_DEVICE_BOUNDS);
    return;  // every block of this sequence leaves its rows alone
  }
  if (tid < a) {
    int s = __ldg(p.path + (size_t)b * p.T + tid);
    if (s < tid || s >= p.T) {  // a path node below its depth or past the draft block
      record_status(p.status, VA_ERR_DEVICE_BOUNDS);
      s = tid;  // leave that row in place
    }
    src[tid] = s;
  }
  __syncthreads();
  const int chunks = p.row_bytes / 16;
  // read every moved row first ...
  for (int e = tid; e < a * chunks; e += blockDim.x) {
    const int j = e / chunks, c = e % chunks;
    if (src[j] == j) continue;
    const uint8_t *r = commit_row(p, base, b, L + src[j], h);
    if (r != nullptr) rows[e] = *reinterpret_cast<const uint4 *>(r + 16 * c);
  }
  __syncthreads();
  // ... then write them to the slots after the prefix
  for (int e = tid; e < a * chunks; e += blockDim.x) {
    const int j = e / chunks, c = e % chunks;
    if (src[j] == j) continue;
    uint8_t *r = commit_row(p, base, b, L + j, h);
    if (r != nullptr && commit_row(p, base, b, L + src[j], h) != nullptr)
      *reinterpret_cast<uint4 *>(r + 16 * c) = rows[e];
  }
  if (first && tid == 0 && p.seqlens_out != nullptr) p.seqlens_out[b] = L + a;
}

cudaError_t launch_commit_kv(const CommitParams &p, cudaStream_t stream) {
  const size_t smem = (size_t)p.T * p.row_bytes;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(commit_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  commit_kv_kernel<<<dim3((unsigned)p.B, (unsigned)p.Hkv, 2), 128, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace va
