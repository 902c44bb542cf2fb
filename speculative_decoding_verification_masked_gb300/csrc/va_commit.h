// Launchers of the steps after verification (va_commit.cu): greedy tree
// acceptance and the KV commit of the accepted rows.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace va {
cudaError_t launch_accept_greedy(int B, int T, const int32_t *parent, const int32_t *draft,
                                 const int32_t *target_next, int32_t *path, int32_t *n_accept, int32_t *bonus,
                                 int *status, cudaStream_t stream);
struct CommitParams {
  int B, T, Hkv;
  int row_bytes;                // D * element size (a multiple of 16)
  void *k, *v;                  // dense [B][len_cap][Hkv][D] or paged [P][page][Hkv][D]
  int len_cap;                  // dense: max_cache_len; paged: max_pages * page size
  const int32_t *page_table;    // nullptr for the dense cache
  int page_shift, max_pages, num_pages;
  const int32_t *seqlens, *path, *n_accept;
  int32_t *seqlens_out;         // may be nullptr
  int *status;                  // may be nullptr
};
cudaError_t launch_commit_kv(const CommitParams &p, cudaStream_t stream);

}  // namespace va
