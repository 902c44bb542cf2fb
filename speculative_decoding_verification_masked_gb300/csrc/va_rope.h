// Launcher of the rotary embedding of the draft block (va_rope.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace va {

struct RopeParams {
  int B, T, Hq, Hkv, D;
  int fp32;                     // element type: 1 = fp32, 0 = bf16
  int vec8;                     // D % 16 == 0 and q, k 16-byte aligned: 8-pair vector items
  double inv_freq[128];         // base^(-2i/D) for i < D/2, formed on the host in fp64
  void *q;                      // [B][T][Hq][D]
  void *k;                      // dense [B][len_cap][Hkv][D] or paged [P][page][Hkv][D]
  int len_cap;                  // dense: max_cache_len; paged: max_pages * page size
  const int32_t *page_table;    // nullptr for the dense cache
  int page_shift, max_pages, num_pages;
  const int32_t *seqlens;       // [B]
  const int32_t *positions;     // [B][T]
  int *status;                  // may be nullptr
};

cudaError_t launch_rope_draft(const RopeParams &p, cudaStream_t stream);

}  // namespace va
