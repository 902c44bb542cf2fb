// Internal interface between the C ABI layer (va_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "verify_attn.h"

namespace va {

// Everything one attention launch needs; plain values and device pointers.
struct AttnParams {
  // shape
  int B, T, Hq, Hkv, D;
  int R;       // packed query rows per (sequence, kv-head) = (Hq/Hkv) * T
  int RG;      // 16-row groups per segment (1, 2 or 4)
  int NRB;     // row blocks per (sequence, kv-head)
  int S;       // segments = B * Hkv * NRB
  int rows_pad;// rows per segment slot in the partial buffers
  int use_tc;  // tcgen05 kernels (bf16, D 128): 1 = rows on TMEM lanes (more than 64
              // packed rows), 2 = keys on TMEM lanes (at most 64), 3 = rows on TMEM
              // lanes, two M-tiles of 128-key TMA tiles (more than 128 rows, dense or
              // paged with pages of 8 rows or more); 0 = mma.sync kernel
  int cps;     // CTAs of the attention kernel resident per SM (1 or 2)
  float scale;
  va_dtype dtype;
  int layout;  // va_layout
  // inputs
  const void *q, *k, *v;
  int len_cap;  // dense/sparse: max_cache_len; paged: max_pages * page_size
  int num_pages, page_shift, max_pages;
  int tma_box;  // rows of one TMA box of the cache (dense 64; paged: the page size, at
                // most 64); 0 = rows gathered with 16-byte cp.async (sparse, pages below 8 rows)
  const int32_t *page_table;
  const int32_t *seqlens;
  const int32_t *indices, *n_indices;
  int max_indices;
  const int32_t *parent;
  const uint32_t *mask;
  int mask_words;
  // rotary embedding on the fly: positions [B][T] (NULL: q and the draft keys
  // are used as stored) and base^(-2i/D) split into fp32 high and low parts
  const int32_t *positions;
  float rope_fhi[64], rope_flo[64];
  // outputs
  void *out;
  int out_align16;  // out is 16-byte aligned (bulk copies allowed)
  float *lse;
  // workspace
  int *status;
  int2 *meta;
  int4 *split_list;              // segments cut over several CTAs: {segment, first slot, parts, 0}
  int *split_count, *split_done;  // list length; merge blocks done (header words)
  int2 *merge_cnt;                // per segment: in-kernel merge counter (.x)
  float *lse_part, *o_part;
  uint64_t wait_ns;
  int test_drop_part;  // test hook: this CTA's parts of split segments never arrive (-1: off)
};

size_t attn_smem_required(const AttnParams &p);
size_t attn_tc_smem_required(const AttnParams &p);
cudaError_t launch_attention_tc(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                                cudaStream_t stream);
size_t attn_tck_smem_required(const AttnParams &p);
size_t attn_tcp_smem_required(const AttnParams &p);
// the two-M-tile kernel merges its split segments itself (cooperative launch)
cudaError_t launch_attention_tcp(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                                 cudaStream_t stream);
// the keys-on-lanes kernel merges split segments itself (cooperative launch)
cudaError_t launch_attention_tck(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                                 cudaStream_t stream);
cudaError_t launch_attention(const AttnParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                             cudaStream_t stream);
cudaError_t launch_combine_generic(int n_rows, int n_parts, int D, const float *o_parts, const float *lse_parts,
                                   va_dtype out_dtype, void *out, float *lse, cudaStream_t stream);
cudaError_t launch_tree_mask(int B, int T, const int32_t *parent, uint32_t *mask, int *status, cudaStream_t stream);
cudaError_t launch_build_index(int B, int Hkv, const int32_t *seqlens, const float *score_draft,
                               const float *score_target, int score_stride, int n_sink, int window, int m_draft,
                               int budget, int32_t *indices, int32_t *n_indices, int *status, bool radix_only,
                               cudaStream_t stream);
cudaError_t launch_wait_selftest(int *status, uint64_t wait_ns, cudaStream_t stream);
cudaError_t launch_validate_index(int B, int Hkv, const int32_t *seqlens, const int32_t *indices,
                                  const int32_t *n_indices, int max_indices, int len_cap, int T, int *status,
                                  cudaStream_t stream);

}  // namespace va
