// Launcher of the head-importance scoring pass (va_score.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace va {

constexpr int kScoreChunk = 128;     // keys per CTA of the score pass (4 warps x 32 keys)
constexpr int kScoreChunk2 = 1024;   // keys per CTA of the reduction pass (256 threads x 4 keys)
constexpr int kScoreUnitRows = 8;    // query rows of one kv-head per MMA unit (the N side)
constexpr int kScoreMaxHeads = 32;   // listed query heads
constexpr int kScoreMaxRows = 256;   // listed heads x T
constexpr int kScoreMaxUnits = 64;   // >= Hkv-groups + rows / 8 for 32 heads and 256 rows

struct ScoreParams {
  int B, T, Hq, Hkv;             // D = 128, bf16
  int max_cache_len;
  float scale_log2;              // score scale x log2(e): scores are kept in base-2 units
  const __nv_bfloat16 *q;        // [B][T][Hq][128]
  const __nv_bfloat16 *k;        // [B][max_cache_len][Hkv][128]
  const int32_t *seqlens;        // [B]
  int R;                         // rows = listed heads x T
  int n_units;
  int n_chunks;                  // ceil(max_cache_len / kScoreChunk)
  int lpad;                      // n_chunks * kScoreChunk: row stride of the score scratch
  float *logits;                 // scratch [B][R][lpad]
  float2 *part;                  // scratch [B][n_chunks][R]: (max, sum of 2^(s - max)) per chunk
  float *score;                  // [B][Hkv][score_stride]
  int score_stride;
  int score_vec4;                // score 16-byte aligned and stride % 4 == 0
  int *status;                   // may be nullptr
  // unit u: kv-head unit_kvh[u], rows unit_row0[u] .. unit_row0[u] + unit_n[u] - 1
  int16_t unit_kvh[kScoreMaxUnits];
  int16_t unit_row0[kScoreMaxUnits];
  int8_t unit_n[kScoreMaxUnits];
  // row r: query head row_head[r] of draft token row_t[r]
  int16_t row_head[kScoreMaxRows];
  int8_t row_t[kScoreMaxRows];
};

// Scratch bytes for B sequences, R rows and caches of max_cache_len slots.
size_t score_scratch_bytes(int B, int R, int max_cache_len);

cudaError_t launch_head_importance(const ScoreParams &p, cudaStream_t stream);

}  // namespace va
