// Rotary position embedding applied inside the attention kernels (LongSpec,
// section 1: the target model keeps its own RoPE base; position ids may be
// arbitrary, e.g. anchor-offset ids).  When a call passes the draft tokens'
// positions, q and the T draft keys are rotated on the fly -- q while it is
// loaded for a segment, the draft keys in the landed K tile before the first
// MMA (or consumer) reads it -- and neither q nor the cache is written.
//
// Layout: rotate-half (element i pairs with i + D/2, i < D/2), angle
// positions[b][t] * base^(-2i/D).  The inverse frequencies come from the host
// in fp64, split into an fp32 high part and the fp32 rounding of the rest.
// Each segment builds a table of (cos, sin) for its sequence's T tokens and
// D/2 frequencies in shared memory; every rotated row reads it.
//
// Angle reduction (Cody-Waite): with p = positions[b][t] exact in fp32
// (|p| < 2^24) and f = f_hi + f_lo,
//   a_hi = fl(p f_hi),  e = p f_hi - a_hi (exact, one FMA),
//   k = rint(a_hi / 2pi),
//   r = ((a_hi - k C1) - k C2) + (e + p f_lo),
// where C1 is 2pi rounded to fp32 and C2 the fp32 rounding of 2pi - C1; the
// two FMAs with C1 and C2 each round a result below 4.2 in magnitude, so r is
// the angle modulo 2pi to about 5e-7 rad for every |p| < 2^24 (an fp32
// product alone would be off by up to a radian there).  sin and cos of r are
// then the library's sincosf.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "va_common.cuh"
#include "va_kernels.h"

namespace va {

constexpr double kTwoPiD = 6.283185307179586476925286766559;
constexpr float kTwoPiC1 = (float)kTwoPiD;                     // 2 pi rounded to fp32
constexpr float kTwoPiC2 = (float)(kTwoPiD - (double)kTwoPiC1);  // the fp32 rounding of the rest
constexpr float kInvTwoPi = (float)(1.0 / kTwoPiD);
constexpr int kRopeMaxPos = 1 << 24;  // |positions| below this (exact in fp32)

__device__ __forceinline__ float2 rope_cos_sin(int pos, float f_hi, float f_lo) {
  const float pf = (float)pos;
  const float a_hi = pf * f_hi;
  const float e = fmaf(pf, f_hi, -a_hi);
  const float k = rintf(a_hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiC1, a_hi);
  r = fmaf(-k, kTwoPiC2, r);
  r += e + pf * f_lo;
  float s, c;
  sincosf(r, &s, &c);
  return make_float2(c, s);
}

// Bytes of the per-segment table (0 when the call rotates nothing).
__host__ __device__ inline int rope_table_bytes(const AttnParams &p) {
  return p.positions != nullptr ? ((p.T * (p.D / 2) * 8 + 15) & ~15) : 0;
}

// (cos, sin) of token t and frequency i at tab[t * (D/2) + i], for sequence
// b, built by threads [0, nthreads) of the block (callers synchronise after).
// A position outside (-2^24, 2^24) is recorded as VA_ERR_DEVICE_BOUNDS and
// taken as 0.
__device__ __forceinline__ void rope_build_table(const AttnParams &p, int b, float2 *tab, int tid, int nthreads) {
  const int half = p.D / 2;
  const int n = p.T * half;
  for (int e = tid; e < n; e += nthreads) {
    const int t = e / half, i = e - t * half;
    int pos = __ldg(p.positions + (size_t)b * p.T + t);
    if (pos <= -kRopeMaxPos || pos >= kRopeMaxPos) {
      if (i == 0) record_status(p.status, VA_ERR_DEVICE_BOUNDS);
      pos = 0;
    }
    tab[e] = rope_cos_sin(pos, p.rope_fhi[i], p.rope_flo[i]);
  }
}

// x' = x cos - y sin, y' = y cos + x sin for the 8 pairs held in two 16-byte
// chunks of bf16 (lo: elements i..i+7, hi: i+D/2..i+D/2+7), rounded back to
// bf16 to nearest even.
__device__ __forceinline__ void rope_rotate8_bf16(uint4 &lo, uint4 &hi, const float2 *cs) {
  uint32_t *a = reinterpret_cast<uint32_t *>(&lo);
  uint32_t *b = reinterpret_cast<uint32_t *>(&hi);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&a[j]));
    const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&b[j]));
    const float2 c0 = cs[2 * j], c1 = cs[2 * j + 1];
    const float x0 = x.x * c0.x - y.x * c0.y, y0 = y.x * c0.x + x.x * c0.y;
    const float x1 = x.y * c1.x - y.y * c1.y, y1 = y.y * c1.x + x.y * c1.y;
    a[j] = pack_bf16(x0, x1);
    b[j] = pack_bf16(y0, y1);
  }
}

// The same for 4 pairs of fp32 (one 16-byte chunk each).
__device__ __forceinline__ void rope_rotate4_f32(float4 &lo, float4 &hi, const float2 *cs) {
  float *x = reinterpret_cast<float *>(&lo);
  float *y = reinterpret_cast<float *>(&hi);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float xv = x[j], yv = y[j];
    x[j] = xv * cs[j].x - yv * cs[j].y;
    y[j] = yv * cs[j].x + xv * cs[j].y;
  }
}

// Rotate key rows [r0, r1) of a K tile in shared memory (layout of the stage
// ring: 128-byte columns of TK rows, 16-byte chunks XOR-swizzled by row % 8),
// row r holding draft token t0 + r - r0, by `nthreads` threads of index tid.
// The caller orders these stores before the tile's readers.
template <typename Tin, int D, int TK>
__device__ __forceinline__ void rope_rotate_tile_rows(uint8_t *tile, int r0, int r1, int t0, const float2 *tab,
                                                      int tid, int nthreads) {
  constexpr int kChunks = D * (int)sizeof(Tin) / 16;  // 16-byte chunks per row
  constexpr int kHalf = kChunks / 2;                  // a chunk's partner, D/2 elements on
  constexpr int kPer = 16 / (int)sizeof(Tin);         // elements per chunk
  const int n = (r1 - r0) * kHalf;
  for (int e = tid; e < n; e += nthreads) {
    const int r = r0 + e / kHalf, c = e % kHalf;
    const float2 *cs = tab + (size_t)(t0 + r - r0) * (D / 2) + c * kPer;
    uint8_t *plo = tile + (c >> 3) * (TK * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
    uint8_t *phi = tile + ((c + kHalf) >> 3) * (TK * 128) + r * 128 + ((((c + kHalf) & 7) ^ (r & 7)) << 4);
    if constexpr (sizeof(Tin) == 2) {
      uint4 lo = *reinterpret_cast<uint4 *>(plo), hi = *reinterpret_cast<uint4 *>(phi);
      rope_rotate8_bf16(lo, hi, cs);
      *reinterpret_cast<uint4 *>(plo) = lo;
      *reinterpret_cast<uint4 *>(phi) = hi;
    } else {
      float4 lo = *reinterpret_cast<float4 *>(plo), hi = *reinterpret_cast<float4 *>(phi);
      rope_rotate4_f32(lo, hi, cs);
      *reinterpret_cast<float4 *>(plo) = lo;
      *reinterpret_cast<float4 *>(phi) = hi;
    }
  }
}

// The same for bf16 tiles as an out-of-line call: a caller whose hot loop
// would otherwise carry the rotation inline (the tcgen05 MMA issuer) keeps
// that loop short.
template <int D, int TK>
__device__ __noinline__ void rope_rotate_tile_rows_bf16_call(uint8_t *tile, int r0, int r1, int t0, const float2 *tab,
                                                            int tid, int nthreads) {
  rope_rotate_tile_rows<__nv_bfloat16, D, TK>(tile, r0, r1, t0, tab, tid, nthreads);
}

}  // namespace va
