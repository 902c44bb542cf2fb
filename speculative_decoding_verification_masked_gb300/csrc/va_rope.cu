// Rotary position embedding of the draft block, in place (LongSpec, section
// 1: the target model keeps its own RoPE base, and position ids need not be
// consecutive -- e.g. the anchor-offset ids 0, 1, 2, 3, 8192, 8193, ...).
//
// One 128-thread block per (draft token t, sequence b) rotates every query
// head of q[b][t] and the key row of every kv-head at logical slot L_b + t
// of the cache, at the angle positions[b][t] * base^(-2i/D) for the pair
// (i, i + D/2) (rotate-half layout).  The inverse frequencies base^(-2i/D)
// come from the host in fp64; each angle is formed and reduced modulo 2 pi in
// fp64 (five fp64 operations, a Cody-Waite reduction with 2 pi in two parts),
// so that ids far beyond 2^24 radians of phase
// keep their precision; sine and cosine of the reduced angle are taken in fp32 and
// shared by all rows of the token through shared memory.  Rows are rotated
// in fp32 and written back in their own element type (bf16: round to nearest
// even).  When D is a multiple of 16 and the rows are 16-byte aligned, a
// thread takes items of eight pairs and issues the loads of up to four items
// before it writes any; otherwise it rotates one pair at a time.
#include <math.h>

#include "va_common.cuh"
#include "va_rope.h"

namespace va {

template <typename T>
__device__ __forceinline__ float rope_load(const T *p);
template <>
__device__ __forceinline__ float rope_load<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float rope_load<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void rope_store(T *p, float v);
template <>
__device__ __forceinline__ void rope_store<float>(float *p, float v) { *p = v; }
template <>
__device__ __forceinline__ void rope_store<__nv_bfloat16>(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// Address of the key row of kv-head h at logical slot `slot` of sequence b;
// nullptr (recorded) when a page entry is out of range.
template <typename T>
__device__ __forceinline__ T *rope_key_row(const RopeParams &p, int b, int slot, int h) {
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
  return static_cast<T *>(p.k) + (row * p.Hkv + h) * (size_t)p.D;
}

// Rotate pairs i0 .. i0 + 7 of row x (elements i and i + D/2): the eight low
// and eight high elements arrive as two 16-byte (bf16) or 32-byte (fp32)
// vector loads, issued for all of a thread's rows before any is written.
template <typename T>
struct RopeVec;
template <>
struct RopeVec<__nv_bfloat16> {
  uint4 v;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) { v = *reinterpret_cast<const uint4 *>(p); }
  __device__ __forceinline__ void store(__nv_bfloat16 *p) const { *reinterpret_cast<uint4 *>(p) = v; }
};
template <>
struct RopeVec<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float *p) {
    a = *reinterpret_cast<const float4 *>(p);
    b = *reinterpret_cast<const float4 *>(p + 4);
  }
  __device__ __forceinline__ void store(float *p) const {
    *reinterpret_cast<float4 *>(p) = a;
    *reinterpret_cast<float4 *>(p + 4) = b;
  }
};

__device__ __forceinline__ void rope_unpack(const RopeVec<__nv_bfloat16> &r, float (&f)[8]) {
  const uint32_t w[4] = {r.v.x, r.v.y, r.v.z, r.v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}
__device__ __forceinline__ void rope_pack(RopeVec<__nv_bfloat16> &r, const float (&f)[8]) {
  r.v = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
}
__device__ __forceinline__ void rope_unpack(const RopeVec<float> &r, float (&f)[8]) {
  f[0] = r.a.x; f[1] = r.a.y; f[2] = r.a.z; f[3] = r.a.w;
  f[4] = r.b.x; f[5] = r.b.y; f[6] = r.b.z; f[7] = r.b.w;
}
__device__ __forceinline__ void rope_pack(RopeVec<float> &r, const float (&f)[8]) {
  r.a = make_float4(f[0], f[1], f[2], f[3]);
  r.b = make_float4(f[4], f[5], f[6], f[7]);
}

template <typename T>
__global__ void __launch_bounds__(128) rope_draft_kernel(const RopeParams p) {
  __shared__ float cs[128], sn[128];
  __shared__ T *krow[256];  // key rows of this token (nullptr: left alone)
  const int t = blockIdx.x, b = blockIdx.y;
  const int half = p.D / 2;
  const int tid = threadIdx.x;
  const int pos = __ldg(p.positions + (size_t)b * p.T + t);
  const int L = __ldg(p.seqlens + b);
  const bool kv_ok = L >= 0 && L <= p.len_cap - p.T;
  if (!kv_ok && t == 0 && tid == 0) record_status(p.status, VA_ERR_DEVICE_BOUNDS);
  for (int i = tid; i < half; i += blockDim.x) {
    // a_i = pos * base^(-2i/D), reduced to [-pi, pi] in fp64 by the Cody-Waite
    // method: k = rint(a / 2pi), r = (a - k C1) - k C2 with 2 pi split into its
    // fp64 rounding C1 and the fp64 rounding C2 of the remainder 2pi - C1
    // (values of 2 pi and 1 / 2pi to 17 significant digits)
    const double a = (double)pos * p.inv_freq[i];
    const double kq = rint(a * 0.15915494309189535);
    const double r = fma(-kq, 2.4492935982947064e-16, fma(-kq, 6.283185307179586, a));
    float s, c;
    sincosf((float)r, &s, &c);
    cs[i] = c;
    sn[i] = s;
  }
  for (int h = tid; h < p.Hkv; h += blockDim.x) krow[h] = kv_ok ? rope_key_row<T>(p, b, L + t, h) : nullptr;
  __syncthreads();
  T *qrow = static_cast<T *>(p.q) + ((size_t)b * p.T + t) * p.Hq * (size_t)p.D;
  const int rows = p.Hq + p.Hkv;
  if (p.vec8) {
    // items of 8 pairs: (row, i0 = 8 c); up to kItems per thread, loads first
    constexpr int kItems = 4;
    const int per_row = half / 8;
    const int n_items = rows * per_row;
    for (int e0 = tid; e0 < n_items; e0 += kItems * blockDim.x) {
      RopeVec<T> lo[kItems], hi[kItems];
      T *xs[kItems];
#pragma unroll
      for (int u = 0; u < kItems; ++u) {
        const int e = e0 + u * blockDim.x;
        xs[u] = nullptr;
        if (e < n_items) {
          const int row = e / per_row, i0 = (e % per_row) * 8;
          T *x = row < p.Hq ? qrow + (size_t)row * p.D : krow[row - p.Hq];
          if (x != nullptr) {
            xs[u] = x + i0;
            lo[u].load(x + i0);
            hi[u].load(x + i0 + half);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kItems; ++u) {
        if (xs[u] == nullptr) continue;
        const int i0 = ((e0 + u * (int)blockDim.x) % per_row) * 8;
        float fl[8], fh[8], ol[8], oh[8];
        rope_unpack(lo[u], fl);
        rope_unpack(hi[u], fh);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float c = cs[i0 + j], s = sn[i0 + j];
          ol[j] = fmaf(fl[j], c, -fh[j] * s);
          oh[j] = fmaf(fh[j], c, fl[j] * s);
        }
        rope_pack(lo[u], ol);
        rope_pack(hi[u], oh);
        lo[u].store(xs[u]);
        hi[u].store(xs[u] + half);
      }
    }
  } else {
    for (int e = tid; e < rows * half; e += blockDim.x) {
      const int row = e / half, i = e % half;
      T *x = row < p.Hq ? qrow + (size_t)row * p.D : krow[row - p.Hq];
      if (x == nullptr) continue;
      const float lo = rope_load(x + i), hi = rope_load(x + i + half);
      const float c = cs[i], s = sn[i];
      rope_store(x + i, fmaf(lo, c, -hi * s));
      rope_store(x + i + half, fmaf(hi, c, lo * s));
    }
  }
}

cudaError_t launch_rope_draft(const RopeParams &p, cudaStream_t stream) {
  const dim3 grid((unsigned)p.T, (unsigned)p.B);
  if (p.fp32)
    rope_draft_kernel<float><<<grid, 128, 0, stream>>>(p);
  else
    rope_draft_kernel<__nv_bfloat16><<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace va
