// Shared device-side helpers of libverify_attn: PTX wrappers (mbarrier, bulk
// copies, ldmatrix, mma), bounded waits that record a status instead of
// hanging, the workspace layout and the stream-K work plan.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "verify_attn.h"

namespace va {

// ---------------------------------------------------------------------------
// workspace layout (all offsets 256-byte aligned)
//   [0, 256)            header: int status word (first device-side error) at 0,
//                       split-list length at kSplitCountOff, merge-blocks-done
//                       count at kSplitDoneOff (both back to 0 after every merge)
//   mcnt   int2[kMaxSegments]  per segment: the in-kernel merge counter (x;
//                       back to 0 at the end of every call).  At a fixed offset
//                       for every shape, so one workspace serves calls of any
//                       shape it is large enough for.
//   meta   int2[S]      per segment: first partial slot, number of parts
//   split  int4[slots]  segments cut over more than one CTA (the merge's work
//                       list): segment, first partial slot, number of parts
//   lse_p  f32 [slots][rows_pad]
//   o_p    f32 [slots][rows_pad][D]
// The header and the counters are the bookkeeping that must start at zero
// (kBookkeepingBytes); everything after it is written before it is read.
// ---------------------------------------------------------------------------
constexpr size_t kHeaderBytes = 256;
constexpr size_t kSplitCountOff = 64;
constexpr size_t kSplitDoneOff = 128;
constexpr int kMaxSegments = 2048;

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr size_t kMergeCntOff = kHeaderBytes;
constexpr size_t kBookkeepingBytes = kMergeCntOff + ((sizeof(int2) * (size_t)kMaxSegments + 255) & ~size_t(255));

struct WsLayout {
  size_t meta_off, split_off, mcnt_off, lse_off, o_off, total;
};

__host__ __device__ inline WsLayout ws_layout(int S, int slots, int rows_pad, int D) {
  WsLayout w;
  w.mcnt_off = kMergeCntOff;
  w.meta_off = kBookkeepingBytes;
  w.split_off = w.meta_off + align256(sizeof(int2) * (size_t)S);
  w.lse_off = w.split_off + align256(sizeof(int4) * (size_t)slots);
  w.o_off = w.lse_off + align256(sizeof(float) * (size_t)slots * rows_pad);
  w.total = w.o_off + align256(sizeof(float) * (size_t)slots * rows_pad * D);
  return w;
}

// ---------------------------------------------------------------------------
// status word
// ---------------------------------------------------------------------------
__device__ __forceinline__ void record_status(int *status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// small PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most
// `limit_ns`.  Returns false when the limit ran out (nothing is recorded here;
// the caller records VA_ERR_TIMEOUT and unwinds).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Wait of a pipeline role that may have to give up: a phase already complete
// is taken at once; otherwise the role first checks whether another role has
// given up (abort_flag), then waits at most limit_ns, recording
// VA_ERR_TIMEOUT and raising abort_flag when that runs out.  ok turns false
// when the role stops waiting; a role with ok false waits for nothing.
__device__ __forceinline__ void role_wait(uint64_t *bar, uint32_t parity, bool &ok, volatile int *abort_flag,
                                          uint64_t limit_ns, int *status) {
  if (!ok || mbar_try_wait(bar, parity)) return;
  if (*abort_flag) {
    ok = false;
  } else if (!mbar_wait(bar, parity, limit_ns)) {
    record_status(status, VA_ERR_TIMEOUT);
    *abort_flag = 1;
    ok = false;
  }
}

// One tiled TMA box of a 3-D tensor map (coordinates innermost first) into
// shared memory, completing its bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int c0, int c1, int c2, uint64_t *bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 16-byte global -> shared copy (L1 bypass); src_bytes = 0 fills the 16 bytes
// with zeros without reading global memory.
__device__ __forceinline__ void cp_async_16(void *dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Bulk copy shared -> global (16-byte aligned addresses, size a multiple of
// 16), tracked as a bulk group of the issuing thread.
__device__ __forceinline__ void bulk_store_s2g(void *gdst, const void *ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the sources of this thread's bulk groups have been read (the shared memory may be reused)
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk groups have completed (their global writes are performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// L2 policy: data streamed once (KV rows) is marked evict-first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
// (not volatile: a pure register operation the compiler may schedule freely)
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// 2^x by the PTX approximate base-2 exponential (flushes subnormal results to
// zero; relative error ~2^-22, far below the bf16 rounding P gets afterwards).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (one instruction for both lanes of the pair on sm_100+).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// Largest of three (one instruction on sm_100+).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Split two fp32 values into bf16 hi and lo parts (x ~= hi + lo to ~2^-16
// relative), packed as bf16x2 registers for an mma A operand.
__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t &hi, uint32_t &lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 d = sub2(make_float2(x, y), __bfloat1622float2(h));  // both residuals exact
  __nv_bfloat162 l = __floats2bfloat162_rn(d.x, d.y);
  hi = *reinterpret_cast<uint32_t *>(&h);
  lo = *reinterpret_cast<uint32_t *>(&l);
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Block-wide OR of a predicate over the `n` threads of named barrier `id`
// (also a barrier for them).
__device__ __forceinline__ bool bar_red_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Programmatic dependent launch controls.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace va
