// C ABI of libverify_attn: argument validation, workspace planning, launches,
// device status and error reporting.  See include/verify_attn.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>

#include "va_common.cuh"
#include "va_kernels.h"
#include "va_commit.h"
#include "va_score.h"
#include "va_rope.h"
#include "verify_attn_testing.h"

namespace {

thread_local std::string g_last_error;

va_status fail(va_status code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
va_status fail(va_status code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

va_status ok() {
  g_last_error.clear();
  return VA_OK;
}

va_status cuda_fail(cudaError_t e, const char *what) {
  return fail(VA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

using va::kMaxSegments;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s per bounded wait

uint64_t wait_limit_ns() {
  static uint64_t v = [] {
    const char *s = getenv("VA_WAIT_LIMIT_NS");
    if (s != nullptr && *s) {
      const unsigned long long x = strtoull(s, nullptr, 10);
      if (x > 0) return (uint64_t)x;
    }
    return kDefaultWaitNs;
  }();
  return v;
}

// Test hook (verify_attn_testing.h): a wait limit and a dropped part for the
// next attention calls of the process.
std::atomic<unsigned long long> g_test_wait_ns{0};
std::atomic<int> g_test_drop_part{-1};
std::atomic<int> g_test_index_radix{0};  // verify_attn_test_index_path

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// VA_DEBUG_VALIDATE=1: check inputs on the device that the fast path trusts
// (read at every call, so a test may switch it per call)
bool debug_validate() {
  const char *e = getenv("VA_DEBUG_VALIDATE");
  return e != nullptr && strcmp(e, "1") == 0;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over a cache of rows [rows][Hkv][D] (dense: rows = B * len; paged:
// rows = num_pages * page_size): boxes of box_rows tokens x one kv-head x 128
// bytes of the head dimension, 128-byte swizzled.
bool encode_cache_map(CUtensorMap *m, const void *base, va_dtype dt, int D, int Hkv, long long rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint32_t es = dt == VA_DTYPE_BF16 ? 2 : 4;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)Hkv * D * es};
  const cuuint32_t box[3] = {128 / es, 1, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, dt == VA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                   const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int device_sm_count(int *dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  static std::mutex mu;
  static int cache[64] = {0};
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return -1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cache[dev] = n;
  }
  if (dev_out) *dev_out = dev;
  return cache[dev];
}

// Row blocking of the packed (group * T) query rows of one kv-head.
struct RowPlan {
  int R, RG, NRB, rows_pad, S, use_tc, cps;
};

// Kernel choice and row blocking.  More than 64 packed rows (bf16, D 128) go to
// the tcgen05 kernel in blocks of up to 256 rows (two 128-row M-tiles); the
// rest to the mma.sync kernel in blocks of 16, 32 or 64 rows.
// The keys-on-lanes tcgen05 kernel serves bf16 d128 segments of at most 64
// rows; VA_SMALL_ROWS_KERNEL=mma selects the mma.sync kernel for them instead.
bool tck_enabled() {
  const char *e = getenv("VA_SMALL_ROWS_KERNEL");
  return !(e != nullptr && strcmp(e, "mma") == 0);
}

RowPlan row_plan(const va_shape &s) {
  RowPlan r;
  r.R = (s.Hq / s.Hkv) * s.T;
  r.use_tc = 0;
  if (s.dtype == VA_DTYPE_FP32) {
    r.RG = 4;
    r.rows_pad = 64;
  } else if (s.D == 128 && r.R > 64) {
    r.use_tc = 1;
    r.RG = 4;
    r.rows_pad = r.R > 128 ? 256 : 128;
  } else if (s.D == 128 && tck_enabled()) {
    r.use_tc = 2;
    r.RG = 4;
    r.rows_pad = r.R <= 16 ? 16 : (r.R <= 32 ? 32 : 64);
  } else {
    r.RG = r.R <= 16 ? 1 : (r.R <= 32 ? 2 : 4);
    r.rows_pad = 16 * r.RG;
  }
  r.NRB = (r.R + r.rows_pad - 1) / r.rows_pad;
  r.S = s.B * s.Hkv * r.NRB;
  // two CTAs per SM for the mma.sync kernel with small per-warp state
  r.cps = (!r.use_tc && s.dtype == VA_DTYPE_BF16 && r.RG <= 2) ? 2 : 1;
  return r;
}

va_status check_shape(const va_shape *s) {
  if (s == nullptr) return fail(VA_ERR_INVALID_ARG, "shape is NULL");
  if (s->B < 1 || s->T < 1 || s->Hq < 1 || s->Hkv < 1 || s->D < 1)
    return fail(VA_ERR_INVALID_ARG, "shape has a non-positive size (B=%d T=%d Hq=%d Hkv=%d D=%d)", s->B, s->T,
                s->Hq, s->Hkv, s->D);
  if (s->Hq % s->Hkv != 0) return fail(VA_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", s->Hq, s->Hkv);
  if (s->dtype != VA_DTYPE_BF16 && s->dtype != VA_DTYPE_FP32)
    return fail(VA_ERR_INVALID_ARG, "unknown dtype %d", (int)s->dtype);
  if (!(s->scale > 0.f) || !isfinite(s->scale)) return fail(VA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (s->T > 64) return fail(VA_ERR_UNSUPPORTED, "T=%d draft tokens; at most 64 are supported", s->T);
  if (s->dtype == VA_DTYPE_BF16 && s->D != 64 && s->D != 128)
    return fail(VA_ERR_UNSUPPORTED, "bf16 supports D in {64, 128}, got %d", s->D);
  if (s->dtype == VA_DTYPE_FP32 && s->D != 64) return fail(VA_ERR_UNSUPPORTED, "fp32 supports D = 64, got %d", s->D);
  const RowPlan rp = row_plan(*s);
  if ((long long)s->B * s->Hkv * rp.NRB > kMaxSegments)
    return fail(VA_ERR_UNSUPPORTED, "B*Hkv*row_blocks = %lld exceeds %d", (long long)s->B * s->Hkv * rp.NRB,
                kMaxSegments);
  return VA_OK;
}

size_t workspace_bytes(const va_shape &s, int sm_count) {
  const RowPlan rp = row_plan(s);
  const int slots = rp.S + rp.cps * sm_count;  // one partial slot per (segment, CTA) boundary
  return va::ws_layout(rp.S, slots, rp.rows_pad, s.D).total;
}

struct Common {
  const va_shape *shape;
  const void *q;
  const int32_t *seqlens, *parent;
  const uint32_t *mask;
  const int32_t *positions;
  void *out;
  float *lse;
  void *ws;
  size_t ws_bytes;
};

va_status check_common(const Common &c) {
  va_status st = check_shape(c.shape);
  if (st != VA_OK) return st;
  if (c.q == nullptr || c.seqlens == nullptr || c.out == nullptr || c.lse == nullptr)
    return fail(VA_ERR_INVALID_ARG, "q, seqlens, out and lse must not be NULL");
  if (c.parent != nullptr && c.mask != nullptr)
    return fail(VA_ERR_INVALID_ARG, "give tree_parent or tree_mask, not both");
  if (c.positions != nullptr && (!(c.shape->rope_base > 0.f) || !isfinite(c.shape->rope_base)))
    return fail(VA_ERR_INVALID_ARG, "rotating on the fly (positions given) needs shape->rope_base > 0");
  const size_t el = c.shape->dtype == VA_DTYPE_BF16 ? 2 : 4;
  const size_t out_align = el == 2 ? 8 : 4;
  if (!aligned(c.q, 16) || !aligned(c.out, out_align))
    return fail(VA_ERR_INVALID_ARG, "q must be 16-byte aligned and out %zu-byte aligned", out_align);
  if (c.ws == nullptr) return fail(VA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(c.ws, 256)) return fail(VA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  return VA_OK;
}

va_status run_attention(const Common &c, int layout, const void *k, const void *v, int len_cap, int num_pages,
                        int page_size, const int32_t *page_table, int max_pages, const int32_t *indices,
                        const int32_t *n_indices, int max_indices, cudaStream_t stream) {
  const va_shape &s = *c.shape;
  int dev = 0;
  const int sms = device_sm_count(&dev);
  if (sms <= 0) return fail(VA_ERR_CUDA, "no usable CUDA device");
  const size_t need = workspace_bytes(s, sms);
  if (c.ws_bytes < need)
    return fail(VA_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", c.ws_bytes, need);
  const RowPlan rp = row_plan(s);

  va::AttnParams p;
  memset(&p, 0, sizeof p);
  p.B = s.B;
  p.T = s.T;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.D = s.D;
  p.R = rp.R;
  p.RG = rp.RG;
  p.NRB = rp.NRB;
  p.S = rp.S;
  p.rows_pad = rp.rows_pad;
  p.use_tc = rp.use_tc;
  p.cps = rp.cps;
  p.scale = s.scale;
  p.dtype = s.dtype;
  p.layout = layout;
  p.q = c.q;
  p.k = k;
  p.v = v;
  p.len_cap = len_cap;
  p.num_pages = num_pages;
  p.page_shift = 0;
  while ((1 << p.page_shift) < page_size) ++p.page_shift;
  p.max_pages = max_pages;
  p.page_table = page_table;
  p.seqlens = c.seqlens;
  p.indices = indices;
  p.n_indices = n_indices;
  p.max_indices = max_indices;
  p.parent = c.parent;
  p.mask = c.mask;
  p.mask_words = (s.T + 31) / 32;
  p.positions = c.positions;
  if (c.positions != nullptr) {
    for (int i = 0; i < s.D / 2; ++i) {
      const double f = pow((double)s.rope_base, -(double)(2 * i) / s.D);
      p.rope_fhi[i] = (float)f;
      p.rope_flo[i] = (float)(f - (double)p.rope_fhi[i]);
    }
  }
  p.out = c.out;
  p.out_align16 = aligned(c.out, 16) ? 1 : 0;
  p.lse = c.lse;
  const va::WsLayout wl = va::ws_layout(rp.S, rp.S + rp.cps * sms, rp.rows_pad, s.D);
  uint8_t *ws = static_cast<uint8_t *>(c.ws);
  p.status = reinterpret_cast<int *>(ws);
  p.meta = reinterpret_cast<int2 *>(ws + wl.meta_off);
  p.split_list = reinterpret_cast<int4 *>(ws + wl.split_off);
  p.split_count = reinterpret_cast<int *>(ws + va::kSplitCountOff);
  p.split_done = reinterpret_cast<int *>(ws + va::kSplitDoneOff);
  p.merge_cnt = reinterpret_cast<int2 *>(ws + wl.mcnt_off);
  p.lse_part = reinterpret_cast<float *>(ws + wl.lse_off);
  p.o_part = reinterpret_cast<float *>(ws + wl.o_off);
  p.wait_ns = wait_limit_ns();
  p.test_drop_part = g_test_drop_part.load();
  if (const unsigned long long tw = g_test_wait_ns.load()) p.wait_ns = tw;

  CUtensorMap tmk, tmv;
  memset(&tmk, 0, sizeof tmk);
  memset(&tmv, 0, sizeof tmv);
  if (layout == VA_LAYOUT_DENSE) {
    const long long rows = (long long)s.B * len_cap;
    if (rows >= (1ll << 31)) return fail(VA_ERR_UNSUPPORTED, "B * max_cache_len must be below 2^31");
    if (!encode_cache_map(&tmk, k, s.dtype, s.D, s.Hkv, rows, 64) ||
        !encode_cache_map(&tmv, v, s.dtype, s.D, s.Hkv, rows, 64))
      return fail(VA_ERR_CUDA, "could not encode the TMA tensor maps of the cache");
    p.tma_box = 64;
  } else if (layout == VA_LAYOUT_PAGED && page_size >= 8) {
    // one TMA box per page (at most 64 rows): a box lands on whole 1024-byte
    // swizzle atoms of the stage.  Smaller pages, or a pool the map cannot
    // describe, are gathered with cp.async instead.
    const long long rows = (long long)num_pages * page_size;
    const int box = page_size < 64 ? page_size : 64;
    if (rows < (1ll << 31) && encode_cache_map(&tmk, k, s.dtype, s.D, s.Hkv, rows, box) &&
        encode_cache_map(&tmv, v, s.dtype, s.D, s.Hkv, rows, box))
      p.tma_box = box;
  }
  // more than 128 packed rows with K/V tiles by TMA: VA_MANY_ROWS_KERNEL=tcp
  // selects the two-M-tile kernel of 128-key tiles instead of the 64-key
  // rows-on-lanes kernel
  if (p.use_tc == 1 && p.rows_pad == 256 && p.tma_box > 0) {
    const char *e = getenv("VA_MANY_ROWS_KERNEL");
    if (e != nullptr && strcmp(e, "tcp") == 0) p.use_tc = 3;
  }
  // key tiles an upper bound can produce; the grid never exceeds them
  const long long keys_cap = (layout == VA_LAYOUT_SPARSE) ? (long long)max_indices + s.T : (long long)len_cap;
  const long long tile_keys = p.use_tc >= 2 ? 128 : 64;
  const long long tiles_cap = (long long)rp.S * ((keys_cap + tile_keys - 1) / tile_keys);
  if (tiles_cap >= (1ll << 31)) return fail(VA_ERR_UNSUPPORTED, "problem too large (%lld key tiles)", tiles_cap);
  const long long ctas = (long long)rp.cps * sms;
  const int grid = (int)(tiles_cap < ctas ? tiles_cap : ctas);
  if (va::attn_smem_required(p) > 232448) return fail(VA_ERR_UNSUPPORTED, "shared memory plan too large");
  cudaError_t e = va::launch_attention(p, tmk, tmv, grid < 1 ? 1 : grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return ok();
}

}  // namespace

namespace {
va_status commit_common(const va_shape *shape, void *k, void *v, const int32_t *seqlens, const int32_t *path,
                        const int32_t *n_accept, int32_t *seqlens_out, void *workspace, va::CommitParams &cp) {
  if (shape == nullptr) return fail(VA_ERR_INVALID_ARG, "shape is NULL");
  if (shape->B < 1 || shape->T < 1 || shape->Hkv < 1) return fail(VA_ERR_INVALID_ARG, "B, T and Hkv must be >= 1");
  if (shape->T > 64) return fail(VA_ERR_UNSUPPORTED, "T=%d; at most 64 draft tokens are supported", shape->T);
  if (shape->dtype != VA_DTYPE_BF16 && shape->dtype != VA_DTYPE_FP32)
    return fail(VA_ERR_INVALID_ARG, "unknown dtype %d", (int)shape->dtype);
  const int es = shape->dtype == VA_DTYPE_BF16 ? 2 : 4;
  if (shape->D < 1 || (shape->D * es) % 16 != 0 || shape->D * es > 1024)
    return fail(VA_ERR_UNSUPPORTED, "rows of D=%d elements must be a multiple of 16 bytes, at most 1 KB", shape->D);
  if (k == nullptr || v == nullptr || seqlens == nullptr || path == nullptr || n_accept == nullptr)
    return fail(VA_ERR_INVALID_ARG, "caches, seqlens, path and n_accept must not be NULL");
  if (!aligned(k, 16) || !aligned(v, 16)) return fail(VA_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  if (seqlens_out != nullptr && seqlens_out == seqlens)
    return fail(VA_ERR_INVALID_ARG, "seqlens_out must not alias seqlens");
  if (workspace != nullptr && !aligned(workspace, 256)) return fail(VA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  memset(&cp, 0, sizeof cp);
  cp.B = shape->B;
  cp.T = shape->T;
  cp.Hkv = shape->Hkv;
  cp.row_bytes = shape->D * es;
  cp.k = k;
  cp.v = v;
  cp.seqlens = seqlens;
  cp.path = path;
  cp.n_accept = n_accept;
  cp.seqlens_out = seqlens_out;
  cp.status = static_cast<int *>(workspace);
  return VA_OK;
}

va_status rope_common(const va_shape *shape, void *q, void *k, const int32_t *seqlens, const int32_t *positions,
                      float rope_base, void *workspace, va::RopeParams &rp) {
  if (shape == nullptr) return fail(VA_ERR_INVALID_ARG, "shape is NULL");
  const va_shape &s = *shape;
  if (s.B < 1 || s.T < 1 || s.Hq < 1 || s.Hkv < 1 || s.Hq % s.Hkv != 0)
    return fail(VA_ERR_INVALID_ARG, "bad shape (B=%d T=%d Hq=%d Hkv=%d)", s.B, s.T, s.Hq, s.Hkv);
  if (s.T > 64) return fail(VA_ERR_UNSUPPORTED, "T=%d; at most 64 draft tokens are supported", s.T);
  if (s.B > 65535 || s.Hkv > 256) return fail(VA_ERR_UNSUPPORTED, "B <= 65535 and Hkv <= 256 are supported");
  if (s.dtype != VA_DTYPE_BF16 && s.dtype != VA_DTYPE_FP32) return fail(VA_ERR_INVALID_ARG, "unknown dtype %d", (int)s.dtype);
  if (s.D < 2 || s.D > 256 || s.D % 2 != 0) return fail(VA_ERR_UNSUPPORTED, "D=%d; an even D <= 256 is supported", s.D);
  if (!(rope_base > 0.f) || !isfinite(rope_base)) return fail(VA_ERR_INVALID_ARG, "rope_base must be finite and > 0");
  if (q == nullptr || k == nullptr || seqlens == nullptr || positions == nullptr)
    return fail(VA_ERR_INVALID_ARG, "q, the key cache, seqlens and positions must not be NULL");
  const size_t es = s.dtype == VA_DTYPE_BF16 ? 2 : 4;
  if (!aligned(q, es) || !aligned(k, es)) return fail(VA_ERR_INVALID_ARG, "q and the key cache must be element-aligned");
  if (workspace != nullptr && !aligned(workspace, 256)) return fail(VA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  memset(&rp, 0, sizeof rp);
  rp.B = s.B;
  rp.T = s.T;
  rp.Hq = s.Hq;
  rp.Hkv = s.Hkv;
  rp.D = s.D;
  rp.fp32 = s.dtype == VA_DTYPE_FP32 ? 1 : 0;
  rp.vec8 = s.D % 16 == 0 && aligned(q, 16) && aligned(k, 16) ? 1 : 0;
  for (int i = 0; i < s.D / 2; ++i) rp.inv_freq[i] = pow((double)rope_base, -(double)(2 * i) / s.D);
  rp.q = q;
  rp.k = k;
  rp.seqlens = seqlens;
  rp.positions = positions;
  rp.status = static_cast<int *>(workspace);
  return VA_OK;
}
}  // namespace

extern "C" {

size_t verify_attn_workspace_size(const va_shape *shape) {
  if (check_shape(shape) != VA_OK) return 0;
  const int sms = device_sm_count(nullptr);
  if (sms <= 0) return 0;
  return workspace_bytes(*shape, sms);
}

va_status verify_attn_workspace_init(void *workspace, size_t ws_bytes, va_stream stream) {
  if (workspace == nullptr || ws_bytes < va::kHeaderBytes) return fail(VA_ERR_WORKSPACE, "workspace too small");
  if (!aligned(workspace, 256)) return fail(VA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  // all of it: the status word and the merge counters start at zero (the
  // calls return the counters to zero themselves)
  cudaError_t e = cudaMemsetAsync(workspace, 0, ws_bytes, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "workspace init");
  return ok();
}

va_status verify_attn_dense(const va_shape *shape, const void *q, const void *k_cache, const void *v_cache,
                            int max_cache_len, const int32_t *seqlens, const int32_t *tree_parent,
                            const uint32_t *tree_mask, const int32_t *positions, void *out, float *lse,
                            void *workspace, size_t ws_bytes, va_stream stream) {
  Common c{shape, q, seqlens, tree_parent, tree_mask, positions, out, lse, workspace, ws_bytes};
  va_status st = check_common(c);
  if (st != VA_OK) return st;
  if (k_cache == nullptr || v_cache == nullptr) return fail(VA_ERR_INVALID_ARG, "k_cache and v_cache must not be NULL");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return fail(VA_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  if (max_cache_len < shape->T)
    return fail(VA_ERR_INVALID_ARG, "max_cache_len=%d is smaller than T=%d", max_cache_len, shape->T);
  return run_attention(c, VA_LAYOUT_DENSE, k_cache, v_cache, max_cache_len, 0, 1, nullptr, 0, nullptr, nullptr, 0,
                       (cudaStream_t)stream);
}

va_status verify_attn_paged(const va_shape *shape, const void *q, const void *k_pages, const void *v_pages,
                            int num_pages, int page_size, const int32_t *page_table, int max_pages_per_seq,
                            const int32_t *seqlens, const int32_t *tree_parent, const uint32_t *tree_mask,
                            const int32_t *positions, void *out, float *lse, void *workspace, size_t ws_bytes,
                            va_stream stream) {
  Common c{shape, q, seqlens, tree_parent, tree_mask, positions, out, lse, workspace, ws_bytes};
  va_status st = check_common(c);
  if (st != VA_OK) return st;
  if (k_pages == nullptr || v_pages == nullptr || page_table == nullptr)
    return fail(VA_ERR_INVALID_ARG, "k_pages, v_pages and page_table must not be NULL");
  if (!aligned(k_pages, 16) || !aligned(v_pages, 16)) return fail(VA_ERR_INVALID_ARG, "pages must be 16-byte aligned");
  if (page_size < 1 || page_size > 1024 || (page_size & (page_size - 1)) != 0)
    return fail(VA_ERR_INVALID_ARG, "page_size=%d must be a power of two in [1, 1024]", page_size);
  if (num_pages < 1 || max_pages_per_seq < 1) return fail(VA_ERR_INVALID_ARG, "num_pages and max_pages_per_seq must be >= 1");
  const long long cap = (long long)max_pages_per_seq * page_size;
  if (cap < shape->T) return fail(VA_ERR_INVALID_ARG, "max_pages_per_seq*page_size is smaller than T");
  if (cap >= (1ll << 30)) return fail(VA_ERR_UNSUPPORTED, "max_pages_per_seq*page_size too large");
  return run_attention(c, VA_LAYOUT_PAGED, k_pages, v_pages, (int)cap, num_pages, page_size, page_table,
                       max_pages_per_seq, nullptr, nullptr, 0, (cudaStream_t)stream);
}

va_status verify_attn_sparse(const va_shape *shape, const void *q, const void *k_cache, const void *v_cache,
                             int max_cache_len, const int32_t *seqlens, const int32_t *indices,
                             const int32_t *n_indices, int max_indices, const int32_t *tree_parent,
                             const uint32_t *tree_mask, const int32_t *positions, void *out, float *lse,
                             void *workspace, size_t ws_bytes, va_stream stream) {
  Common c{shape, q, seqlens, tree_parent, tree_mask, positions, out, lse, workspace, ws_bytes};
  va_status st = check_common(c);
  if (st != VA_OK) return st;
  if (k_cache == nullptr || v_cache == nullptr || indices == nullptr || n_indices == nullptr)
    return fail(VA_ERR_INVALID_ARG, "k_cache, v_cache, indices and n_indices must not be NULL");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return fail(VA_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  if (max_cache_len < shape->T)
    return fail(VA_ERR_INVALID_ARG, "max_cache_len=%d is smaller than T=%d", max_cache_len, shape->T);
  if (max_indices < 0) return fail(VA_ERR_INVALID_ARG, "max_indices must be >= 0");
  if (debug_validate()) {
    // validation mode: the verify sets are checked on the device first
    cudaError_t e = va::launch_validate_index(shape->B, shape->Hkv, seqlens, indices, n_indices, max_indices,
                                              max_cache_len, shape->T, static_cast<int *>(workspace),
                                              (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "validation launch");
  }
  return run_attention(c, VA_LAYOUT_SPARSE, k_cache, v_cache, max_cache_len, 0, 1, nullptr, 0, indices, n_indices,
                       max_indices, (cudaStream_t)stream);
}

va_status verify_attn_combine(int n_rows, int n_parts, int D, const float *o_parts, const float *lse_parts,
                              va_dtype out_dtype, void *out, float *lse, va_stream stream) {
  if (n_rows < 0 || n_parts < 1) return fail(VA_ERR_INVALID_ARG, "n_rows must be >= 0 and n_parts >= 1");
  if (D != 64 && D != 128) return fail(VA_ERR_UNSUPPORTED, "D must be 64 or 128, got %d", D);
  if (n_parts > 1024) return fail(VA_ERR_UNSUPPORTED, "at most 1024 parts per merge, got %d", n_parts);
  if (out_dtype != VA_DTYPE_BF16 && out_dtype != VA_DTYPE_FP32) return fail(VA_ERR_INVALID_ARG, "unknown out dtype");
  if (o_parts == nullptr || lse_parts == nullptr || out == nullptr)
    return fail(VA_ERR_INVALID_ARG, "o_parts, lse_parts and out must not be NULL");
  if (!aligned(o_parts, 16)) return fail(VA_ERR_INVALID_ARG, "o_parts must be 16-byte aligned");
  if (n_rows == 0) return ok();
  cudaError_t e =
      va::launch_combine_generic(n_rows, n_parts, D, o_parts, lse_parts, out_dtype, out, lse, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return ok();
}

va_status verify_tree_mask_from_parents(int B, int T, const int32_t *parent, uint32_t *mask, void *workspace,
                                        va_stream stream) {
  if (B < 1 || T < 1) return fail(VA_ERR_INVALID_ARG, "B and T must be >= 1");
  if (T > 64) return fail(VA_ERR_UNSUPPORTED, "T=%d; at most 64 draft tokens are supported", T);
  if (parent == nullptr || mask == nullptr) return fail(VA_ERR_INVALID_ARG, "parent and mask must not be NULL");
  if (workspace != nullptr && !aligned(workspace, 256)) return fail(VA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaError_t e = va::launch_tree_mask(B, T, parent, mask, static_cast<int *>(workspace), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "tree mask launch");
  return ok();
}

va_status verify_build_index(int B, int Hkv, const int32_t *seqlens, const float *score_draft,
                             const float *score_target, int score_stride, int n_sink, int window, int m_draft,
                             int budget, int32_t *indices, int32_t *n_indices, void *workspace, va_stream stream) {
  if (B < 1 || Hkv < 1) return fail(VA_ERR_INVALID_ARG, "B and Hkv must be >= 1");
  if (seqlens == nullptr || score_draft == nullptr || score_target == nullptr || indices == nullptr ||
      n_indices == nullptr)
    return fail(VA_ERR_INVALID_ARG, "seqlens, scores, indices and n_indices must not be NULL");
  if (n_sink < 0 || window < 0 || m_draft < 0 || budget < 1 || score_stride < 1)
    return fail(VA_ERR_INVALID_ARG, "negative selection size or empty budget/stride");
  if (budget < n_sink + window)
    return fail(VA_ERR_INVALID_ARG, "budget=%d is smaller than n_sink + window = %d", budget, n_sink + window);
  if ((long long)B * Hkv > (1ll << 30)) return fail(VA_ERR_UNSUPPORTED, "too many (sequence, head) rows");
  if (workspace != nullptr && !aligned(workspace, 256)) return fail(VA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaError_t e = va::launch_build_index(B, Hkv, seqlens, score_draft, score_target, score_stride, n_sink, window,
                                         m_draft, budget, indices, n_indices, static_cast<int *>(workspace),
                                         g_test_index_radix.load() != 0, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "index launch");
  return ok();
}

va_status verify_accept_greedy(int B, int T, const int32_t *parent, const int32_t *draft_tokens,
                               const int32_t *target_next, int32_t *path, int32_t *n_accept, int32_t *bonus,
                               void *workspace, va_stream stream) {
  if (B < 1 || T < 1) return fail(VA_ERR_INVALID_ARG, "B and T must be >= 1");
  if (T > 64) return fail(VA_ERR_UNSUPPORTED, "T=%d; at most 64 draft tokens are supported", T);
  if (parent == nullptr || draft_tokens == nullptr || target_next == nullptr || path == nullptr ||
      n_accept == nullptr || bonus == nullptr)
    return fail(VA_ERR_INVALID_ARG, "parent, draft_tokens, target_next, path, n_accept and bonus must not be NULL");
  if (workspace != nullptr && !aligned(workspace, 256)) return fail(VA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaError_t e = va::launch_accept_greedy(B, T, parent, draft_tokens, target_next, path, n_accept, bonus,
                                           static_cast<int *>(workspace), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "acceptance launch");
  return ok();
}


va_status verify_commit_kv_dense(const va_shape *shape, void *k_cache, void *v_cache, int max_cache_len,
                                 const int32_t *seqlens, const int32_t *path, const int32_t *n_accept,
                                 int32_t *seqlens_out, void *workspace, va_stream stream) {
  va::CommitParams cp;
  va_status st = commit_common(shape, k_cache, v_cache, seqlens, path, n_accept, seqlens_out, workspace, cp);
  if (st != VA_OK) return st;
  if (max_cache_len < shape->T)
    return fail(VA_ERR_INVALID_ARG, "max_cache_len=%d is smaller than T=%d", max_cache_len, shape->T);
  cp.len_cap = max_cache_len;
  cudaError_t e = va::launch_commit_kv(cp, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "commit launch");
  return ok();
}

size_t verify_head_importance_scratch_size(int B, int T, int n_heads, int max_cache_len) {
  if (B < 1 || T < 1 || n_heads < 1 || max_cache_len < 1) return 0;
  return va::score_scratch_bytes(B, n_heads * T, max_cache_len);
}

va_status verify_head_importance(const va_shape *shape, const void *q, const void *k_cache, int max_cache_len,
                                 const int32_t *seqlens, const int32_t *heads, int n_heads, float *score,
                                 int score_stride, void *scratch, size_t scratch_bytes, void *workspace,
                                 va_stream stream) {
  if (shape == nullptr) return fail(VA_ERR_INVALID_ARG, "shape is NULL");
  const va_shape &s = *shape;
  if (s.B < 1 || s.T < 1 || s.Hq < 1 || s.Hkv < 1 || s.Hq % s.Hkv != 0)
    return fail(VA_ERR_INVALID_ARG, "bad shape (B=%d T=%d Hq=%d Hkv=%d)", s.B, s.T, s.Hq, s.Hkv);
  if (!(s.scale > 0.f) || !isfinite(s.scale)) return fail(VA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (s.dtype != VA_DTYPE_BF16 || s.D != 128)
    return fail(VA_ERR_UNSUPPORTED, "the scoring pass supports bf16 with D = 128");
  if (s.T > 64) return fail(VA_ERR_UNSUPPORTED, "T=%d; at most 64 tokens are supported", s.T);
  if (s.B > 65535) return fail(VA_ERR_UNSUPPORTED, "B=%d; at most 65535 sequences", s.B);
  if (heads == nullptr || n_heads < 1) return fail(VA_ERR_INVALID_ARG, "list at least one query head");
  if (n_heads > va::kScoreMaxHeads || n_heads * s.T > va::kScoreMaxRows)
    return fail(VA_ERR_UNSUPPORTED, "n_heads=%d x T=%d: at most %d heads and %d rows", n_heads, s.T,
                va::kScoreMaxHeads, va::kScoreMaxRows);
  for (int i = 0; i < n_heads; ++i)
    if (heads[i] < 0 || heads[i] >= s.Hq) return fail(VA_ERR_INVALID_ARG, "heads[%d]=%d is not in [0, Hq)", i, heads[i]);
  if (q == nullptr || k_cache == nullptr || seqlens == nullptr || score == nullptr || scratch == nullptr)
    return fail(VA_ERR_INVALID_ARG, "q, k_cache, seqlens, score and scratch must not be NULL");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(score, 4))
    return fail(VA_ERR_INVALID_ARG, "q and k_cache must be 16-byte aligned, score 4-byte aligned");
  if (max_cache_len < 1 || score_stride < 1)
    return fail(VA_ERR_INVALID_ARG, "max_cache_len and score_stride must be >= 1");
  if (max_cache_len > (1 << 30)) return fail(VA_ERR_UNSUPPORTED, "max_cache_len above 2^30");
  if (!aligned(scratch, 256)) return fail(VA_ERR_WORKSPACE, "scratch must be 256-byte aligned");
  const size_t need = va::score_scratch_bytes(s.B, n_heads * s.T, max_cache_len);
  if (scratch_bytes < need) return fail(VA_ERR_WORKSPACE, "scratch has %zu bytes, %zu needed", scratch_bytes, need);
  if (workspace != nullptr && !aligned(workspace, 256)) return fail(VA_ERR_WORKSPACE, "workspace must be 256-byte aligned");

  va::ScoreParams p;
  memset(&p, 0, sizeof p);
  p.B = s.B;
  p.T = s.T;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.max_cache_len = max_cache_len;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.k = static_cast<const __nv_bfloat16 *>(k_cache);
  p.seqlens = seqlens;
  p.R = n_heads * s.T;
  p.n_chunks = (max_cache_len + va::kScoreChunk - 1) / va::kScoreChunk;
  p.lpad = p.n_chunks * va::kScoreChunk;
  p.logits = static_cast<float *>(scratch);
  p.part = reinterpret_cast<float2 *>(static_cast<uint8_t *>(scratch) +
                                      va::align256(sizeof(float) * (size_t)s.B * p.R * p.lpad));
  p.score = score;
  p.score_stride = score_stride;
  p.score_vec4 = aligned(score, 16) && score_stride % 4 == 0;
  p.status = static_cast<int *>(workspace);
  // rows grouped by kv-head (a stable order of the listed heads), T rows per
  // head; a unit is at most kScoreUnitRows consecutive rows of one kv-head
  const int group = s.Hq / s.Hkv;
  int order[va::kScoreMaxHeads];
  for (int i = 0; i < n_heads; ++i) order[i] = i;
  for (int i = 1; i < n_heads; ++i)  // insertion sort by kv-head, stable
    for (int j = i; j > 0 && heads[order[j - 1]] / group > heads[order[j]] / group; --j) {
      const int t = order[j];
      order[j] = order[j - 1];
      order[j - 1] = t;
    }
  int r = 0;
  for (int i = 0; i < n_heads; ++i)
    for (int t = 0; t < s.T; ++t, ++r) {
      p.row_head[r] = (int16_t)heads[order[i]];
      p.row_t[r] = (int8_t)t;
    }
  int nu = 0;
  for (int r0 = 0; r0 < p.R;) {
    const int kvh = p.row_head[r0] / group;
    int n = 0;
    while (r0 + n < p.R && n < va::kScoreUnitRows && p.row_head[r0 + n] / group == kvh) ++n;
    if (nu == va::kScoreMaxUnits) return fail(VA_ERR_UNSUPPORTED, "too many (kv-head, row block) units");
    p.unit_kvh[nu] = (int16_t)kvh;
    p.unit_row0[nu] = (int16_t)r0;
    p.unit_n[nu] = (int8_t)n;
    ++nu;
    r0 += n;
  }
  p.n_units = nu;
  cudaError_t e = va::launch_head_importance(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "scoring launch");
  return ok();
}

va_status verify_rope_draft_dense(const va_shape *shape, void *q, void *k_cache, int max_cache_len,
                                  const int32_t *seqlens, const int32_t *positions, float rope_base,
                                  void *workspace, va_stream stream) {
  va::RopeParams rp;
  va_status st = rope_common(shape, q, k_cache, seqlens, positions, rope_base, workspace, rp);
  if (st != VA_OK) return st;
  if (max_cache_len < shape->T)
    return fail(VA_ERR_INVALID_ARG, "max_cache_len=%d is smaller than T=%d", max_cache_len, shape->T);
  rp.len_cap = max_cache_len;
  cudaError_t e = va::launch_rope_draft(rp, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope launch");
  return ok();
}

va_status verify_rope_draft_paged(const va_shape *shape, void *q, void *k_pages, int num_pages, int page_size,
                                  const int32_t *page_table, int max_pages_per_seq, const int32_t *seqlens,
                                  const int32_t *positions, float rope_base, void *workspace, va_stream stream) {
  va::RopeParams rp;
  va_status st = rope_common(shape, q, k_pages, seqlens, positions, rope_base, workspace, rp);
  if (st != VA_OK) return st;
  if (page_table == nullptr) return fail(VA_ERR_INVALID_ARG, "page_table must not be NULL");
  if (page_size < 1 || page_size > 1024 || (page_size & (page_size - 1)) != 0)
    return fail(VA_ERR_INVALID_ARG, "page_size=%d must be a power of two in [1, 1024]", page_size);
  if (num_pages < 1 || max_pages_per_seq < 1) return fail(VA_ERR_INVALID_ARG, "num_pages and max_pages_per_seq must be >= 1");
  const long long cap = (long long)max_pages_per_seq * page_size;
  if (cap < shape->T || cap >= (1ll << 31))
    return fail(VA_ERR_INVALID_ARG, "max_pages_per_seq * page_size = %lld must be in [T, 2^31)", cap);
  rp.len_cap = (int)cap;
  rp.page_table = page_table;
  rp.num_pages = num_pages;
  rp.max_pages = max_pages_per_seq;
  int shift = 0;
  while ((1 << shift) < page_size) ++shift;
  rp.page_shift = shift;
  cudaError_t e = va::launch_rope_draft(rp, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope launch");
  return ok();
}

va_status verify_commit_kv_paged(const va_shape *shape, void *k_pages, void *v_pages, int num_pages, int page_size,
                                 const int32_t *page_table, int max_pages_per_seq, const int32_t *seqlens,
                                 const int32_t *path, const int32_t *n_accept, int32_t *seqlens_out,
                                 void *workspace, va_stream stream) {
  va::CommitParams cp;
  va_status st = commit_common(shape, k_pages, v_pages, seqlens, path, n_accept, seqlens_out, workspace, cp);
  if (st != VA_OK) return st;
  if (page_table == nullptr) return fail(VA_ERR_INVALID_ARG, "page_table must not be NULL");
  if (page_size < 1 || page_size > 1024 || (page_size & (page_size - 1)) != 0)
    return fail(VA_ERR_INVALID_ARG, "page_size=%d must be a power of two in [1, 1024]", page_size);
  if (num_pages < 1 || max_pages_per_seq < 1) return fail(VA_ERR_INVALID_ARG, "num_pages and max_pages_per_seq must be >= 1");
  const long long cap = (long long)max_pages_per_seq * page_size;
  if (cap < shape->T || cap >= (1ll << 31))
    return fail(VA_ERR_INVALID_ARG, "max_pages_per_seq * page_size = %lld must be in [T, 2^31)", cap);
  cp.len_cap = (int)cap;
  cp.page_table = page_table;
  cp.num_pages = num_pages;
  cp.max_pages = max_pages_per_seq;
  while ((1 << cp.page_shift) < page_size) ++cp.page_shift;
  cudaError_t e = va::launch_commit_kv(cp, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "commit launch");
  return ok();
}

va_status verify_attn_check_status(void *workspace, va_stream stream) {
  if (workspace == nullptr) return fail(VA_ERR_WORKSPACE, "workspace is NULL");
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int status = 0;
  e = cudaMemcpy(&status, workspace, sizeof status, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (status != 0) {
    // the status word and the merge kernel's list length are reset here; the
    // per-segment merge counters of a call that stopped at a timeout may not be
    // (their size depends on the workspace, which this call is not given):
    // verify_attn_workspace_init restores them
    e = cudaMemset(workspace, 0, va::kHeaderBytes);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    switch (status) {
      case VA_ERR_TIMEOUT:
        return fail(VA_ERR_TIMEOUT, "a bounded device wait ran out");
      case VA_ERR_DEVICE_BOUNDS:
        return fail(VA_ERR_DEVICE_BOUNDS, "device saw an out-of-range seqlen, page, index or parent");
      case VA_ERR_DEVICE_INVALID:
        return fail(VA_ERR_DEVICE_INVALID, "validation: a verify set is not strictly increasing (out of order or "
                                           "an index listed twice)");
      default:
        return fail((va_status)status, "device status %d", status);
    }
  }
  return ok();
}

const char *verify_attn_last_error(void) { return g_last_error.c_str(); }

const char *verify_attn_version(void) { return "verify_attn 0.1 sm_103a"; }

// Test hooks declared in verify_attn_testing.h.
va_status verify_attn_test_inject(unsigned long long wait_ns, int drop_part) {
  if (wait_ns > 100000000ull) return fail(VA_ERR_INVALID_ARG, "wait_ns must be at most 0.1 s");
  g_test_wait_ns.store(wait_ns);
  g_test_drop_part.store(drop_part < 0 ? -1 : drop_part);
  return ok();
}

va_status verify_attn_test_index_path(int mode) {
  if (mode != 0 && mode != 1) return fail(VA_ERR_INVALID_ARG, "mode must be 0 or 1");
  g_test_index_radix.store(mode);
  return ok();
}

va_status verify_attn_selftest_wait_timeout(void *workspace, unsigned long long wait_ns, va_stream stream) {
  if (workspace == nullptr || !aligned(workspace, 256)) return fail(VA_ERR_WORKSPACE, "bad workspace");
  if (wait_ns == 0 || wait_ns > 100000000ull) return fail(VA_ERR_INVALID_ARG, "wait_ns must be in (0, 0.1 s]");
  cudaError_t e = va::launch_wait_selftest(static_cast<int *>(workspace), wait_ns, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Entry point that allocates nothing (declared in verify_attn.h).
//
// Some callers cannot hand the library a workspace: a plugin that is given only
// its input and output tensors by a host framework and has no handle on that
// framework's device allocator, or a deployment that fixes its device memory at
// start-up and forbids any allocation afterwards.  For them the scratch this
// call needs (partial results, segment bookkeeping, the device status word)
// lives in one file-scope device array of fixed size, which every GPU that
// loads this library holds until the process exits.
// ---------------------------------------------------------------------------
constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

namespace {
std::mutex g_static_mu;
void *g_static_addr[64] = {nullptr};  // device address of g_static_scratch, per device

// Resolve the device address of the static scratch for the current device
// (once per device, with that device current).  In host code the array's name
// is only a host-side stand-in, so kernels must receive this address instead.
va_status static_scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(VA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_addr[dev] == nullptr) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_static_addr[dev] = ptr;
  }
  *out = g_static_addr[dev];
  return VA_OK;
}
}  // namespace

extern "C" va_status verify_attn_dense_noalloc(const va_shape *shape, const void *q, const void *k_cache,
                                               const void *v_cache, int max_cache_len, const int32_t *seqlens,
                                               const int32_t *tree_parent, const uint32_t *tree_mask,
                                               const int32_t *positions, void *out, float *lse,
                                               int32_t *device_status, va_stream stream) {
  va_status st = check_shape(shape);
  if (st != VA_OK) return st;
  const size_t need = verify_attn_workspace_size(shape);
  if (need == 0) return fail(VA_ERR_CUDA, "no usable CUDA device");
  if (need > kStaticScratchBytes)
    return fail(VA_ERR_UNSUPPORTED,
                "this shape needs %zu bytes of scratch; the static scratch of verify_attn_dense_noalloc holds %zu "
                "bytes -- use verify_attn_dense with a caller workspace",
                need, kStaticScratchBytes);
  void *scratch = nullptr;
  st = static_scratch_address(&scratch);
  if (st != VA_OK) return st;
  // the bookkeeping (status word, merge list length, per-segment merge
  // counters) starts at zero for every call, whatever the previous call's shape
  // or outcome; the rest of the scratch is written before it is read
  cudaError_t e = cudaMemsetAsync(scratch, 0, va::kBookkeepingBytes, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the static scratch bookkeeping");
  st = verify_attn_dense(shape, q, k_cache, v_cache, max_cache_len, seqlens, tree_parent, tree_mask, positions, out,
                         lse, scratch, kStaticScratchBytes, stream);
  if (st != VA_OK) return st;
  if (device_status != nullptr) {
    e = cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "copying the device status word");
  }
  return ok();
}
