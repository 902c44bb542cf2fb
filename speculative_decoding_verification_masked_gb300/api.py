"""Thin Python binding of libverify_attn.so (C ABI in include/verify_attn.h).

Argument marshalling only: every function here takes torch tensors that live
on the GPU, checks dtypes/shapes enough to build the C call, passes raw device
pointers and the current CUDA stream, and raises ``VerifyAttnError`` when the
library returns a non-OK status.  All computation happens in the CUDA kernels;
there is no fallback path, and importing the library fails loudly when it has
not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

VA_OK, VA_ERR_INVALID_ARG, VA_ERR_UNSUPPORTED, VA_ERR_WORKSPACE, VA_ERR_CUDA, VA_ERR_TIMEOUT, \
    VA_ERR_DEVICE_BOUNDS, VA_ERR_DEVICE_INVALID = range(8)
VA_DTYPE_BF16, VA_DTYPE_FP32 = 0, 2
STATUS_NAMES = {0: "VA_OK", 1: "VA_ERR_INVALID_ARG", 2: "VA_ERR_UNSUPPORTED", 3: "VA_ERR_WORKSPACE",
                4: "VA_ERR_CUDA", 5: "VA_ERR_TIMEOUT", 6: "VA_ERR_DEVICE_BOUNDS", 7: "VA_ERR_DEVICE_INVALID"}


class VerifyAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class VaShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
                ("D", ctypes.c_int), ("dtype", ctypes.c_int), ("scale", ctypes.c_float),
                ("rope_base", ctypes.c_float)]


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_SIGS = {
    "verify_attn_workspace_size": (_SZ, [ctypes.POINTER(VaShape)]),
    "verify_attn_workspace_init": (_I, [_P, _SZ, _P]),
    "verify_attn_dense": (_I, [ctypes.POINTER(VaShape), _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "verify_attn_paged": (_I, [ctypes.POINTER(VaShape), _P, _P, _P, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P, _P,
                               _SZ, _P]),
    "verify_attn_sparse": (_I, [ctypes.POINTER(VaShape), _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P,
                                _SZ, _P]),
    "verify_attn_combine": (_I, [_I, _I, _I, _P, _P, _I, _P, _P, _P]),
    "verify_tree_mask_from_parents": (_I, [_I, _I, _P, _P, _P, _P]),
    "verify_build_index": (_I, [_I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "verify_accept_greedy": (_I, [_I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "verify_commit_kv_dense": (_I, [ctypes.POINTER(VaShape), _P, _P, _I, _P, _P, _P, _P, _P, _P]),
    "verify_commit_kv_paged": (_I, [ctypes.POINTER(VaShape), _P, _P, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P]),
    "verify_rope_draft_dense": (_I, [ctypes.POINTER(VaShape), _P, _P, _I, _P, _P, ctypes.c_float, _P, _P]),
    "verify_rope_draft_paged": (_I, [ctypes.POINTER(VaShape), _P, _P, _I, _I, _P, _I, _P, _P, ctypes.c_float, _P,
                                     _P]),
    "verify_head_importance_scratch_size": (_SZ, [_I, _I, _I, _I]),
    "verify_head_importance": (_I, [ctypes.POINTER(VaShape), _P, _P, _I, _P, _P, _I, _P, _I, _P, _SZ, _P, _P]),
    "verify_attn_check_status": (_I, [_P, _P]),
    "verify_attn_last_error": (ctypes.c_char_p, []),
    "verify_attn_version": (ctypes.c_char_p, []),
    "verify_attn_selftest_wait_timeout": (_I, [_P, ctypes.c_ulonglong, _P]),
    "verify_attn_test_inject": (_I, [ctypes.c_ulonglong, _I]),
    "verify_attn_test_index_path": (_I, [_I]),
    "verify_attn_dense_noalloc": (_I, [ctypes.POINTER(VaShape), _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
}


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True):
    """The loaded ctypes library (built on first use when nvcc is available)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libverify_attn.so is not built ({path}); run __graft_entry__.build()")
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _check(status: int):
    if status != VA_OK:
        msg = lib().verify_attn_last_error().decode()
        raise VerifyAttnError(status, msg)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor or None")
    if not t.is_cuda:
        raise ValueError("tensor arguments must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return VA_DTYPE_BF16
    if t.dtype == torch.float32:
        return VA_DTYPE_FP32
    raise TypeError(f"unsupported element type {t.dtype}; use bfloat16 or float32")


def make_shape(B, T, Hq, Hkv, D, dtype_code, scale=None, rope_base=0.0) -> VaShape:
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    return VaShape(int(B), int(T), int(Hq), int(Hkv), int(D), int(dtype_code), float(scale), float(rope_base))


def workspace_size(shape: VaShape) -> int:
    return int(lib().verify_attn_workspace_size(ctypes.byref(shape)))


class Workspace:
    """Caller-owned device scratch for the attention calls, initialised once."""

    def __init__(self, nbytes: int, device=None, stream=None):
        nbytes = max(int(nbytes), 256)
        self.buffer = torch.empty(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        base = self.buffer.data_ptr()
        self.offset = (-base) % 256
        self.nbytes = nbytes
        _check(lib().verify_attn_workspace_init(self.ptr, self.nbytes, _stream(stream)))

    @property
    def ptr(self) -> int:
        return self.buffer.data_ptr() + self.offset

    @classmethod
    def for_shape(cls, shape: VaShape, device=None, stream=None) -> "Workspace":
        n = workspace_size(shape)
        if n == 0:
            _check(VA_ERR_INVALID_ARG)
        return cls(n, device=device, stream=stream)


# ----------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ----------------------------------------------------------------------------

def _shape_of(q, Hkv, scale, rope_base=0.0):
    B, T, Hq, D = q.shape
    return make_shape(B, T, Hq, Hkv, D, _dtype_code(q), scale, rope_base)


def _outputs(q, out, lse):
    B, T, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device)
    return out, lse


def verify_attn_dense(q, k_cache, v_cache, seqlens, tree_parent=None, tree_mask=None, positions=None,
                      out=None, lse=None, workspace: Workspace = None, scale=None, stream=None, rope_base=0.0):
    """Dense-cache verification attention; returns (out [B][T][Hq][D], lse [B][Hq][T]).
    With positions [B][T] int32 (and rope_base > 0) q and the draft keys are
    rotated inside the kernels."""
    shape = _shape_of(q, k_cache.shape[2], scale, rope_base)
    out, lse = _outputs(q, out, lse)
    ws = workspace or Workspace.for_shape(shape, q.device, stream)
    _check(lib().verify_attn_dense(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[1],
                                   _ptr(seqlens), _ptr(tree_parent), _ptr(tree_mask), _ptr(positions), _ptr(out),
                                   _ptr(lse), ws.ptr, ws.nbytes, _stream(stream)))
    return out, lse


def verify_attn_dense_noalloc(q, k_cache, v_cache, seqlens, tree_parent=None, tree_mask=None, positions=None,
                              out=None, lse=None, device_status=None, scale=None, stream=None, rope_base=0.0):
    """verify_attn_dense without a workspace (fixed 8 MiB static device scratch inside
    the library) for callers that cannot allocate; see include/verify_attn.h."""
    shape = _shape_of(q, k_cache.shape[2], scale, rope_base)
    out, lse = _outputs(q, out, lse)
    _check(lib().verify_attn_dense_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                           k_cache.shape[1], _ptr(seqlens), _ptr(tree_parent), _ptr(tree_mask),
                                           _ptr(positions), _ptr(out), _ptr(lse), _ptr(device_status),
                                           _stream(stream)))
    return out, lse


def verify_attn_paged(q, k_pages, v_pages, page_table, seqlens, tree_parent=None, tree_mask=None, positions=None,
                      out=None, lse=None, workspace: Workspace = None, scale=None, stream=None, rope_base=0.0):
    """Paged-cache verification attention; pages [P][page][Hkv][D], page_table int32 [B][max_pages]."""
    shape = _shape_of(q, k_pages.shape[2], scale, rope_base)
    out, lse = _outputs(q, out, lse)
    ws = workspace or Workspace.for_shape(shape, q.device, stream)
    _check(lib().verify_attn_paged(ctypes.byref(shape), _ptr(q), _ptr(k_pages), _ptr(v_pages), k_pages.shape[0],
                                   k_pages.shape[1], _ptr(page_table), page_table.shape[1], _ptr(seqlens),
                                   _ptr(tree_parent), _ptr(tree_mask), _ptr(positions), _ptr(out), _ptr(lse),
                                   ws.ptr, ws.nbytes, _stream(stream)))
    return out, lse


def verify_attn_sparse(q, k_cache, v_cache, seqlens, indices, n_indices, tree_parent=None, tree_mask=None,
                       positions=None, out=None, lse=None, workspace: Workspace = None, scale=None, stream=None,
                       rope_base=0.0):
    """Sparse verification over per-(sequence, kv-head) verify index sets [B][Hkv][max_indices]."""
    shape = _shape_of(q, k_cache.shape[2], scale, rope_base)
    out, lse = _outputs(q, out, lse)
    ws = workspace or Workspace.for_shape(shape, q.device, stream)
    _check(lib().verify_attn_sparse(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[1],
                                    _ptr(seqlens), _ptr(indices), _ptr(n_indices), indices.shape[2],
                                    _ptr(tree_parent), _ptr(tree_mask), _ptr(positions), _ptr(out), _ptr(lse),
                                    ws.ptr, ws.nbytes, _stream(stream)))
    return out, lse


def verify_attn_combine(o_parts, lse_parts, out_dtype=torch.float32, out=None, lse=None, stream=None):
    """Log-sum-exp merge of partials: o_parts f32 [S][R][D], lse_parts f32 [S][R] -> (out [R][D], lse [R])."""
    S, R, D = o_parts.shape
    if out is None:
        out = torch.empty(R, D, dtype=out_dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty(R, dtype=torch.float32, device=o_parts.device)
    _check(lib().verify_attn_combine(R, S, D, _ptr(o_parts), _ptr(lse_parts), _dtype_code(out), _ptr(out), _ptr(lse),
                                     _stream(stream)))
    return out, lse


def verify_tree_mask_from_parents(parent, mask=None, workspace: Workspace = None, stream=None):
    """Ancestor-or-self bitmask uint32-as-int32 [B][T][ceil(T/32)] from parent int32 [B][T]."""
    B, T = parent.shape
    if mask is None:
        mask = torch.empty(B, T, (T + 31) // 32, dtype=torch.int32, device=parent.device)
    _check(lib().verify_tree_mask_from_parents(B, T, _ptr(parent), _ptr(mask),
                                               workspace.ptr if workspace is not None else None, _stream(stream)))
    return mask


def verify_build_index(seqlens, score_draft, score_target, n_sink, window, m_draft, budget, indices=None,
                       n_indices=None, workspace: Workspace = None, stream=None):
    """Verify index sets: returns (indices int32 [B][Hkv][budget], n_indices int32 [B][Hkv])."""
    B, Hkv, stride = score_draft.shape
    if indices is None:
        indices = torch.empty(B, Hkv, budget, dtype=torch.int32, device=score_draft.device)
    if n_indices is None:
        n_indices = torch.empty(B, Hkv, dtype=torch.int32, device=score_draft.device)
    _check(lib().verify_build_index(B, Hkv, _ptr(seqlens), _ptr(score_draft), _ptr(score_target), stride, n_sink,
                                    window, m_draft, budget, _ptr(indices), _ptr(n_indices),
                                    workspace.ptr if workspace is not None else None, _stream(stream)))
    return indices, n_indices


def verify_accept_greedy(parent, draft_tokens, target_next, path=None, n_accept=None, bonus=None,
                         workspace: Workspace = None, stream=None):
    """Greedy tree acceptance: returns (path int32 [B][T], n_accept int32 [B], bonus int32 [B])."""
    B, T = parent.shape
    dev = parent.device
    if path is None:
        path = torch.empty(B, T, dtype=torch.int32, device=dev)
    if n_accept is None:
        n_accept = torch.empty(B, dtype=torch.int32, device=dev)
    if bonus is None:
        bonus = torch.empty(B, dtype=torch.int32, device=dev)
    _check(lib().verify_accept_greedy(B, T, _ptr(parent), _ptr(draft_tokens), _ptr(target_next), _ptr(path),
                                      _ptr(n_accept), _ptr(bonus), workspace.ptr if workspace is not None else None,
                                      _stream(stream)))
    return path, n_accept, bonus


def verify_commit_kv_dense(k_cache, v_cache, seqlens, path, n_accept, seqlens_out=None,
                           workspace: Workspace = None, stream=None):
    """Move the accepted draft rows of k_cache / v_cache [B][len][Hkv][D] in
    place to the slots after each prefix; returns seqlens + n_accept."""
    B, cap, Hkv, D = k_cache.shape
    T = path.shape[1]
    if seqlens_out is None:
        seqlens_out = torch.empty(B, dtype=torch.int32, device=k_cache.device)
    shape = make_shape(B, T, Hkv, Hkv, D, _dtype_code(k_cache), 1.0)
    _check(lib().verify_commit_kv_dense(ctypes.byref(shape), _ptr(k_cache), _ptr(v_cache), cap, _ptr(seqlens),
                                        _ptr(path), _ptr(n_accept), _ptr(seqlens_out),
                                        workspace.ptr if workspace is not None else None, _stream(stream)))
    return seqlens_out


def verify_commit_kv_paged(k_pages, v_pages, page_table, seqlens, path, n_accept, seqlens_out=None,
                           workspace: Workspace = None, stream=None):
    """The same commit through a page table; pages [P][page][Hkv][D]."""
    P, ps, Hkv, D = k_pages.shape
    B, max_pages = page_table.shape
    T = path.shape[1]
    if seqlens_out is None:
        seqlens_out = torch.empty(B, dtype=torch.int32, device=k_pages.device)
    shape = make_shape(B, T, Hkv, Hkv, D, _dtype_code(k_pages), 1.0)
    _check(lib().verify_commit_kv_paged(ctypes.byref(shape), _ptr(k_pages), _ptr(v_pages), P, ps, _ptr(page_table),
                                        max_pages, _ptr(seqlens), _ptr(path), _ptr(n_accept), _ptr(seqlens_out),
                                        workspace.ptr if workspace is not None else None, _stream(stream)))
    return seqlens_out


def verify_rope_draft_dense(q, k_cache, seqlens, positions, rope_base=10000.0, workspace: Workspace = None,
                            stream=None):
    """Rotate, in place, every head of q [B][T][Hq][D] and the draft key rows
    (slots L_b .. L_b+T-1) of k_cache [B][len][Hkv][D] at positions [B][T]."""
    B, T, Hq, D = q.shape
    _, cap, Hkv, _ = k_cache.shape
    shape = make_shape(B, T, Hq, Hkv, D, _dtype_code(q), 1.0)
    _check(lib().verify_rope_draft_dense(ctypes.byref(shape), _ptr(q), _ptr(k_cache), cap, _ptr(seqlens),
                                         _ptr(positions), float(rope_base),
                                         workspace.ptr if workspace is not None else None, _stream(stream)))


def verify_rope_draft_paged(q, k_pages, page_table, seqlens, positions, rope_base=10000.0,
                            workspace: Workspace = None, stream=None):
    """The same rotation through a page table; pages [P][page][Hkv][D]."""
    B, T, Hq, D = q.shape
    P, ps, Hkv, _ = k_pages.shape
    shape = make_shape(B, T, Hq, Hkv, D, _dtype_code(q), 1.0)
    _check(lib().verify_rope_draft_paged(ctypes.byref(shape), _ptr(q), _ptr(k_pages), P, ps, _ptr(page_table),
                                         page_table.shape[1], _ptr(seqlens), _ptr(positions), float(rope_base),
                                         workspace.ptr if workspace is not None else None, _stream(stream)))


class ScoreScratch:
    """Caller-owned device scratch of the scoring pass (256-byte aligned)."""

    def __init__(self, B, T, n_heads, max_cache_len, device=None):
        n = int(lib().verify_head_importance_scratch_size(int(B), int(T), int(n_heads), int(max_cache_len)))
        if n == 0:
            _check(VA_ERR_INVALID_ARG)
        self.buffer = torch.empty(n + 256, dtype=torch.uint8, device=device or "cuda")
        self.offset = (-self.buffer.data_ptr()) % 256
        self.nbytes = n

    @property
    def ptr(self) -> int:
        return self.buffer.data_ptr() + self.offset


def verify_head_importance(q, k_cache, seqlens, heads, score=None, score_stride=None, scale=None,
                           scratch: ScoreScratch = None, workspace: Workspace = None, stream=None):
    """Importance map of the committed positions from the listed query heads:
    returns score fp32 [B][Hkv][score_stride] (entries past each L_b untouched;
    a new tensor is zero-filled there)."""
    B, T, Hq, D = q.shape
    _, cap, Hkv, _ = k_cache.shape
    heads = [int(h) for h in heads]
    if score is None:
        score = torch.zeros(B, Hkv, score_stride or cap, dtype=torch.float32, device=q.device)
    stride = score.shape[-1]
    if scratch is None:
        scratch = ScoreScratch(B, T, len(heads), cap, device=q.device)
    shape = make_shape(B, T, Hq, Hkv, D, _dtype_code(q), scale)
    harr = (ctypes.c_int32 * len(heads))(*heads)
    _check(lib().verify_head_importance(ctypes.byref(shape), _ptr(q), _ptr(k_cache), cap, _ptr(seqlens),
                                        ctypes.cast(harr, ctypes.c_void_p), len(heads), _ptr(score), stride,
                                        scratch.ptr, scratch.nbytes,
                                        workspace.ptr if workspace is not None else None, _stream(stream)))
    return score


def verify_attn_check_status(workspace: Workspace, stream=None):
    """Synchronise the stream and raise if a kernel recorded a device-side error."""
    _check(lib().verify_attn_check_status(workspace.ptr, _stream(stream)))


def version() -> str:
    return lib().verify_attn_version().decode()
