"""verify_attn_dense_noalloc: the entry point for callers that cannot allocate.

Such callers (a plugin handed only its input and output buffers by a framework
that owns the device allocator, or a deployment that forbids allocation after
start-up) get the dense verification attention with its scratch in a fixed
static device array inside the library.  This file is collected last on
purpose.  Through the C ABI it checks calls in a row whose shapes differ (so
the bookkeeping inside the shared array moves between calls): each agrees
bit for bit with the workspace entry point verify_attn_dense on the same
inputs, and with the fp64 oracle within the parity bars (out 2e-3, lse 1e-3).
It also checks that a shape whose scratch does not fit is refused.  It passes
alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_masked_gb300 as va
import workloads as W
from tests.gpu_util import compare
from speculative_decoding_verification_masked_gb300 import api

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()


def _noalloc_call(w, q, k, v, seqlens, parent):
    """Call the C entry point directly (ctypes), outputs and status preallocated here."""
    L = api.lib()
    shape = api.make_shape(w.B, w.T, w.Hq, w.Hkv, w.D, api.VA_DTYPE_BF16, w.scale)
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.T, dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = L.verify_attn_dense_noalloc(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(), k.shape[1],
                                     seqlens.data_ptr(), parent.data_ptr(), None, None, out.data_ptr(),
                                     lse.data_ptr(), status.data_ptr(), api._stream())
    assert rc == api.VA_OK, L.verify_attn_last_error().decode()
    torch.cuda.synchronize()
    return out, lse, int(status.item())


def _workspace_call(w, q, k, v, seqlens, parent):
    out, lse = va.verify_attn_dense(q, k, v, seqlens, tree_parent=parent)
    torch.cuda.synchronize()
    return out, lse


def test_noalloc_matches_workspace_entry_point_calls_in_a_row():
    # chain B1, then two sequences, then 16 draft tokens (64 packed rows), then
    # B1 again: the segment count and the row blocking change from call to call
    cases = [("chain", 21, dict(L=5000)), ("chain", 22, dict(B=2, L_lo=3000, L_hi=12345)),
             ("chain", 23, dict(T=16, L=7000)), ("chain", 24, dict(L=12345))]
    for name, seed, over in cases:
        w = W.make_workload(name, seed=seed, **over)
        q, k, v = w.q.cuda(), w.k_cache.cuda(), w.v_cache.cuda()
        seqlens, parent = _dev_i32(w.seqlens), _dev_i32(w.parent)
        ref_out, ref_lse = _workspace_call(w, q, k, v, seqlens, parent)
        out, lse, status = _noalloc_call(w, q, k, v, seqlens, parent)
        assert status == api.VA_OK
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), "same kernel, same inputs: same bits"
        compare(out, lse, oracle.verify(w), strict=True)


def test_noalloc_refuses_a_shape_beyond_its_scratch():
    L = api.lib()
    big = api.make_shape(64, 16, 32, 8, 128, api.VA_DTYPE_BF16)  # 512 segments: ~22 MB of scratch
    assert L.verify_attn_workspace_size(ctypes.byref(big)) > 8 << 20
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = L.verify_attn_dense_noalloc(ctypes.byref(big), fake, fake, fake, 9000, fake, None, None, None, fake, fake,
                                     None, api._stream())
    assert rc == api.VA_ERR_UNSUPPORTED
    assert "static scratch" in L.verify_attn_last_error().decode()
