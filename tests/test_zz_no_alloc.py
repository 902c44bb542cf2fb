"""verify_attn_dense_noalloc: the entry point for callers that cannot allocate.

Such callers (a plugin handed only its input and output buffers by a framework
that owns the device allocator, or a deployment that forbids allocation after
start-up) get the dense verification attention with its scratch in a fixed
static device array inside the library.  This file is collected last on
purpose: it checks, through the C ABI, that two calls in a row agree with the
workspace entry point verify_attn_dense on the same inputs, within the parity
tolerances (out 2e-3, lse 1e-3), and that a shape whose scratch does not fit is
refused.  It passes alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_verification_masked_gb300 as va
import workloads as W
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


def test_noalloc_matches_workspace_entry_point_two_calls():
    for seed, L in ((21, 5000), (22, 12345)):  # two calls in a row, different lengths
        w = W.make_workload("chain", seed=seed, L=L)
        q, k, v = w.q.cuda(), w.k_cache.cuda(), w.v_cache.cuda()
        seqlens, parent = _dev_i32(w.seqlens), _dev_i32(w.parent)
        ref_out, ref_lse = _workspace_call(w, q, k, v, seqlens, parent)
        out, lse, status = _noalloc_call(w, q, k, v, seqlens, parent)
        assert status == api.VA_OK
        assert float((out.float() - ref_out.float()).abs().max()) <= 2e-3
        assert float((lse - ref_lse).abs().max()) <= 1e-3


def test_noalloc_refuses_a_shape_beyond_its_scratch():
    L = api.lib()
    big = api.make_shape(64, 16, 32, 8, 128, api.VA_DTYPE_BF16)  # 512 segments: ~22 MB of scratch
    assert L.verify_attn_workspace_size(ctypes.byref(big)) > 8 << 20
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = L.verify_attn_dense_noalloc(ctypes.byref(big), fake, fake, fake, 9000, fake, None, None, None, fake, fake,
                                     None, api._stream())
    assert rc == api.VA_ERR_UNSUPPORTED
    assert "static scratch" in L.verify_attn_last_error().decode()
