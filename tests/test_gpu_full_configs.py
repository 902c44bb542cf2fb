"""GPU parity at the measured workloads' full sizes, in the same launch
configuration the benchmark times.  chain, sparse and paged are compared on
every output; tree on two whole kv-head groups (8 of 32 heads, all 64 draft
tokens), which the oracle computes in seconds."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_masked_gb300 as va
import workloads as W
from tests.gpu_util import compare, dev_i32, run_library

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.mark.parametrize("name", ["tiny", "chain", "paged"])
def test_full_config(name):
    w = W.make_workload(name)
    mode = "mask" if w.parent is None else "parent"
    out, lse = run_library(w, mode)
    ref = oracle.verify(w)
    eo, el, mx = compare(out, lse, ref, strict=True)
    print(f"{name}: max|err| out {eo:.2e} lse {el:.2e} max|out| {mx:.3f}")


def test_full_sparse_with_library_index():
    w = W.make_workload("sparse")
    idx, n = va.verify_build_index(dev_i32(w.seqlens), torch.from_numpy(w.score_draft).cuda(),
                                   torch.from_numpy(w.score_target).cuda(), w.n_sink, w.window, w.m_draft, w.budget)
    ref_idx, ref_n = oracle.build_verify_index(w.score_draft, w.score_target, w.seqlens, w.n_sink, w.window,
                                               w.m_draft, w.budget)
    assert np.array_equal(n.cpu().numpy(), ref_n)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    out, lse = run_library(w, "parent", indices=idx, n_indices=n)
    ref = oracle.verify(w, indices=ref_idx, n_indices=ref_n)
    compare(out, lse, ref, strict=True)


def test_full_tree_two_head_groups():
    w = W.make_workload("tree")
    out, lse = run_library(w, "parent")
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    g = w.group
    vis = oracle.draft_visibility(w)
    q = W.bf16_bits(w.q)
    k = W.bf16_bits(w.k_cache)
    v = W.bf16_bits(w.v_cache)
    for h in (0, w.Hkv - 1):
        ro, rl = oracle.attention_dense(q[:, :, h * g:(h + 1) * g], k[:, :, h:h + 1], v[:, :, h:h + 1], w.seqlens,
                                        vis, w.scale)
        assert np.abs(out[:, :, h * g:(h + 1) * g] - ro).max() <= 2e-3
        assert np.abs(lse[:, h * g:(h + 1) * g] - rl).max() <= 1e-3
