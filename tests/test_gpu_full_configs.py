"""GPU parity at the measured workloads' full sizes, in the same launch
configuration the benchmark times, on every output (the 131,072-token tree
workload's oracle takes about 20 s on 8 host cores)."""
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


def test_full_tree_every_head():
    """The long-context tree workload on all 32 heads, every output."""
    w = W.make_workload("tree")
    out, lse = run_library(w, "parent")
    ref = oracle.verify(w)
    eo, el, mx = compare(out, lse, ref, strict=True)
    print(f"tree: max|err| out {eo:.2e} lse {el:.2e} max|out| {mx:.3f}")
