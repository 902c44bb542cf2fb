"""Helpers shared by the GPU tests: move a workload to the device and run the
library's entry points on it; compare with the oracle at the stated tolerances."""
import numpy as np
import torch

import speculative_decoding_verification_masked_gb300 as va

# bf16 outputs: max-abs 2e-3; lse: max-abs 1e-3 (fp32 outputs held to the same bar).
# Cases with few visible keys have |out| ~ 1, where the bf16 output format alone
# rounds by up to half an ulp (2^-9 * 2^floor(log2|out|), e.g. 7.8e-3 at |out| = 3);
# for those, compare(strict=False) adds that half ulp of the reference value.
OUT_TOL = 2e-3
LSE_TOL = 1e-3


def half_ulp(ref, dtype):
    """Half a unit in the last place of the output format at |ref| (bf16: 8 significant bits)."""
    bits = 8 if dtype == torch.bfloat16 else 24
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - bits), 0.0)


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a).astype(np.int32))).cuda()


def dev_words(words):
    """uint32 bitmask words -> int32 device tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(np.asarray(words, dtype=np.uint32)).view(np.int32)).cuda()


def run_library(w, mode="parent", indices=None, n_indices=None, workspace=None):
    """Run one verification on workload ``w``.

    mode: 'parent' (tree parents -> fused mask), 'mask' (explicit bitmask words:
    the workload's own or, for trees, the library's tree_mask kernel output),
    'causal' (no mask argument).  Returns (out, lse) on the device.
    """
    q = w.q.cuda()
    seqlens = dev_i32(w.seqlens)
    parent = mask = None
    if mode == "parent":
        assert w.parent is not None
        parent = dev_i32(w.parent)
    elif mode == "mask":
        if w.mask_words is not None:
            mask = dev_words(w.mask_words)
        else:
            mask = va.verify_tree_mask_from_parents(dev_i32(w.parent))
    elif mode != "causal":
        raise ValueError(mode)
    if w.layout == "dense":
        return va.verify_attn_dense(q, w.k_cache.cuda(), w.v_cache.cuda(), seqlens, tree_parent=parent,
                                    tree_mask=mask, workspace=workspace)
    if w.layout == "paged":
        return va.verify_attn_paged(q, w.k_pages.cuda(), w.v_pages.cuda(), dev_i32(w.page_table), seqlens,
                                    tree_parent=parent, tree_mask=mask, workspace=workspace)
    if w.layout == "sparse":
        return va.verify_attn_sparse(q, w.k_cache.cuda(), w.v_cache.cuda(), seqlens, indices, n_indices,
                                     tree_parent=parent, tree_mask=mask, workspace=workspace)
    raise ValueError(w.layout)


def compare(out, lse, ref, tol_out=OUT_TOL, tol_lse=LSE_TOL, strict=False):
    """Element-wise comparison with the oracle; returns (max_abs_out, max_abs_lse, max|ref|).

    strict=True holds every output to tol_out; otherwise each output may also
    differ by the half ulp of its bf16 rounding (see above)."""
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    ro, rl = ref["out"], ref["lse"]
    assert o.shape == ro.shape and l.shape == rl.shape
    assert np.array_equal(np.isneginf(l), np.isneginf(rl)), "empty-row pattern differs"
    fin = np.isfinite(rl)
    err = np.abs(o - ro)
    eo = float(err.max()) if o.size else 0.0
    el = float(np.abs(l[fin] - rl[fin]).max()) if fin.any() else 0.0
    assert np.all(np.isfinite(o)), "non-finite output"
    if strict:
        assert eo <= tol_out, f"out max-abs error {eo:.3e} > {tol_out}"
    else:
        excess = err - (tol_out + half_ulp(ro, out.dtype))
        assert excess.max() <= 0, f"out error {eo:.3e} exceeds 2e-3 + half ulp by {excess.max():.3e}"
    assert el <= tol_lse, f"lse max-abs error {el:.3e} > {tol_lse}"
    return eo, el, float(np.abs(ro).max())
