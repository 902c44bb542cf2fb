"""GPU parity of the rotary embedding of the draft block against the oracle.

Tolerance, from the arithmetic: the kernel reduces each angle in fp64 and
takes sine and cosine of the reduced angle in fp32 (error ~2e-7 in each),
then forms x cos -/+ y sin in fp32.  So before the final rounding a rotated
element is off by at most about 5e-7 (|x| + |y|) for its pair (x, y); the
bf16 store then rounds to nearest, within half an ulp, i.e. 2^-8 of the
value.  Bars: bf16 |gpu - oracle| <= 2^-8 |oracle| + 2e-6 (|x| + |y|); fp32
|gpu - oracle| <= 2e-6 (|x| + |y|); every row that is not rotated is
bit-identical.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_masked_gb300 as va
import workloads as W
from tests.gpu_util import compare, dev_i32

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)


def _host(t):
    t = t.contiguous().cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def _pair_mag(x):
    """|x_i| + |x_{i+D/2}| for every element of rows x [..., D] (f64)."""
    x = np.abs(oracle._widen(x))
    h = x.shape[-1] // 2
    m = x[..., :h] + x[..., h:]
    return np.concatenate([m, m], axis=-1)


def _close(got, want, x_in, dtype):
    got = oracle._widen(got)
    err = np.abs(got - want)
    bound = 2e-6 * _pair_mag(x_in)
    if dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * np.abs(want)
    assert np.all(err <= bound), f"worst excess {(err - bound).max():.3e}"


def _positions(kind, L, T, parent, rng):
    depth = np.stack([W.chain_depths(p) for p in parent])
    if kind == "tree":
        return (L[:, None] + depth).astype(np.int32)
    if kind == "anchor":  # 4 anchors, then consecutive ids from a large offset
        base = np.array([0, 1, 2, 3] + [8192 + i for i in range(max(0, T - 4))])[:T]
        return np.tile(base, (len(L), 1)).astype(np.int32)
    if kind == "large":
        return rng.integers(0, 1 << 24, size=(len(L), T)).astype(np.int32)
    raise ValueError(kind)


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 64)])
@pytest.mark.parametrize("T", [1, 5, 16, 64])
@pytest.mark.parametrize("kind", ["tree", "anchor", "large"])
def test_rope_dense_matches_oracle(dtype, D, T, kind):
    rng = np.random.default_rng(T * 7 + D)
    B, Hq, Hkv = 5, 8, 2
    L = rng.integers(0, 200, size=B).astype(np.int32)
    cap = int(L.max()) + T + 3
    parent = np.stack([W.random_parents(T, rng) for _ in range(B)])
    pos = _positions(kind, L, T, parent, rng)
    if kind == "tree":
        pos[1] += 131072  # the same tree far into a long context
    q = torch.from_numpy(rng.standard_normal((B, T, Hq, D)).astype(np.float32)).to(dtype)
    k = torch.from_numpy(rng.standard_normal((B, cap, Hkv, D)).astype(np.float32)).to(dtype)
    qh, kh = _host(q), _host(k)
    want_q, want_k = oracle.rope_draft_dense(qh, kh, L, pos, 10000.0)
    qd, kd = q.cuda(), k.cuda()
    va.verify_rope_draft_dense(qd, kd, dev_i32(L), dev_i32(pos), 10000.0)
    torch.cuda.synchronize()
    gq, gk = _host(qd), _host(kd)
    _close(gq, want_q, qh, dtype)
    for b in range(B):
        rows = slice(int(L[b]), int(L[b]) + T)
        _close(gk[b, rows], want_k[b, rows], kh[b, rows], dtype)
        keep = np.ones(cap, bool)
        keep[rows] = False
        assert np.array_equal(gk[b, keep], kh[b, keep]), "a row outside the draft block changed"


@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_rope_paged_matches_oracle(page_size):
    w = W.make_workload("paged", seed=page_size, B=6, L_lo=5, L_hi=300, page_size=page_size, spare_pages=3,
                        tree="random")
    rng = np.random.default_rng(page_size)
    pos = _positions("tree", w.seqlens, w.T, w.parent, rng)
    qh, kh = _host(w.q), _host(w.k_pages)
    want_q, want_k = oracle.rope_draft_paged(qh, kh, w.page_table, page_size, w.seqlens, pos, 500000.0)
    qd, kd = w.q.cuda(), w.k_pages.cuda()
    va.verify_rope_draft_paged(qd, kd, dev_i32(w.page_table), dev_i32(w.seqlens), dev_i32(pos), 500000.0)
    torch.cuda.synchronize()
    gq, gk = _host(qd), _host(kd)
    _close(gq, want_q, qh, torch.bfloat16)
    touched = np.zeros(kh.shape[:2], bool)
    for b in range(w.B):
        for t in range(w.T):
            slot = int(w.seqlens[b]) + t
            touched[w.page_table[b][slot // page_size], slot % page_size] = True
    _close(gk[touched], want_k[touched], kh[touched], torch.bfloat16)
    assert np.array_equal(gk[~touched], kh[~touched])


def test_rope_bad_seqlen_is_reported_and_keys_left_alone():
    rng = np.random.default_rng(1)
    B, T, Hq, Hkv, D = 2, 4, 4, 2, 64
    cap = 50
    L = np.array([10, 48], np.int32)  # 48 + 4 > 50
    pos = (L[:, None] + np.arange(T)).astype(np.int32)
    q = torch.from_numpy(rng.standard_normal((B, T, Hq, D)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((B, cap, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    ws = va.Workspace(256)
    qd, kd = q.cuda(), k.cuda()
    va.verify_rope_draft_dense(qd, kd, dev_i32(L), dev_i32(pos), 10000.0, workspace=ws)
    with pytest.raises(va.VerifyAttnError) as ei:
        va.verify_attn_check_status(ws)
    assert ei.value.status == va.api.VA_ERR_DEVICE_BOUNDS
    assert np.array_equal(_host(kd)[1], _host(k)[1])  # the bad sequence's keys are untouched
    want_q, want_k = oracle.rope_draft_dense(_host(q)[:1], _host(k)[:1], L[:1], pos[:1], 10000.0)
    _close(_host(qd), oracle.rope_rotate(_host(q), pos[:, :, None], 10000.0), _host(q), torch.bfloat16)
    _close(_host(kd)[0, 10:14], want_k[0, 10:14], _host(k)[0, 10:14], torch.bfloat16)


def _bf16_bits(x64):
    """f64 -> bf16 bit patterns by round to nearest even (through fp32)."""
    return _host(torch.from_numpy(np.ascontiguousarray(x64, dtype=np.float32)).to(torch.bfloat16))


def test_rope_then_verification_matches_oracle():
    """Rotation, then tree verification attention: against the oracle's
    rotation stored as bf16, then the oracle attention."""
    w = W.make_workload("tree", seed=4, L=1500, T=16, depth=5)
    depth = np.stack([W.chain_depths(p) for p in w.parent])
    pos = (w.seqlens[:, None] + depth).astype(np.int32)
    qh, kh, vh = _host(w.q), _host(w.k_cache), _host(w.v_cache)
    rq, rk = oracle.rope_draft_dense(qh, kh, w.seqlens, pos, 10000.0)
    vis = oracle.draft_visibility(w)
    ref_out, ref_lse = oracle.attention_dense(_bf16_bits(rq), _bf16_bits(rk), vh, w.seqlens, vis, w.scale)
    qd, kd, vd = w.q.cuda(), w.k_cache.cuda(), w.v_cache.cuda()
    seq = dev_i32(w.seqlens)
    va.verify_rope_draft_dense(qd, kd, seq, dev_i32(pos), 10000.0)
    out, lse = va.verify_attn_dense(qd, kd, vd, seq, tree_parent=dev_i32(w.parent))
    torch.cuda.synchronize()
    compare(out, lse, {"out": ref_out, "lse": ref_lse})


def test_rope_tree_then_commit_is_a_plain_sequence():
    """Draft keys rotated at L + depth and then committed along the accepted
    path sit at slot L + j rotated at position L + j: the committed prefix is
    what a plain sequence would hold."""
    rng = np.random.default_rng(8)
    B, T, Hq, Hkv, D = 6, 16, 8, 2, 128
    L = rng.integers(10, 300, size=B).astype(np.int32)
    cap = int(L.max()) + T + 2
    parent = np.stack([W.random_parents(T, rng) for _ in range(B)]).astype(np.int32)
    depth = np.stack([W.chain_depths(p) for p in parent])
    pos = (L[:, None] + depth).astype(np.int32)
    q = torch.from_numpy(rng.standard_normal((B, T, Hq, D)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((B, cap, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    v = k.clone()
    draft = rng.integers(0, 2, size=(B, T)).astype(np.int32)
    tgt = rng.integers(0, 2, size=(B, T + 1)).astype(np.int32)
    path, n, _ = oracle.greedy_accept(parent, draft, tgt)
    kd, vd = k.cuda(), v.cuda()
    seq = dev_i32(L)
    va.verify_rope_draft_dense(q.cuda(), kd, seq, dev_i32(pos), 10000.0)
    va.verify_commit_kv_dense(kd, vd, seq, dev_i32(path), dev_i32(n))
    torch.cuda.synchronize()
    gk, kh = _host(kd), _host(k)
    assert n.sum() > 0
    for b in range(B):
        for j in range(int(n[b])):
            src = kh[b, L[b] + path[b, j]]
            want = oracle.rope_rotate(src, L[b] + j, 10000.0)  # the plain sequence position of slot L + j
            _close(gk[b, L[b] + j], want, src, torch.bfloat16)


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 40), (torch.float32, 40), (torch.bfloat16, 256),
                                     (torch.bfloat16, 2)])
def test_rope_other_head_dims(dtype, D):
    """D not a multiple of 16 (the one-pair-per-thread path), the largest D
    (128 pairs) and the smallest."""
    rng = np.random.default_rng(D)
    B, T, Hq, Hkv = 3, 7, 4, 2
    L = np.array([0, 17, 90], np.int32)
    cap = int(L.max()) + T + 1
    pos = (L[:, None] + np.arange(T) + 70000).astype(np.int32)
    q = torch.from_numpy(rng.standard_normal((B, T, Hq, D)).astype(np.float32)).to(dtype)
    k = torch.from_numpy(rng.standard_normal((B, cap, Hkv, D)).astype(np.float32)).to(dtype)
    qh, kh = _host(q), _host(k)
    want_q, want_k = oracle.rope_draft_dense(qh, kh, L, pos, 10000.0)
    qd, kd = q.cuda(), k.cuda()
    va.verify_rope_draft_dense(qd, kd, dev_i32(L), dev_i32(pos), 10000.0)
    torch.cuda.synchronize()
    _close(_host(qd), want_q, qh, dtype)
    gk = _host(kd)
    for b in range(B):
        rows = slice(int(L[b]), int(L[b]) + T)
        _close(gk[b, rows], want_k[b, rows], kh[b, rows], dtype)
        keep = np.ones(cap, bool)
        keep[rows] = False
        assert np.array_equal(gk[b, keep], kh[b, keep])


def test_rope_rows_not_16_byte_aligned():
    """q and the cache one element past a 16-byte boundary: the vector path is
    not taken; same results."""
    rng = np.random.default_rng(3)
    B, T, Hq, Hkv, D = 2, 5, 4, 2, 64
    L = np.array([3, 40], np.int32)
    cap = 50
    pos = (L[:, None] + np.arange(T)).astype(np.int32)
    qf = torch.from_numpy(rng.standard_normal(B * T * Hq * D + 1).astype(np.float32)).to(torch.bfloat16).cuda()
    kf = torch.from_numpy(rng.standard_normal(B * cap * Hkv * D + 1).astype(np.float32)).to(torch.bfloat16).cuda()
    qd = qf[1:].view(B, T, Hq, D)
    kd = kf[1:].view(B, cap, Hkv, D)
    qh, kh = _host(qd), _host(kd)
    want_q, want_k = oracle.rope_draft_dense(qh, kh, L, pos, 10000.0)
    va.verify_rope_draft_dense(qd, kd, dev_i32(L), dev_i32(pos), 10000.0)
    torch.cuda.synchronize()
    _close(_host(qd), want_q, qh, torch.bfloat16)
    gk = _host(kd)
    for b in range(B):
        rows = slice(int(L[b]), int(L[b]) + T)
        _close(gk[b, rows], want_k[b, rows], kh[b, rows], torch.bfloat16)


# ----------------------------------------------------------------------------
# rotation inside the attention kernels (positions passed to verify_attn_*)
# ----------------------------------------------------------------------------

def _to_dtype(x64, dtype):
    """The oracle's f64 rotation rounded once to the element type (what the
    separate rotation pass stores and the fused kernels feed their MMAs)."""
    return torch.from_numpy(np.ascontiguousarray(x64)).to(dtype)


def _rotated_copy(w, pos, base):
    """A copy of workload w whose q and draft key rows carry the oracle's
    rotation at pos (rounded to w's element type)."""
    import copy

    r = copy.copy(w)
    dt = w.q.dtype
    if w.layout == "paged":
        q64, k64 = oracle.rope_draft_paged(_host(w.q), _host(w.k_pages), w.page_table, w.page_size, w.seqlens, pos,
                                           base)
        r.k_pages = _to_dtype(k64, dt)
    else:
        q64, k64 = oracle.rope_draft_dense(_host(w.q), _host(w.k_cache), w.seqlens, pos, base)
        r.k_cache = _to_dtype(k64, dt)
    r.q = _to_dtype(q64, dt)
    return r


FUSED_CASES = {
    # keys on TMEM lanes: 16 / 32 / 64 packed rows, TMA tiles and gathers
    "tck16_dense": ("chain", dict(B=2, Hq=8, Hkv=2, T=4, L_lo=1500, L_hi=3000), "parent", None),
    "tck32_dense": ("chain", dict(B=2, Hkv=2, Hq=8, L_lo=1500, L_hi=5000), "parent", None),
    "tck64_paged16": ("paged", dict(B=3, Hkv=2, Hq=8, L_lo=1500, L_hi=2500, page_size=16), "mask", None),
    "tck64_paged4": ("paged", dict(B=3, Hkv=2, Hq=8, L_lo=1500, L_hi=2500, page_size=4), "mask", None),
    "tck32_sparse": ("sparse", dict(B=2, Hkv=2, Hq=8, T=8, L_lo=3000, L_hi=5000, budget=600, m_draft=200,
                                    window=64), "parent", None),
    # rows on TMEM lanes: one and two M-tiles, 64-key kernel and the two-M-tile kernel
    "tc1_dense": ("tree", dict(B=2, Hkv=2, Hq=8, T=24, L=2600, depth=4), "parent", None),
    "tc2_dense": ("tree", dict(B=2, Hkv=2, Hq=8, L_lo=1500, L_hi=3000), "parent", None),
    "tcp_dense": ("tree", dict(B=2, Hkv=2, Hq=8, L_lo=1500, L_hi=3000), "parent", ("VA_MANY_ROWS_KERNEL", "tcp")),
    # 464 segments with the 32 KB rotary table: the rows-on-lanes kernel's
    # shared memory holds only its 3-stage ring then
    "tc2_short_ring": ("tree", dict(B=58, Hkv=8, Hq=32, L=1500), "parent", None),
    "tc1_paged16": ("paged", dict(B=2, Hkv=2, Hq=8, T=32, L_lo=1500, L_hi=2000, page_size=16, tree="depth", depth=5),
                    "parent", None),
    "tc2_sparse": ("sparse", dict(B=1, Hkv=2, Hq=8, T=40, L_lo=3000, L_hi=4000, budget=700, m_draft=200, window=64,
                                  tree="depth", depth=5), "parent", None),
    # mma.sync (bf16 d64, and d128 by route) and the fp32 SIMT path
    "mma_d64": ("chain", dict(B=2, Hq=32, Hkv=8, T=5, D=64, L_lo=1500, L_hi=3000), "parent", None),
    "mma_d128": ("chain", dict(B=2, Hkv=2, Hq=8, L_lo=1500, L_hi=3000), "parent", ("VA_SMALL_ROWS_KERNEL", "mma")),
    "fp32_tiny": ("tiny", dict(L=3000), "parent", None),
}


@pytest.mark.parametrize("kind", ["tree", "anchor", "large"])
@pytest.mark.parametrize("case", list(FUSED_CASES))
def test_rotation_inside_attention_matches_oracle(case, kind, monkeypatch):
    """One fused call on unrotated q and cache against the rotation oracle
    followed by the attention oracle, strict bars (prefixes of 1500 tokens or
    more keep |out| well below 0.5, where the bf16 rounding of the output
    itself stays under 1e-3); q and the cache are left untouched by the call."""
    name, over, mode, env = FUSED_CASES[case]
    if env is not None:
        monkeypatch.setenv(*env)
    w = W.make_workload(name, seed=len(case) * 31 + len(kind), **over)
    rng = np.random.default_rng(len(case) + 7 * len(kind))
    parent = w.parent if w.parent is not None else np.tile(np.arange(-1, w.T - 1), (w.B, 1))
    pos = _positions(kind, w.seqlens, w.T, parent, rng)
    base = 500000.0 if kind == "large" else 10000.0
    ref_w = _rotated_copy(w, pos, base)
    kw = {}
    if w.layout == "sparse":
        ref = oracle.verify(ref_w)
        kw = dict(indices=dev_i32(ref["indices"]), n_indices=dev_i32(ref["n_indices"]))
    else:
        ref = oracle.verify(ref_w)
    q = w.q.cuda()
    seqlens, dpos = dev_i32(w.seqlens), dev_i32(pos)
    drafts = dict(tree_parent=dev_i32(w.parent)) if mode == "parent" else dict(tree_mask=torch.from_numpy(
        np.ascontiguousarray(w.mask_words).view(np.int32)).cuda())
    if w.layout == "paged":
        k, v = w.k_pages.cuda(), w.v_pages.cuda()
        out, lse = va.verify_attn_paged(q, k, v, dev_i32(w.page_table), seqlens, positions=dpos, rope_base=base,
                                        **drafts)
    elif w.layout == "sparse":
        k, v = w.k_cache.cuda(), w.v_cache.cuda()
        out, lse = va.verify_attn_sparse(q, k, v, seqlens, kw["indices"], kw["n_indices"], positions=dpos,
                                         rope_base=base, **drafts)
    else:
        k, v = w.k_cache.cuda(), w.v_cache.cuda()
        out, lse = va.verify_attn_dense(q, k, v, seqlens, positions=dpos, rope_base=base, **drafts)
    torch.cuda.synchronize()
    if w.dtype == "fp32":
        compare(out, lse, ref, tol_out=1e-4, tol_lse=1e-4, strict=True)
    else:
        compare(out, lse, ref, strict=True)
    # nothing the caller passed in is written
    assert torch.equal(q.cpu(), w.q)
    assert torch.equal(k.cpu(), w.k_pages if w.layout == "paged" else w.k_cache)


def test_rotation_inside_attention_noalloc_and_equal_to_the_pass():
    """The fused rotation through the allocation-free entry point, and against
    the separate pass followed by an unrotated call: the same bf16 inputs reach
    the MMAs in both, so the results agree to the last bits but for the
    rounding of the rotation itself (fp32 in the kernels, fp64 in the pass)."""
    w = W.make_workload("chain", seed=301, L=4000)
    pos = (w.seqlens[:, None] + np.arange(w.T)[None]).astype(np.int32)
    q, k, v = w.q.cuda(), w.k_cache.cuda(), w.v_cache.cuda()
    seqlens, dpos, par = dev_i32(w.seqlens), dev_i32(pos), dev_i32(w.parent)
    fused, lse_f = va.api.verify_attn_dense_noalloc(q, k, v, seqlens, tree_parent=par, positions=dpos,
                                                    rope_base=10000.0)
    q2, k2 = q.clone(), k.clone()
    va.verify_rope_draft_dense(q2, k2, seqlens, dpos, 10000.0)
    sep, lse_s = va.verify_attn_dense(q2, k2, v, seqlens, tree_parent=par)
    torch.cuda.synchronize()
    assert float((fused.float() - sep.float()).abs().max()) <= 2e-3
    assert float((lse_f - lse_s).abs().max()) <= 1e-3
    compare(fused, lse_f, oracle.verify(_rotated_copy(w, pos, 10000.0)), strict=True)


def test_rotation_inside_attention_position_out_of_range_is_reported():
    w = W.make_workload("chain", seed=302, L=500)
    pos = (w.seqlens[:, None] + np.arange(w.T)[None]).astype(np.int32)
    pos[0, 3] = 1 << 25
    shape = va.make_shape(w.B, w.T, w.Hq, w.Hkv, w.D, 0, rope_base=10000.0)
    ws = va.Workspace.for_shape(shape)
    va.verify_attn_dense(w.q.cuda(), w.k_cache.cuda(), w.v_cache.cuda(), dev_i32(w.seqlens),
                         tree_parent=dev_i32(w.parent), positions=dev_i32(pos), rope_base=10000.0, workspace=ws)
    with pytest.raises(va.VerifyAttnError) as ei:
        va.verify_attn_check_status(ws)
    assert ei.value.status == va.api.VA_ERR_DEVICE_BOUNDS
