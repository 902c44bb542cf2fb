"""Property tests of the oracle's rotary embedding and importance map over
random shapes (hypothesis; skipped where it is not installed).  The
properties are the defining ones: a rotation keeps each pair's length,
rotations compose by adding positions, q.k depends on the positions only
through their difference; each (head, token) attention distribution has
unit mass, and permuting the committed rows permutes the importances."""
import numpy as np
import pytest

import oracle

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402


@settings(max_examples=60, deadline=None)
@given(half=st.integers(1, 64), pos=st.integers(-(1 << 20), 1 << 20), shift=st.integers(-5000, 5000),
       base=st.sampled_from([10000.0, 500000.0, 1e6]), seed=st.integers(0, 2**31 - 1))
def test_rope_properties(half, pos, shift, base, seed):
    rng = np.random.default_rng(seed)
    D = 2 * half
    q, k = rng.standard_normal((2, D))
    r = oracle.rope_rotate(q, pos, base)
    assert np.allclose(r[:half] ** 2 + r[half:] ** 2, q[:half] ** 2 + q[half:] ** 2, rtol=1e-9, atol=1e-12)
    assert np.allclose(oracle.rope_rotate(r, shift, base), oracle.rope_rotate(q, pos + shift, base), atol=1e-7)
    d1 = oracle.rope_rotate(q, pos, base) @ oracle.rope_rotate(k, pos - 7, base)
    d2 = oracle.rope_rotate(q, pos + shift, base) @ oracle.rope_rotate(k, pos + shift - 7, base)
    assert abs(d1 - d2) < 1e-7 * (1 + np.abs(q) @ np.abs(k))


@settings(max_examples=40, deadline=None)
@given(T=st.integers(1, 6), Hkv=st.integers(1, 3), group=st.integers(1, 3), D=st.sampled_from([4, 8, 16]),
       L=st.integers(1, 40), n_heads=st.integers(1, 4), scale=st.floats(0.05, 2.0), seed=st.integers(0, 2**31 - 1))
def test_importance_properties(T, Hkv, group, D, L, n_heads, scale, seed):
    rng = np.random.default_rng(seed)
    Hq = Hkv * group
    q = rng.standard_normal((1, T, Hq, D))
    k = rng.standard_normal((1, L + T, Hkv, D))
    heads = rng.integers(0, Hq, size=n_heads).tolist()
    Ls = np.array([L], np.int32)
    imp = oracle.head_importance(q, k, Ls, heads, scale)
    assert abs(imp[0].sum() - n_heads * T) < 1e-9 * n_heads * T
    assert np.all(imp[0, L:] == 0.0) and np.all(imp[0, :L] > 0.0)
    perm = rng.permutation(L)
    k2 = k.copy()
    k2[0, :L] = k[0, perm]
    imp2 = oracle.head_importance(q, k2, Ls, heads, scale)
    assert np.allclose(imp2[0, :L], imp[0, perm], rtol=1e-10, atol=1e-14)


@settings(max_examples=40, deadline=None)
@given(T=st.integers(1, 6), Hkv=st.integers(1, 2), group=st.integers(1, 3), D=st.sampled_from([4, 8]),
       n=st.integers(1, 24), density=st.floats(0.1, 1.0), scale=st.floats(0.05, 1.5),
       seed=st.integers(0, 2**31 - 1))
def test_masked_attention_against_torch(T, Hkv, group, D, n, density, scale, seed):
    """The C oracle's masked attention equals torch's fp64 softmax attention on
    random shapes and masks; rows with no visible key give out 0, lse -inf."""
    import torch

    rng = np.random.default_rng(seed)
    Hq = Hkv * group
    q = rng.standard_normal((T, Hq, D))
    k = rng.standard_normal((n, Hkv, D))
    v = rng.standard_normal((n, Hkv, D))
    vis = rng.random((T, n)) < density
    out, lse = oracle.masked_attention(q, k, v, vis, scale)
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(group, dim=0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(group, dim=0)
    m = torch.from_numpy(vis)
    s = torch.einsum("htd,hnd->htn", qt, kt) * scale
    s = s.masked_fill(~m, float("-inf"))
    want_lse = torch.logsumexp(s, dim=-1)  # [Hq][T]
    p = torch.where(m, torch.exp(s - want_lse[..., None].clamp_min(-1e300)), torch.zeros_like(s))
    want = torch.einsum("htn,hnd->htd", p, vt).permute(1, 0, 2).numpy()
    empty = ~vis.any(axis=1)
    assert np.allclose(out[~empty], want[~empty], rtol=0, atol=1e-11)
    assert np.all(out[empty] == 0.0)
    fin = ~empty
    assert np.allclose(lse[:, fin], want_lse.numpy()[:, fin], rtol=0, atol=1e-11)
    assert np.all(np.isneginf(lse[:, empty]))


@settings(max_examples=40, deadline=None)
@given(S=st.integers(1, 6), R=st.integers(1, 5), D=st.sampled_from([2, 4]), cut=st.integers(0, 6),
       seed=st.integers(0, 2**31 - 1))
def test_lse_merge_split_invariance(S, R, D, cut, seed):
    """Merging all parts at once equals merging two groups first and then their
    results (the merge is a softmax over the union of keys)."""
    rng = np.random.default_rng(seed)
    o = rng.standard_normal((S, R, D))
    lse = rng.standard_normal((S, R)) * 3
    full, full_lse = oracle.lse_merge(o, lse)
    c = min(cut, S)
    if 0 < c < S:
        a, la = oracle.lse_merge(o[:c], lse[:c])
        b, lb = oracle.lse_merge(o[c:], lse[c:])
        two, two_lse = oracle.lse_merge(np.stack([a, b]), np.stack([la, lb]))
        assert np.allclose(two, full, atol=1e-12) and np.allclose(two_lse, full_lse, atol=1e-12)
