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
