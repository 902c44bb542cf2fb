"""Host-only checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports every symbol the headers declare, and rejects bad
arguments with the documented status before touching any device."""
import ctypes
import glob
import os
import re

import pytest

import speculative_decoding_verification_masked_gb300 as va
from speculative_decoding_verification_masked_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            if not m.group(0).lstrip().startswith(("typedef", "#")):
                names.add(m.group(1))
    return names


def test_library_builds_and_exports_every_declared_symbol():
    L = api.lib()
    names = _declared_functions()
    assert {"verify_attn_dense", "verify_attn_paged", "verify_attn_sparse", "verify_attn_combine",
            "verify_tree_mask_from_parents", "verify_build_index", "verify_attn_workspace_size",
            "verify_attn_check_status"} <= names
    for n in sorted(names):
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
    assert va.version().endswith("sm_103a")


FAKE = 1 << 20  # a non-NULL address validation never dereferences


def _shape(**kw):
    d = dict(B=1, T=8, Hq=32, Hkv=8, D=128, dtype=0, scale=0.088, rope_base=0.0)
    d.update(kw)
    return api.VaShape(d["B"], d["T"], d["Hq"], d["Hkv"], d["D"], d["dtype"], d["scale"], d["rope_base"])


def _dense(shape, parent=None, mask=None, ws=FAKE, q=FAKE, max_len=100, positions=None):
    L = api.lib()
    return L.verify_attn_dense(ctypes.byref(shape) if shape is not None else None, q, FAKE, FAKE, max_len, FAKE,
                               parent, mask, positions, FAKE, FAKE, ws, 1 << 30, None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=0), api.VA_ERR_INVALID_ARG),
    (dict(Hq=30), api.VA_ERR_INVALID_ARG),
    (dict(dtype=7), api.VA_ERR_INVALID_ARG),
    (dict(scale=0.0), api.VA_ERR_INVALID_ARG),
    (dict(T=65), api.VA_ERR_UNSUPPORTED),
    (dict(D=96), api.VA_ERR_UNSUPPORTED),
    (dict(dtype=2, D=128), api.VA_ERR_UNSUPPORTED),
    (dict(B=300, Hkv=8), api.VA_ERR_UNSUPPORTED),
])
def test_bad_shapes_rejected_on_host(kw, code):
    assert _dense(_shape(**kw)) == code
    assert api.lib().verify_attn_last_error()


def test_rotation_on_the_fly_needs_a_base():
    """positions given: the shape must carry the model's RoPE base (checked
    before anything is enqueued)."""
    assert _dense(_shape(), positions=FAKE) == api.VA_ERR_INVALID_ARG
    assert "rope_base" in api.lib().verify_attn_last_error().decode()
    assert _dense(_shape(rope_base=float("nan")), positions=FAKE) == api.VA_ERR_INVALID_ARG
    assert _dense(_shape(rope_base=-1.0), positions=FAKE) == api.VA_ERR_INVALID_ARG


def test_bad_pointers_rejected_on_host():
    assert _dense(None) == api.VA_ERR_INVALID_ARG
    assert _dense(_shape(), q=None) == api.VA_ERR_INVALID_ARG
    assert _dense(_shape(), parent=FAKE, mask=FAKE) == api.VA_ERR_INVALID_ARG
    assert _dense(_shape(), ws=None) == api.VA_ERR_WORKSPACE
    assert _dense(_shape(), ws=FAKE + 16) == api.VA_ERR_WORKSPACE
    assert _dense(_shape(), q=FAKE + 4) == api.VA_ERR_INVALID_ARG
    assert _dense(_shape(), max_len=3) == api.VA_ERR_INVALID_ARG


def test_paged_sparse_index_mask_combine_argument_checks():
    L = api.lib()
    s = _shape()
    bad_page = L.verify_attn_paged(ctypes.byref(s), FAKE, FAKE, FAKE, 10, 12, FAKE, 4, FAKE, None, None, None, FAKE,
                                   FAKE, FAKE, 1 << 30, None)
    assert bad_page == api.VA_ERR_INVALID_ARG
    no_idx = L.verify_attn_sparse(ctypes.byref(s), FAKE, FAKE, FAKE, 100, FAKE, None, FAKE, 16, None, None, None,
                                  FAKE, FAKE, FAKE, 1 << 30, None)
    assert no_idx == api.VA_ERR_INVALID_ARG
    assert L.verify_build_index(1, 1, FAKE, FAKE, FAKE, 100, 4, 256, 10, 200, FAKE, FAKE, None, None) == \
        api.VA_ERR_INVALID_ARG  # budget < sinks + window
    assert L.verify_tree_mask_from_parents(1, 65, FAKE, FAKE, None, None) == api.VA_ERR_UNSUPPORTED
    assert L.verify_attn_combine(4, 0, 128, FAKE, FAKE, 0, FAKE, FAKE, None) == api.VA_ERR_INVALID_ARG
    assert L.verify_attn_combine(4, 2, 96, FAKE, FAKE, 0, FAKE, FAKE, None) == api.VA_ERR_UNSUPPORTED
    assert L.verify_attn_workspace_size(None) == 0


def test_acceptance_and_commit_argument_checks():
    """The after-verification entry points reject bad arguments on the host,
    before any device work."""
    L = api.lib()
    acc = L.verify_accept_greedy
    assert acc(0, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == api.VA_ERR_INVALID_ARG
    assert acc(1, 65, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == api.VA_ERR_UNSUPPORTED
    assert acc(1, 4, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, None) == api.VA_ERR_INVALID_ARG
    assert acc(1, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 16, None) == api.VA_ERR_WORKSPACE
    s = _shape()
    dense = L.verify_commit_kv_dense
    assert dense(None, FAKE, FAKE, 100, FAKE, FAKE, FAKE, None, None, None) == api.VA_ERR_INVALID_ARG
    assert dense(ctypes.byref(s), None, FAKE, 100, FAKE, FAKE, FAKE, None, None, None) == api.VA_ERR_INVALID_ARG
    assert dense(ctypes.byref(s), FAKE + 4, FAKE, 100, FAKE, FAKE, FAKE, None, None, None) == api.VA_ERR_INVALID_ARG
    assert dense(ctypes.byref(s), FAKE, FAKE, 3, FAKE, FAKE, FAKE, None, None, None) == api.VA_ERR_INVALID_ARG
    # seqlens_out must not alias seqlens
    assert dense(ctypes.byref(s), FAKE, FAKE, 100, FAKE + 256, FAKE, FAKE, FAKE + 256, None, None) == \
        api.VA_ERR_INVALID_ARG
    big = _shape(T=65)
    assert dense(ctypes.byref(big), FAKE, FAKE, 100, FAKE, FAKE, FAKE, None, None, None) == api.VA_ERR_UNSUPPORTED
    paged = L.verify_commit_kv_paged
    assert paged(ctypes.byref(s), FAKE, FAKE, 10, 12, FAKE, 4, FAKE, FAKE, FAKE, None, None, None) == \
        api.VA_ERR_INVALID_ARG  # page size not a power of two
    assert paged(ctypes.byref(s), FAKE, FAKE, 10, 16, None, 4, FAKE, FAKE, FAKE, None, None, None) == \
        api.VA_ERR_INVALID_ARG  # no page table


def test_head_importance_argument_checks():
    """The scoring pass rejects bad shapes, head lists and buffers on the host."""
    L = api.lib()
    f = L.verify_head_importance

    def call(shape=None, heads=(3, 17), q=FAKE, scratch=FAKE, nbytes=1 << 30, max_len=100, stride=100, ws=None):
        s = shape or _shape(T=5)
        harr = (ctypes.c_int32 * max(1, len(heads)))(*heads)
        return f(ctypes.byref(s), q, FAKE, max_len, FAKE, ctypes.cast(harr, ctypes.c_void_p), len(heads), FAKE,
                 stride, scratch, nbytes, ws, None)

    assert call(heads=(3, 32)) == api.VA_ERR_INVALID_ARG        # head out of range
    assert call(heads=()) == api.VA_ERR_INVALID_ARG             # empty list
    assert call(heads=tuple(range(33))) == api.VA_ERR_UNSUPPORTED  # more than 32 heads
    assert call(shape=_shape(T=64), heads=(0, 1, 2, 3, 4)) == api.VA_ERR_UNSUPPORTED  # 320 rows
    assert call(shape=_shape(T=5, D=64)) == api.VA_ERR_UNSUPPORTED
    assert call(shape=_shape(T=5, dtype=2, D=64)) == api.VA_ERR_UNSUPPORTED
    assert call(shape=_shape(T=5, Hq=30)) == api.VA_ERR_INVALID_ARG
    assert call(q=None) == api.VA_ERR_INVALID_ARG
    assert call(q=FAKE + 8) == api.VA_ERR_INVALID_ARG
    assert call(scratch=FAKE + 16) == api.VA_ERR_WORKSPACE
    assert call(nbytes=1024) == api.VA_ERR_WORKSPACE
    assert call(ws=FAKE + 16) == api.VA_ERR_WORKSPACE
    assert call(stride=0) == api.VA_ERR_INVALID_ARG
    need = L.verify_head_importance_scratch_size(16, 5, 2, 32773)
    chunks = (32773 + 127) // 128  # 128-key chunks of the score pass
    assert need == 16 * 10 * chunks * 128 * 4 + (-(-16 * chunks * 10 * 8 // 256)) * 256
    assert L.verify_head_importance_scratch_size(0, 5, 2, 100) == 0


def test_rope_argument_checks():
    L = api.lib()
    d = L.verify_rope_draft_dense
    p = L.verify_rope_draft_paged
    s = _shape(T=5)
    assert d(None, FAKE, FAKE, 100, FAKE, FAKE, 10000.0, None, None) == api.VA_ERR_INVALID_ARG
    assert d(ctypes.byref(s), None, FAKE, 100, FAKE, FAKE, 10000.0, None, None) == api.VA_ERR_INVALID_ARG
    assert d(ctypes.byref(s), FAKE, FAKE, 100, FAKE, None, 10000.0, None, None) == api.VA_ERR_INVALID_ARG
    assert d(ctypes.byref(s), FAKE, FAKE, 100, FAKE, FAKE, 0.0, None, None) == api.VA_ERR_INVALID_ARG
    assert d(ctypes.byref(s), FAKE, FAKE, 100, FAKE, FAKE, float("inf"), None, None) == api.VA_ERR_INVALID_ARG
    assert d(ctypes.byref(s), FAKE + 1, FAKE, 100, FAKE, FAKE, 10000.0, None, None) == api.VA_ERR_INVALID_ARG
    assert d(ctypes.byref(s), FAKE, FAKE, 4, FAKE, FAKE, 10000.0, None, None) == api.VA_ERR_INVALID_ARG
    assert d(ctypes.byref(_shape(T=5, D=65)), FAKE, FAKE, 100, FAKE, FAKE, 1e4, None, None) == api.VA_ERR_UNSUPPORTED
    assert d(ctypes.byref(_shape(T=5, D=258)), FAKE, FAKE, 100, FAKE, FAKE, 1e4, None, None) == api.VA_ERR_UNSUPPORTED
    assert d(ctypes.byref(_shape(T=65)), FAKE, FAKE, 100, FAKE, FAKE, 1e4, None, None) == api.VA_ERR_UNSUPPORTED
    assert d(ctypes.byref(s), FAKE, FAKE, 100, FAKE, FAKE, 1e4, FAKE + 16, None) == api.VA_ERR_WORKSPACE
    assert p(ctypes.byref(s), FAKE, FAKE, 10, 12, FAKE, 4, FAKE, FAKE, 1e4, None, None) == api.VA_ERR_INVALID_ARG
    assert p(ctypes.byref(s), FAKE, FAKE, 10, 16, None, 4, FAKE, FAKE, 1e4, None, None) == api.VA_ERR_INVALID_ARG
