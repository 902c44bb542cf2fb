"""GPU parity of the steps after verification: greedy tree acceptance and the
KV commit, against the oracle (bit-exact: integer results and copied rows)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_masked_gb300 as va
import workloads as W
from tests.gpu_util import dev_i32

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _accept_case(seed, B, T, vocab):
    rng = np.random.default_rng(seed)
    parent = np.stack([W.random_parents(T, rng) for _ in range(B)]).astype(np.int32)
    draft = rng.integers(0, vocab, size=(B, T)).astype(np.int32)
    tgt = rng.integers(0, vocab, size=(B, T + 1)).astype(np.int32)
    return parent, draft, tgt


def _gpu_accept(parent, draft, tgt, ws=None):
    path, n, bonus = va.verify_accept_greedy(dev_i32(parent), dev_i32(draft), dev_i32(tgt), workspace=ws)
    torch.cuda.synchronize()
    return path.cpu().numpy(), n.cpu().numpy(), bonus.cpu().numpy()


def test_accept_hand_fixture():
    with open(os.path.join(GOLD, "greedy_accept_hand.json")) as f:
        g = json.load(f)
    path, n, bonus = _gpu_accept(np.array(g["parent"]), np.array(g["draft_tokens"]), np.array(g["target_next"]))
    assert path.tolist() == g["path"] and n.tolist() == g["n_accept"] and bonus.tolist() == g["bonus"]


@pytest.mark.parametrize("T", [1, 2, 7, 31, 32, 33, 63, 64])
@pytest.mark.parametrize("vocab", [2, 3, 50])
def test_accept_matches_oracle(T, vocab):
    parent, draft, tgt = _accept_case(T * 100 + vocab, 37, T, vocab)
    parent[0] = W.chain_parents(T)
    draft[1] = tgt[1, :T]  # a chain-like row where many nodes match
    got = _gpu_accept(parent, draft, tgt)
    want = oracle.greedy_accept(parent, draft, tgt)
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


def test_accept_bad_parent_is_reported():
    ws = va.Workspace(256)
    parent = np.array([[-1, 0, 5, 1]], np.int32)  # parent[2] = 5 is not earlier
    draft = np.array([[1, 2, 3, 4]], np.int32)
    tgt = np.array([[1, 2, 3, 3, 9]], np.int32)
    path, n, bonus = _gpu_accept(parent, draft, tgt, ws)
    with pytest.raises(va.VerifyAttnError) as ei:
        va.verify_attn_check_status(ws)
    assert ei.value.status == va.api.VA_ERR_DEVICE_BOUNDS
    # node 2 counts as rejected (and as a root for the walk): the same as a
    # tree where it hangs off the prefix with a token nobody predicts
    want_path, want_n, want_b = oracle.greedy_accept(np.array([[-1, 0, -1, 1]], np.int32),
                                                     np.array([[1, 2, -7, 4]], np.int32), tgt)
    assert n.tolist() == want_n.tolist() and path.tolist() == want_path.tolist() and bonus.tolist() == want_b.tolist()


def _dense_case(seed, B, T, Hkv, D, dtype, extra=5):
    rng = np.random.default_rng(seed)
    L = rng.integers(0, 300, size=B).astype(np.int32)
    L[0] = 0
    cap = int(L.max()) + T + extra
    k = torch.from_numpy(rng.standard_normal((B, cap, Hkv, D)).astype(np.float32)).to(dtype)
    v = torch.from_numpy(rng.standard_normal((B, cap, Hkv, D)).astype(np.float32)).to(dtype)
    return L, k, v


def _bits(t):
    t = t.contiguous().cpu()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.view(torch.int32).numpy()


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 64)])
@pytest.mark.parametrize("T", [1, 5, 16, 64])
def test_commit_dense_matches_oracle(dtype, D, T):
    B, Hkv = 6, 3
    L, k, v = _dense_case(T + D, B, T, Hkv, D, dtype)
    parent, draft, tgt = _accept_case(T + 7, B, T, 2)
    path, n, _ = oracle.greedy_accept(parent, draft, tgt)
    path[0, :T] = np.arange(T)  # sequence 0: everything accepted in place (nothing moves)
    n[0] = T
    n[1] = 0  # sequence 1: nothing accepted
    path[1] = -1
    kw, vw, Lw = oracle.commit_kv_dense(_bits(k), _bits(v), L, path, n)
    kd, vd = k.cuda(), v.cuda()
    Lo = va.verify_commit_kv_dense(kd, vd, dev_i32(L), dev_i32(path), dev_i32(n))
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kd), kw) and np.array_equal(_bits(vd), vw)
    assert Lo.cpu().numpy().tolist() == Lw.tolist()


@pytest.mark.parametrize("page_size", [1, 4, 16, 64])
def test_commit_paged_matches_oracle(page_size):
    w = W.make_workload("paged", seed=page_size, B=5, L_lo=3, L_hi=300, page_size=page_size, spare_pages=4, T=16,
                        tree="random")
    rng = np.random.default_rng(page_size)
    draft = rng.integers(0, 2, size=(w.B, w.T)).astype(np.int32)
    tgt = rng.integers(0, 2, size=(w.B, w.T + 1)).astype(np.int32)
    path, n, _ = oracle.greedy_accept(w.parent, draft, tgt)
    kw, vw, Lw = oracle.commit_kv_paged(_bits(w.k_pages), _bits(w.v_pages), w.page_table, page_size, w.seqlens,
                                        path, n)
    kd, vd = w.k_pages.cuda(), w.v_pages.cuda()
    Lo = va.verify_commit_kv_paged(kd, vd, dev_i32(w.page_table), dev_i32(w.seqlens), dev_i32(path), dev_i32(n))
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kd), kw) and np.array_equal(_bits(vd), vw)
    assert Lo.cpu().numpy().tolist() == Lw.tolist()


def test_accept_then_commit_on_device():
    """The two steps chained on the device, at the paged workload's shape
    (B64, T16, 16-row pages), against the oracle chained on the host."""
    w = W.make_workload("paged", seed=3, tree="random", L_lo=100, L_hi=600)
    rng = np.random.default_rng(4)
    tgt = rng.integers(0, 3, size=(w.B, w.T + 1)).astype(np.int32)
    draft = rng.integers(0, 3, size=(w.B, w.T)).astype(np.int32)
    path_w, n_w, bonus_w = oracle.greedy_accept(w.parent, draft, tgt)
    kw, vw, Lw = oracle.commit_kv_paged(_bits(w.k_pages), _bits(w.v_pages), w.page_table, w.page_size, w.seqlens,
                                        path_w, n_w)
    path, n, bonus = va.verify_accept_greedy(dev_i32(w.parent), dev_i32(draft), dev_i32(tgt))
    kd, vd = w.k_pages.cuda(), w.v_pages.cuda()
    Lo = va.verify_commit_kv_paged(kd, vd, dev_i32(w.page_table), dev_i32(w.seqlens), path, n)
    torch.cuda.synchronize()
    assert np.array_equal(path.cpu().numpy(), path_w) and np.array_equal(bonus.cpu().numpy(), bonus_w)
    assert np.array_equal(_bits(kd), kw) and np.array_equal(_bits(vd), vw)
    assert Lo.cpu().numpy().tolist() == Lw.tolist()


def test_commit_bad_path_entry_is_reported_and_left_in_place():
    B, T, Hkv, D = 2, 4, 2, 64
    L, k, v = _dense_case(9, B, T, Hkv, D, torch.bfloat16)
    path = np.array([[2, 9, -1, -1], [1, 2, 3, -1]], np.int32)  # 9 is past the draft block
    n = np.array([2, 3], np.int32)
    ws = va.Workspace(256)
    kd, vd = k.cuda(), v.cuda()
    va.verify_commit_kv_dense(kd, vd, dev_i32(L), dev_i32(path), dev_i32(n), workspace=ws)
    with pytest.raises(va.VerifyAttnError) as ei:
        va.verify_attn_check_status(ws)
    assert ei.value.status == va.api.VA_ERR_DEVICE_BOUNDS
    fixed = path.copy()
    fixed[0, 1] = 1  # the bad entry's row stays where it is
    kw, vw, _ = oracle.commit_kv_dense(_bits(k), _bits(v), L, fixed, n)
    assert np.array_equal(_bits(kd), kw) and np.array_equal(_bits(vd), vw)
