"""GPU parity of the head-importance scoring pass against the oracle.

Tolerance, from the arithmetic: the kernel forms each score q.k from the same
bf16 values as the oracle, with fp32 accumulation of 128 products (error of a
few 1e-5 in a score of a few units), scaled into base 2, and exponentiates
with the hardware's 2^x (relative error ~2^-22).  An error e in a score moves
the probability by a relative e * ln 2, and the row's log-sum-exp adds one
more such term; each importance is a sum of such probabilities, so the bar is
relative: |gpu - oracle| <= 2e-4 |oracle| (plus 1e-12 for the flushed
subnormal tail), with every kv-head row bit-identical and untouched entries
past each L_b.
"""
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

RTOL = 2e-4
ATOL = 1e-12
SENTINEL = -7.0


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _case(seed, B, T, Hq, Hkv, seqlens, extra=3):
    rng = np.random.default_rng(seed)
    cap = int(max(seqlens)) + T + extra
    q = torch.from_numpy(rng.standard_normal((B, T, Hq, 128)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((B, cap, Hkv, 128)).astype(np.float32)).to(torch.bfloat16)
    return q, k, np.asarray(seqlens, np.int32)


def _run(q, k, L, heads, scale, stride=None, ws=None):
    B, _, Hkv = q.shape[0], q.shape[1], k.shape[2]
    stride = stride or k.shape[1]
    score = torch.full((B, Hkv, stride), SENTINEL, dtype=torch.float32, device="cuda")
    va.verify_head_importance(q.cuda(), k.cuda(), dev_i32(L), heads, score=score, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    return score.cpu().numpy()


def _check(got, want, L, R):
    B, Hkv, stride = got.shape
    for b in range(B):
        n = int(L[b])
        for g in range(Hkv):
            assert np.array_equal(got[b, g], got[b, 0]), "kv-head rows differ"
        row = got[b, 0]
        assert np.all(row[n:] == SENTINEL), "entries past L were written"
        err = np.abs(row[:n].astype(np.float64) - want[b, :n])
        bound = RTOL * np.abs(want[b, :n]) + ATOL
        assert np.all(err <= bound), f"seq {b}: worst excess {(err - bound).max():.3e} (L={n})"
        if n:
            assert abs(row[:n].astype(np.float64).sum() - R) <= 1e-4 * R


@pytest.mark.parametrize("T,heads", [(1, [1]), (5, [1, 6]), (5, [0, 1, 2]), (5, [5, 5]), (16, [3, 4]),
                                     (8, [7, 0, 3, 4, 2])])
def test_importance_matches_oracle(T, heads):
    """Ragged prefixes around the 128-key chunk and 1024-key block edges, one
    empty sequence; units split by kv-head and at 8 rows."""
    L = [1, 255, 256, 257, 1023, 1500, 3000, 0]
    q, k, L = _case(T * 31 + len(heads), len(L), T, 8, 2, L)
    got = _run(q, k, L, heads, 0.0884)
    want = oracle.head_importance(_bits(q), _bits(k), L, heads, 0.0884)
    _check(got, want, L, len(heads) * T)


def test_importance_unaligned_stride_and_scale():
    """An output stride that is not a multiple of 4 (scalar stores) and a
    larger score scale (sharper distributions)."""
    L = [700, 1025, 33]
    q, k, L = _case(5, 3, 4, 4, 4, L)
    got = _run(q, k, L, [2, 3], 0.3, stride=k.shape[1] + 1)
    want = oracle.head_importance(_bits(q), _bits(k), L, [2, 3], 0.3)
    _check(got, want, L, 8)


def test_importance_full_size_sparse_workload():
    """The sparse workload's shape (B16, T5, Hq32/Hkv8, prefixes 16K-32K) and
    its two synthetic retrieval heads, every position checked."""
    w = W.make_workload("sparse", seed=0)
    got = _run(w.q, w.k_cache, w.seqlens, list(w.score_heads), w.scale)
    want = oracle.head_importance(_bits(w.q), _bits(w.k_cache), w.seqlens, list(w.score_heads), w.scale)
    _check(got, want, w.seqlens, len(w.score_heads) * w.T)


def test_importance_bad_seqlen_is_reported_and_clamped():
    L = np.array([300, 10_000], np.int32)  # the second is past the cache
    q, k, _ = _case(9, 2, 2, 8, 2, [300, 300])
    ws = va.Workspace(256)
    got = _run(q, k, L, [1], 0.0884, ws=ws)
    with pytest.raises(va.VerifyAttnError) as ei:
        va.verify_attn_check_status(ws)
    assert ei.value.status == va.api.VA_ERR_DEVICE_BOUNDS
    cap = k.shape[1]
    want = oracle.head_importance(_bits(q), _bits(k), np.array([300, cap], np.int32), [1], 0.0884)
    _check(got, want, np.array([300, cap]), 2)


def test_importance_feeds_the_index_builder():
    """The map goes straight into verify_build_index as its target signal; the
    set it selects is valid for those scores: sinks and window present, the
    size min(budget, L), and no unchosen candidate scores above a chosen one
    outside the draft picks."""
    w = W.make_workload("sparse", seed=2, B=4, L_lo=3000, L_hi=5000, budget=512, window=64, m_draft=100)
    sd = torch.from_numpy(w.score_draft).cuda()
    imp = torch.zeros_like(sd)
    va.verify_head_importance(w.q.cuda(), w.k_cache.cuda(), dev_i32(w.seqlens), list(w.score_heads), score=imp,
                              scale=w.scale)
    idx, n = va.verify_build_index(dev_i32(w.seqlens), sd, imp, w.n_sink, w.window, w.m_draft, w.budget)
    idx, n, imp_h = idx.cpu().numpy(), n.cpu().numpy(), imp.cpu().numpy()
    for b in range(w.B):
        L = int(w.seqlens[b])
        fixed = set(range(w.n_sink)) | set(range(L - w.window, L))
        for h in range(w.Hkv):
            sel = idx[b, h, : n[b, h]]
            assert n[b, h] == min(w.budget, L) and np.all(np.diff(sel) > 0)
            assert fixed <= set(sel.tolist())
            cand = np.setdiff1d(np.arange(L), np.array(sorted(fixed)))
            sd_b = w.score_draft[b, h, :L]
            order = np.lexsort((cand, -sd_b[cand]))
            draft_pick = set(cand[order[: w.m_draft]].tolist())
            rest_sel = np.array(sorted(set(sel.tolist()) - fixed - draft_pick))
            rest_out = np.array(sorted(set(cand.tolist()) - set(sel.tolist())))
            if len(rest_sel) and len(rest_out):
                assert imp_h[b, h, rest_sel].min() >= imp_h[b, h, rest_out].max()


@pytest.mark.parametrize("T,Hq,Hkv,heads", [(64, 8, 2, [0, 1, 4, 5]), (8, 32, 8, list(range(32)))])
def test_importance_largest_row_counts(T, Hq, Hkv, heads):
    """256 rows: 64 tokens of four heads on two kv-heads, and all 32 heads of
    eight kv-heads -- the row and head limits, 32 units."""
    L = [300, 129, 1]
    q, k, L = _case(T + Hq, len(L), T, Hq, Hkv, L)
    got = _run(q, k, L, heads, 0.0884)
    want = oracle.head_importance(_bits(q), _bits(k), L, heads, 0.0884)
    _check(got, want, L, len(heads) * T)
