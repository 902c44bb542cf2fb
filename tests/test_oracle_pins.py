"""Pins for the fp64 oracle: it is checked against things other than itself.

* a pure-Python brute force written independently (oracle/twin.py);
* torch's scaled_dot_product_attention / logsumexp in float64 (library routines);
* closed forms and hand-derived fixtures under tests/golden/;
* the invariants the method rests on: divide-and-aggregate exactness
  (LongSpec 2.C), chain = causal, full verify set = dense (Dustin 3),
  paged = contiguous (HiSpec 2), tree relabelling, mask monotonicity;
* networkx's ancestor relation for the tree visibility.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import twin
import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _f64(a):
    """Host array (bf16 bits / fp32 / fp64) -> float64 by exact widening, test side."""
    if isinstance(a, torch.Tensor):
        return a.to(torch.float64).numpy()
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _rand_case(seed, T=5, Hq=4, Hkv=2, D=8, n=11, dtype="fp32", density=0.6):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, Hq, D)).astype(np.float32)
    k = rng.standard_normal((n, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((n, Hkv, D)).astype(np.float32)
    vis = rng.random((T, n)) < density
    if dtype == "bf16":
        q, k, v = (W.bf16_bits(torch.from_numpy(x).to(torch.bfloat16)) for x in (q, k, v))
    return q, k, v, vis


def _sdpa(q, k, v, vis, scale):
    """torch float64 SDPA with an explicit boolean mask; GQA by repeating kv heads."""
    q, k, v = (torch.from_numpy(_f64(x)) for x in (q, k, v))
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    qh = q.permute(1, 0, 2)  # [Hq][T][D]
    kh = k.permute(1, 0, 2).repeat_interleave(g, dim=0)
    vh = v.permute(1, 0, 2).repeat_interleave(g, dim=0)
    m = torch.from_numpy(np.asarray(vis, dtype=bool))
    out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=m, scale=scale)
    scores = torch.einsum("htd,hnd->htn", qh, kh) * scale
    lse = torch.logsumexp(scores.masked_fill(~m, float("-inf")), dim=-1)  # [Hq][T]
    return out.permute(1, 0, 2).numpy(), lse.numpy()


# ----------------------------------------------------------------------------
# cross-implementation pins
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_c_oracle_matches_pure_python_twin(seed, dtype):
    q, k, v, vis = _rand_case(seed, dtype=dtype)
    vis[0, :] = False  # one row with no visible key (C10 reading: out 0, lse -inf)
    scale = 1 / math.sqrt(q.shape[-1])
    out, lse = oracle.masked_attention(q, k, v, vis, scale)
    tout, tlse = twin.attention(_f64(q).tolist(), _f64(k).tolist(), _f64(v).tolist(), vis.tolist(), scale)
    np.testing.assert_allclose(out, np.array(tout), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(tlse), rtol=0, atol=1e-12)
    assert np.all(np.isneginf(lse[:, 0]))


@pytest.mark.parametrize("seed", range(4))
def test_masked_attention_matches_torch_sdpa(seed):
    q, k, v, vis = _rand_case(100 + seed, T=7, Hq=8, Hkv=2, D=16, n=40, dtype="bf16")
    vis[:, 0] = True  # every row sees at least one key (SDPA cannot express an empty row)
    scale = 0.3
    out, lse = oracle.masked_attention(q, k, v, vis, scale)
    ref, ref_lse = _sdpa(q, k, v, vis, scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_single_token_self_only_is_plain_decode_attention():
    """T=1 with the root alone: verification reduces to one decode step over prefix + itself."""
    w = W.make_workload("tiny", seed=3, T=1, L=37)
    r = oracle.verify(w)
    q = w.q[0].numpy()                    # [1][Hq][D]
    k = w.k_cache[0, :38].numpy()         # prefix + the token itself
    v = w.v_cache[0, :38].numpy()
    ref, ref_lse = _sdpa(q, k, v, np.ones((1, 38), bool), w.scale)
    np.testing.assert_allclose(r["out"][0], ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["lse"][0], ref_lse, rtol=0, atol=1e-12)


def test_chain_is_causal_attention():
    """A draft chain gives the textbook causal mask over prefix + draft."""
    w = W.make_workload("chain", seed=1, L=45, Hq=4, Hkv=2, D=16)
    vis = oracle.draft_visibility(w)
    assert np.array_equal(vis[0], np.tril(np.ones((w.T, w.T), bool)))
    r = oracle.verify(w)
    L, T = 45, w.T
    causal = torch.ones(T, L + T, dtype=torch.bool).tril(diagonal=L).numpy()
    ref, ref_lse = _sdpa(W.bf16_bits(w.q[0]), W.bf16_bits(w.k_cache[0, :L + T]),
                         W.bf16_bits(w.v_cache[0, :L + T]), causal, w.scale)
    np.testing.assert_allclose(r["out"][0], ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["lse"][0], ref_lse, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# closed forms and hand-derived fixtures
# ----------------------------------------------------------------------------

def test_golden_hand_masked_softmax():
    g = json.load(open(os.path.join(GOLD, "masked_softmax_hand.json")))
    out, lse = oracle.masked_attention(np.array(g["q"]), np.array(g["k"]), np.array(g["v"]),
                                       np.array(g["visible"], bool), g["scale"])
    np.testing.assert_allclose(out, np.array(g["out"]), rtol=1e-14, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(g["lse"]), rtol=1e-14, atol=1e-14)


def test_zero_query_averages_visible_values():
    """q = 0 makes every score 0: out is the plain mean of the visible values, lse = ln(count)."""
    rng = np.random.default_rng(7)
    T, Hq, Hkv, D, n = 4, 2, 1, 8, 23
    q = np.zeros((T, Hq, D))
    k = rng.standard_normal((n, Hkv, D))
    v = rng.standard_normal((n, Hkv, D))
    vis = rng.random((T, n)) < 0.5
    vis[:, 3] = True
    out, lse = oracle.masked_attention(q, k, v, vis, 1.0)
    for i in range(T):
        np.testing.assert_allclose(out[i, 0], v[vis[i], 0].mean(axis=0), atol=1e-13)
        np.testing.assert_allclose(lse[:, i], math.log(vis[i].sum()), atol=1e-14)


def test_single_visible_key_returns_its_value():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((3, 2, 4))
    k = rng.standard_normal((5, 1, 4))
    v = rng.standard_normal((5, 1, 4))
    vis = np.zeros((3, 5), bool)
    vis[0, 2] = vis[1, 4] = vis[2, 0] = True
    out, lse = oracle.masked_attention(q, k, v, vis, 0.5)
    for i, j in [(0, 2), (1, 4), (2, 0)]:
        for h in range(2):
            np.testing.assert_allclose(out[i, h], v[j, 0], atol=1e-15)
            np.testing.assert_allclose(lse[h, i], 0.5 * q[i, h] @ k[j, 0], atol=1e-14)


def test_golden_tree_mask_and_networkx_ancestors():
    nx = pytest.importorskip("networkx")
    g = json.load(open(os.path.join(GOLD, "tree_mask_hand.json")))
    words = oracle.tree_mask_words(np.array([g["parent"]]))
    assert words[0, :, 0].tolist() == g["words"]
    rng = np.random.default_rng(11)
    for T in (1, 2, 7, 33, 64):
        for kind in ("random", "depth"):
            if kind == "depth" and T < 8:
                continue
            p = W.random_parents(T, rng) if kind == "random" else W.depth_tree_parents(T, 6, rng)[0]
            G = nx.DiGraph()
            G.add_nodes_from(range(T))
            G.add_edges_from((int(p[i]), i) for i in range(T) if p[i] >= 0)
            vis = oracle.tree_visibility(p)
            for i in range(T):
                expect = nx.ancestors(G, i) | {i}
                assert set(np.nonzero(vis[i])[0].tolist()) == expect


def test_tree_visibility_rejects_non_topological_parents():
    with pytest.raises(ValueError):
        oracle.tree_visibility(np.array([-1, 2, 0], np.int32))


def test_lse_merge_closed_forms():
    o1 = np.array([[[1.0, 2.0]]])
    o2 = np.array([[[3.0, -2.0]]])
    out, lse = oracle.lse_merge(np.concatenate([o1, o2]), np.array([[0.7], [0.7]]))
    np.testing.assert_allclose(out, [[2.0, 0.0]], atol=1e-15)      # equal partitions: plain mean
    np.testing.assert_allclose(lse, [0.7 + math.log(2)], atol=1e-15)
    out, lse = oracle.lse_merge(np.concatenate([o1, o2]), np.array([[-np.inf], [1.5]]))
    np.testing.assert_allclose(out, [[3.0, -2.0]], atol=0)           # an empty part contributes nothing
    np.testing.assert_allclose(lse, [1.5], atol=0)
    out, lse = oracle.lse_merge(np.concatenate([o1, o2]), np.array([[-np.inf], [-np.inf]]))
    assert np.all(out == 0) and np.isneginf(lse[0])
    # weights e^a/(e^a+e^b): ln 3 vs 0 -> 3/4, 1/4
    out, lse = oracle.lse_merge(np.concatenate([o1, o2]), np.array([[math.log(3)], [0.0]]))
    np.testing.assert_allclose(out, [[0.75 * 1 + 0.25 * 3, 0.75 * 2 - 0.25 * 2]], atol=1e-15)
    np.testing.assert_allclose(lse, [math.log(4)], atol=1e-15)


# ----------------------------------------------------------------------------
# invariants of the method
# ----------------------------------------------------------------------------

def _prefix_tree_split(q, k, v, vis, scale, cuts):
    """Attention over consecutive key ranges [c_i, c_{i+1}) merged by the oracle's LSE merge."""
    T, Hq, D = q.shape
    parts_o, parts_l = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, l = oracle.masked_attention(q, k[a:b], v[a:b], vis[:, a:b], scale)
        parts_o.append(o.reshape(T * Hq, D))
        parts_l.append(l.T.reshape(T * Hq))
    out, lse = oracle.lse_merge(np.stack(parts_o), np.stack(parts_l))
    return out.reshape(T, Hq, D), lse.reshape(T, Hq).T


def test_divide_and_aggregate_is_exact_at_every_split_point():
    """LongSpec 2.C: cache part (no mask) + speculative part (mask) merged by LSE = unsplit."""
    w = W.make_workload("tiny", seed=5, L=24, T=6, Hq=2, D=8)
    vis_t = oracle.draft_visibility(w)[0]
    L, T = 24, 6
    q = W.bf16_bits(w.q[0].to(torch.bfloat16))
    k = W.bf16_bits(w.k_cache[0, :L + T].to(torch.bfloat16))
    v = W.bf16_bits(w.v_cache[0, :L + T].to(torch.bfloat16))
    vis = np.concatenate([np.ones((T, L), bool), vis_t], axis=1)
    ref, ref_lse = oracle.masked_attention(q, k, v, vis, w.scale)
    for s in range(0, L + T + 1):
        out, lse = _prefix_tree_split(q, k, v, vis, w.scale, [0, s, L + T])
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)
    rng = np.random.default_rng(0)
    for _ in range(20):
        cuts = sorted(set([0, L + T] + rng.integers(0, L + T, size=4).tolist()))
        out, lse = _prefix_tree_split(q, k, v, vis, w.scale, cuts)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
        # merge order does not matter
        T_, Hq, D = q.shape
        parts = [oracle.masked_attention(q, k[a:b], v[a:b], vis[:, a:b], w.scale) for a, b in zip(cuts[:-1], cuts[1:])]
        perm = rng.permutation(len(parts))
        o2, l2 = oracle.lse_merge(np.stack([parts[p][0].reshape(-1, D) for p in perm]),
                                  np.stack([parts[p][1].T.reshape(-1) for p in perm]))
        np.testing.assert_allclose(o2.reshape(T_, Hq, D), ref, rtol=0, atol=1e-12)


def test_sparse_with_every_position_equals_dense():
    """Dustin 3-4: attention over a verify set that lists every cached position is dense attention."""
    w = W.make_workload("sparse", seed=2, B=2, Hq=4, Hkv=2, D=16, L_lo=30, L_hi=50, n_sink=2, window=4,
                        budget=64, m_draft=3)
    Lmax = int(w.seqlens.max())
    idx = np.full((w.B, w.Hkv, Lmax), -1, np.int32)
    cnt = np.zeros((w.B, w.Hkv), np.int32)
    for b in range(w.B):
        idx[b, :, : w.seqlens[b]] = np.arange(w.seqlens[b])
        cnt[b] = w.seqlens[b]
    rs = oracle.verify(w, indices=idx, n_indices=cnt)
    wd = W.make_workload("sparse", seed=2, B=2, Hq=4, Hkv=2, D=16, L_lo=30, L_hi=50, n_sink=2, window=4,
                         budget=64, m_draft=3, layout="dense")
    rd = oracle.verify(wd)
    np.testing.assert_array_equal(rs["out"], rd["out"])
    np.testing.assert_array_equal(rs["lse"], rd["lse"])


@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_paged_equals_contiguous(page_size):
    """HiSpec 2: attention through a block table equals attention over the contiguous sequence."""
    w = W.make_workload("paged", seed=4, B=3, Hq=4, Hkv=2, D=16, L_lo=5, L_hi=60, T=6, page_size=page_size,
                        spare_pages=3)
    r = oracle.verify(w)
    # rebuild a dense cache by hand from pages (independent of oracle.gather_pages)
    Lmax = int(w.seqlens.max()) + w.T
    kd = torch.zeros(w.B, Lmax, w.Hkv, w.D, dtype=torch.bfloat16)
    vd = torch.zeros_like(kd)
    for b in range(w.B):
        for t in range(int(w.seqlens[b]) + w.T):
            pg = int(w.page_table[b, t // page_size])
            kd[b, t] = w.k_pages[pg, t % page_size]
            vd[b, t] = w.v_pages[pg, t % page_size]
    vis = oracle.draft_visibility(w)
    out, lse = oracle.attention_dense(W.bf16_bits(w.q), W.bf16_bits(kd), W.bf16_bits(vd), w.seqlens, vis, w.scale)
    np.testing.assert_array_equal(r["out"], out)
    np.testing.assert_array_equal(r["lse"], lse)


def test_removing_a_mask_bit_changes_only_its_row():
    q, k, v, vis = _rand_case(21, T=6, n=15)
    vis[:, :3] = True
    out, lse = oracle.masked_attention(q, k, v, vis, 0.4)
    i, j = 4, int(np.nonzero(vis[4])[0][-1])
    vis2 = vis.copy()
    vis2[i, j] = False
    out2, lse2 = oracle.masked_attention(q, k, v, vis2, 0.4)
    other = [r for r in range(6) if r != i]
    np.testing.assert_array_equal(out2[other], out[other])
    np.testing.assert_array_equal(lse2[:, other], lse[:, other])
    assert np.abs(out2[i] - out[i]).max() > 1e-6


def test_tree_relabelling_permutes_outputs():
    """Renumbering tree nodes (keeping parent[i] < i) permutes queries and draft keys alike."""
    rng = np.random.default_rng(3)
    T, L = 9, 13
    parent = W.random_parents(T, rng)
    # a topological relabelling: order nodes by (depth, random key)
    depth = W.chain_depths(parent)
    order = sorted(range(T), key=lambda n: (depth[n], rng.random()))
    new = {o: i for i, o in enumerate(order)}
    parent2 = np.array([-1 if parent[o] < 0 else new[int(parent[o])] for o in order], np.int32)
    q, k, v, _ = _rand_case(5, T=T, n=L + T)
    vis1 = np.concatenate([np.ones((T, L), bool), oracle.tree_visibility(parent)], 1)
    vis2 = np.concatenate([np.ones((T, L), bool), oracle.tree_visibility(parent2)], 1)
    q2 = q[order]
    keyperm = list(range(L)) + [L + o for o in order]
    out1, lse1 = oracle.masked_attention(q, k, v, vis1, 0.3)
    out2, lse2 = oracle.masked_attention(q2, k[keyperm], v[keyperm], vis2, 0.3)
    np.testing.assert_allclose(out2, out1[order], atol=1e-13)
    np.testing.assert_allclose(lse2, lse1[:, order], atol=1e-13)


# ----------------------------------------------------------------------------
# verify-set selection (Dustin section 1)
# ----------------------------------------------------------------------------

def _brute_index(sd, st, L, n_sink, window, m, budget):
    """Selection by explicit Python sorting, no numpy."""
    fixed = sorted(set(range(min(n_sink, L))) | set(range(max(0, L - window), L)))
    cand = [p for p in range(L) if p not in fixed]
    room = budget - len(fixed)
    dpick = sorted(cand, key=lambda p: (-float(sd[p]), p))[: max(0, min(m, room))]
    rest = [p for p in cand if p not in dpick]
    tpick = sorted(rest, key=lambda p: (-float(st[p]), p))[: max(0, room - len(dpick))]
    return sorted(fixed + dpick + tpick)


def test_golden_verify_index_hand():
    g = json.load(open(os.path.join(GOLD, "verify_index_hand.json")))
    L = g["L"]
    sd = np.full((1, 1, L), g["score_draft"]["default"], np.float32)
    st = np.full((1, 1, L), g["score_target"]["default"], np.float32)
    for p, s in g["score_draft"]["set"].items():
        sd[0, 0, int(p)] = s
    for p, s in g["score_target"]["set"].items():
        st[0, 0, int(p)] = s
    idx, cnt = oracle.build_verify_index(sd, st, np.array([L]), g["n_sink"], g["window"], g["m_draft"],
                                         g["budget"])
    assert cnt[0, 0] == len(g["indices"])
    assert idx[0, 0, : cnt[0, 0]].tolist() == g["indices"]


@pytest.mark.parametrize("seed", range(5))
def test_verify_index_matches_brute_force_and_invariants(seed):
    rng = np.random.default_rng(seed)
    B, Hkv = 3, 2
    seqlens = np.array([7, 40, 90])
    # coarse scores force many ties
    sd = (rng.integers(0, 6, size=(B, Hkv, 90)) / 5).astype(np.float32)
    st = (rng.integers(0, 6, size=(B, Hkv, 90)) / 5).astype(np.float32)
    n_sink, window, m, budget = 3, 5, 6, 20
    idx, cnt = oracle.build_verify_index(sd, st, seqlens, n_sink, window, m, budget)
    for b in range(B):
        L = int(seqlens[b])
        for h in range(Hkv):
            sel = idx[b, h, : cnt[b, h]].tolist()
            assert sel == _brute_index(sd[b, h], st[b, h], L, n_sink, window, m, budget)
            assert len(sel) == min(budget, L)
            assert sel == sorted(set(sel)) and all(0 <= p < L for p in sel)
            assert set(range(min(n_sink, L))) <= set(sel)
            assert set(range(max(0, L - window), L)) <= set(sel)
            assert np.all(idx[b, h, cnt[b, h]:] == -1)


def test_verify_index_rejects_budget_below_fixed_part():
    with pytest.raises(ValueError):
        oracle.build_verify_index(np.zeros((1, 1, 9), np.float32), np.zeros((1, 1, 9), np.float32),
                                  np.array([9]), 4, 4, 0, 7)


def test_draft_block_masks():
    """FlexDraft 1: masked tokens see their own block bidirectionally; across blocks isolated or causal."""
    iso = W.block_draft_mask(8, 4, "isolated")
    cau = W.block_draft_mask(8, 4, "causal")
    words_iso = oracle.bool_to_words(iso)[:, 0].tolist()
    words_cau = oracle.bool_to_words(cau)[:, 0].tolist()
    assert words_iso == [0x0F] * 4 + [0xF0] * 4
    assert words_cau == [0x0F] * 4 + [0xFF] * 4
    assert np.array_equal(oracle.words_to_bool(W.pack_bits(cau), 8), cau)


# ----------------------------------------------------------------------------
# greedy acceptance and KV commit
# ----------------------------------------------------------------------------

def test_greedy_accept_hand():
    with open(os.path.join(GOLD, "greedy_accept_hand.json")) as f:
        g = json.load(f)
    path, n, bonus = oracle.greedy_accept(np.array(g["parent"], np.int32), np.array(g["draft_tokens"], np.int32),
                                          np.array(g["target_next"], np.int32))
    assert path.tolist() == g["path"]
    assert n.tolist() == g["n_accept"]
    assert bonus.tolist() == g["bonus"]


def _accept_brute_force(parent, draft, tgt):
    """Every root path of the tree, taken whole: accepted when each of its nodes
    carries the target's token after its predecessor (the prefix for the first)."""
    T = len(parent)
    best = []
    for end in range(T):
        nodes = []
        t = end
        while t >= 0:
            nodes.append(t)
            t = parent[t]
        nodes = nodes[::-1]
        prev = -1
        good = True
        for t in nodes:
            if draft[t] != tgt[prev + 1]:
                good = False
                break
            prev = t
        if good and len(nodes) > len(best):  # ends scanned in increasing order: ties keep the smaller end
            best = nodes
    bonus = tgt[best[-1] + 1] if best else tgt[0]
    return best, bonus


@pytest.mark.parametrize("seed", range(40))
def test_greedy_accept_brute_force(seed):
    rng = np.random.default_rng(seed)
    B, T = 3, int(rng.integers(1, 13))
    parent = np.stack([W.random_parents(T, rng) for _ in range(B)]).astype(np.int32)
    vocab = int(rng.integers(2, 5))  # small vocabulary: many matches, ties between siblings
    draft = rng.integers(0, vocab, size=(B, T)).astype(np.int32)
    tgt = rng.integers(0, vocab, size=(B, T + 1)).astype(np.int32)
    path, n, bonus = oracle.greedy_accept(parent, draft, tgt)
    for b in range(B):
        want, wb = _accept_brute_force(parent[b].tolist(), draft[b].tolist(), tgt[b].tolist())
        assert n[b] == len(want) and path[b, : n[b]].tolist() == want
        assert np.all(path[b, n[b]:] == -1)
        assert bonus[b] == wb


def test_greedy_accept_chain_is_prefix_match():
    """On a chain the committed length is the first position where draft and
    target disagree (the usual greedy speculative decoding rule)."""
    rng = np.random.default_rng(5)
    T = 9
    parent = np.array([W.chain_parents(T)] * 4, np.int32)
    tgt = rng.integers(0, 100, size=(4, T + 1)).astype(np.int32)
    draft = tgt[:, :T].copy()
    for b, m in enumerate([0, 3, 8, T]):  # first mismatch at m (T: none)
        if m < T:
            draft[b, m] += 1
    path, n, bonus = oracle.greedy_accept(parent, draft, tgt)
    assert n.tolist() == [0, 3, 8, T]
    for b, m in enumerate([0, 3, 8, T]):
        assert path[b, :m].tolist() == list(range(m))
        assert bonus[b] == tgt[b, m]


def test_commit_kv_hand():
    with open(os.path.join(GOLD, "commit_kv_hand.json")) as f:
        g = json.load(f)
    rows = np.array(g["rows_before"], np.float32)[None, :, None, :]  # [B=1][slots][Hkv=1][D=2]
    k, v, L = oracle.commit_kv_dense(rows, rows + 100, np.array([g["seqlen"]], np.int32),
                                     np.array([g["path"]], np.int32), np.array([g["n_accept"]], np.int32))
    assert k[0, :, 0].tolist() == g["rows_after"]
    assert (v - 100)[0, :, 0].tolist() == g["rows_after"]
    assert L.tolist() == [g["seqlen_after"]]


def test_commit_kv_paged_equals_dense():
    """Committing through a page table and re-reading the sequence equals
    committing the contiguous copy of the same sequence (HiSpec 2: paged =
    contiguous)."""
    rng = np.random.default_rng(11)
    B, Hkv, D, T, ps = 3, 2, 4, 6, 4
    L = np.array([5, 0, 9], np.int32)
    need = (L + T + ps - 1) // ps
    P = int(need.sum()) + 2
    perm = rng.permutation(P)
    table = np.full((B, int(need.max())), -1, np.int32)
    off = 0
    for b in range(B):
        table[b, : need[b]] = perm[off: off + need[b]]
        off += need[b]
    kp = rng.standard_normal((P, ps, Hkv, D)).astype(np.float32)
    vp = rng.standard_normal((P, ps, Hkv, D)).astype(np.float32)
    parent = np.stack([W.random_parents(T, rng) for _ in range(B)]).astype(np.int32)
    tgt = rng.integers(0, 2, size=(B, T + 1)).astype(np.int32)
    draft = rng.integers(0, 2, size=(B, T)).astype(np.int32)
    path, n, _ = oracle.greedy_accept(parent, draft, tgt)
    k2, v2, L2 = oracle.commit_kv_paged(kp, vp, table, ps, L, path, n)
    for b in range(B):
        cap = int(L[b]) + T
        kd = oracle.gather_pages(kp, table[b], cap, ps)[None]
        vd = oracle.gather_pages(vp, table[b], cap, ps)[None]
        kc, vc, Lc = oracle.commit_kv_dense(kd, vd, L[b:b + 1], path[b:b + 1], n[b:b + 1])
        assert np.array_equal(oracle.gather_pages(k2, table[b], cap, ps), kc[0])
        assert np.array_equal(oracle.gather_pages(v2, table[b], cap, ps), vc[0])
        assert L2[b] == Lc[0] == L[b] + n[b]


def test_commit_kv_identity_and_untouched_rows():
    rng = np.random.default_rng(3)
    k = rng.standard_normal((2, 20, 3, 4)).astype(np.float32)
    L = np.array([7, 10], np.int32)
    ident = np.array([[0, 1, 2, -1], [0, 1, -1, -1]], np.int32)
    k2, _, L2 = oracle.commit_kv_dense(k, k, L, ident, np.array([3, 2], np.int32))
    assert np.array_equal(k2, k) and L2.tolist() == [10, 12]
    moved = np.array([[2, 3, -1, -1], [1, -1, -1, -1]], np.int32)
    k3, _, _ = oracle.commit_kv_dense(k, k, L, moved, np.array([2, 1], np.int32))
    assert np.array_equal(k3[0, 7], k[0, 9]) and np.array_equal(k3[0, 8], k[0, 10])
    assert np.array_equal(k3[1, 10], k[1, 11])
    changed = np.zeros(k.shape[:2], bool)
    changed[0, 7:9] = True
    changed[1, 10] = True
    assert np.array_equal(k3[~changed], k[~changed])


# ----------------------------------------------------------------------------
# importance map of a few query heads (the scoring pass that feeds the verify set)
# ----------------------------------------------------------------------------

def test_head_importance_hand():
    with open(os.path.join(GOLD, "head_importance_hand.json")) as f:
        g = json.load(f)
    q = np.array(g["q"], np.float64)[None]
    k = np.array(g["k"], np.float64)[None]
    for case in g["cases"]:
        imp = oracle.head_importance(q, k, np.array(g["seqlens"], np.int32), case["heads"], g["scale"])
        assert np.allclose(imp[0], case["importance"], rtol=0.0, atol=1e-12), case["heads"]


def _importance_case(seed, B=3, T=4, Hq=8, Hkv=2, D=16, Lmax=40):
    rng = np.random.default_rng(seed)
    q = W.bf16_bits(torch.from_numpy(rng.standard_normal((B, T, Hq, D)).astype(np.float32)).to(torch.bfloat16))
    k = W.bf16_bits(torch.from_numpy(rng.standard_normal((B, Lmax, Hkv, D)).astype(np.float32)).to(torch.bfloat16))
    L = rng.integers(1, Lmax - T + 1, size=B).astype(np.int32)
    L[0] = Lmax - T
    return q, k, L


@pytest.mark.parametrize("seed", range(4))
def test_head_importance_matches_torch_softmax(seed):
    """Against torch's softmax in float64 over einsum scores (library routines)."""
    q, k, L = _importance_case(seed)
    heads = [1, 6, 6, 3]
    scale = 0.3
    imp = oracle.head_importance(q, k, L, heads, scale)
    qt, kt = torch.from_numpy(_f64(q)), torch.from_numpy(_f64(k))
    group = q.shape[2] // k.shape[2]
    for b in range(len(L)):
        want = torch.zeros(k.shape[1], dtype=torch.float64)
        for h in heads:
            s = torch.einsum("td,ld->tl", qt[b, :, h], kt[b, : L[b], h // group]) * scale
            want[: L[b]] += torch.softmax(s, dim=-1).sum(dim=0)
        assert np.allclose(imp[b], want.numpy(), rtol=0.0, atol=1e-12)


def test_head_importance_single_head_and_token_is_scipy_softmax():
    scipy_special = pytest.importorskip("scipy.special")
    q, k, L = _importance_case(7, T=1)
    for h in range(q.shape[2]):
        imp = oracle.head_importance(q, k, L, [h], 0.25)
        for b in range(len(L)):
            kv = h // (q.shape[2] // k.shape[2])
            want = scipy_special.softmax(0.25 * (_f64(k[b, : L[b], kv]) @ _f64(q[b, 0, h])))
            assert np.allclose(imp[b, : L[b]], want, rtol=0.0, atol=1e-13)
            assert np.all(imp[b, L[b]:] == 0.0)


def test_head_importance_mass_and_equal_keys():
    """Each (head, token) distribution sums to one over the L committed keys;
    with all keys of a kv-head equal it is uniform, 1/L per key."""
    q, k, L = _importance_case(3)
    heads = [0, 5, 7]
    T = q.shape[1]
    imp = oracle.head_importance(q, k, L, heads, 0.4)
    for b in range(len(L)):
        assert abs(imp[b].sum() - len(heads) * T) < 1e-11
        assert np.all(imp[b, L[b]:] == 0.0)
    flat = k.copy()
    flat[:, :, :, :] = k[:, :1, :, :]  # every row equals row 0
    imp = oracle.head_importance(q, flat, L, heads, 0.4)
    for b in range(len(L)):
        assert np.allclose(imp[b, : L[b]], len(heads) * T / L[b], rtol=1e-13, atol=0.0)


def test_head_importance_follows_the_prefix_rows_only():
    """Permuting the committed rows permutes the importances; the rows after
    the prefix (draft slots) do not enter."""
    q, k, L = _importance_case(5)
    heads = [2, 4]
    imp = oracle.head_importance(q, k, L, heads, 0.5)
    rng = np.random.default_rng(9)
    k2 = k.copy()
    perms = []
    for b in range(len(L)):
        p = rng.permutation(int(L[b]))
        perms.append(p)
        k2[b, : L[b]] = k[b, p]
        k2[b, L[b]:] = k[b, L[b]:] ^ np.uint16(0x1234)  # draft and spare rows changed
    imp2 = oracle.head_importance(q, k2, L, heads, 0.5)
    for b in range(len(L)):
        assert np.allclose(imp2[b, : L[b]], imp[b, perms[b]], rtol=0.0, atol=1e-12)
        assert np.all(imp2[b, L[b]:] == 0.0)


# ----------------------------------------------------------------------------
# rotary position embedding of the draft block
# ----------------------------------------------------------------------------

def test_rope_hand():
    with open(os.path.join(GOLD, "rope_hand.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        out = oracle.rope_rotate(np.array(case["x"], np.float64), case["pos"], g["base"])
        assert np.allclose(out, case["out"], rtol=0.0, atol=1e-15), case


@pytest.mark.parametrize("seed", range(3))
def test_rope_matches_complex_rotation(seed):
    """Each pair (x_i, x_{i+D/2}) is the complex number x_i + i x_{i+D/2}
    multiplied by exp(i pos theta_i), theta_i = base^(-2i/D) (numpy complex)."""
    rng = np.random.default_rng(seed)
    D, base = 128, 500000.0
    x = rng.standard_normal((6, D))
    pos = rng.integers(0, 140000, size=6)
    z = (x[:, : D // 2] + 1j * x[:, D // 2:]) * np.exp(1j * pos[:, None] * base ** (-np.arange(0, D, 2) / D))
    want = np.concatenate([z.real, z.imag], axis=1)
    assert np.allclose(oracle.rope_rotate(x, pos, base), want, rtol=0.0, atol=1e-9)


def test_rope_invariants():
    """Rotations keep each pair's length, compose by adding positions, and make
    q.k depend on the positions only through their difference."""
    rng = np.random.default_rng(4)
    D, base = 64, 10000.0
    q, k = rng.standard_normal((2, D))
    r = oracle.rope_rotate(q, 37, base)
    h = D // 2
    assert np.allclose(r[:h] ** 2 + r[h:] ** 2, q[:h] ** 2 + q[h:] ** 2, rtol=1e-12)
    assert np.allclose(oracle.rope_rotate(r, 1000, base), oracle.rope_rotate(q, 1037, base), atol=1e-10)
    d1 = oracle.rope_rotate(q, 500, base) @ oracle.rope_rotate(k, 480, base)
    d2 = oracle.rope_rotate(q, 9020, base) @ oracle.rope_rotate(k, 9000, base)
    assert abs(d1 - d2) < 1e-9
    assert np.array_equal(oracle.rope_rotate(q, 0, base), q)


def test_rope_draft_rows_only():
    """Only the T draft rows after each prefix are rotated, each at its token's
    position (a tree's positions: L_b + depth), and a paged cache gives the
    same rows as the contiguous one."""
    rng = np.random.default_rng(6)
    B, T, Hq, Hkv, D, ps = 3, 5, 4, 2, 8, 4
    L = np.array([6, 0, 11], np.int32)
    cap = int(L.max()) + T + 2
    q = rng.standard_normal((B, T, Hq, D)).astype(np.float32)
    k = rng.standard_normal((B, cap, Hkv, D)).astype(np.float32)
    parent = np.stack([W.random_parents(T, rng) for _ in range(B)])
    pos = L[:, None] + np.stack([W.chain_depths(p) for p in parent])
    qr, kr = oracle.rope_draft_dense(q, k, L, pos, 10000.0)
    for b in range(B):
        for t in range(T):
            assert np.allclose(qr[b, t], oracle.rope_rotate(q[b, t], pos[b, t], 10000.0), atol=0)
            assert np.allclose(kr[b, L[b] + t], oracle.rope_rotate(k[b, L[b] + t], pos[b, t], 10000.0), atol=0)
        keep = np.ones(cap, bool)
        keep[L[b]:L[b] + T] = False
        assert np.array_equal(kr[b, keep], k[b, keep].astype(np.float64))
    # paged: the same sequences behind a shuffled page table
    need = (L + T + ps - 1) // ps
    P = int(need.sum()) + 1
    perm = rng.permutation(P)
    table = np.full((B, int(need.max())), -1, np.int32)
    pages = rng.standard_normal((P, ps, Hkv, D)).astype(np.float32)
    off = 0
    for b in range(B):
        table[b, : need[b]] = perm[off: off + need[b]]
        off += need[b]
    qp, kp = oracle.rope_draft_paged(q, pages, table, ps, L, pos, 10000.0)
    assert np.array_equal(qp, qr)
    for b in range(B):
        n = int(L[b]) + T
        dense = oracle.gather_pages(pages, table[b], n, ps)[None]
        _, kd = oracle.rope_draft_dense(q[b:b + 1], dense, L[b:b + 1], pos[b:b + 1], 10000.0)
        assert np.array_equal(oracle.gather_pages(kp, table[b], n, ps), kd[0])
