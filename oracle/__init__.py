"""fp64 CPU oracle for speculative-decoding verification attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The CUDA library never imports,
links or calls it, and it shares no code with the CUDA sources.

The attention, the log-sum-exp merge and the tree visibility are evaluated by
``verify_oracle.c`` (plain C, fp64, OpenMP over rows).  This module builds that
file with gcc, widens nothing itself, and assembles for each sequence the
explicit key list and the explicit full visibility matrix the C code consumes:

* dense   (LongSpec 2.C "Hybrid Tree Attention"): keys are cache rows
  0 .. L_b+T-1; prefix rows are visible to every draft token (the cache part
  carries no mask), draft rows L_b+j are visible per the draft bitmask.
* paged   (HiSpec 2, "batched inference" with paged attention and block
  tables): the page table is resolved into a separate contiguous copy of the
  sequence first, then treated as dense.
* sparse  (Dustin 1 and 3, verification over a fixed-size set I_verify): the
  prefix keys are the cache rows listed in the verify set of that kv-head,
  followed by the draft rows.

The verify-set selection (Dustin 1, "hybrid attention aggregation") is here
too, written as a full stable sort of candidates by (score descending, index
ascending), and so is the importance map of a few query heads that feeds it
(Dustin 1 and 2), written with numpy in fp64.

Readings where the pages are silent are documented with each function.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "verify_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, F32, F64 = 0, 2, 3


def build(force: bool = False) -> str:
    """Compile verify_oracle.c into a shared library (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_masked_attention.restype = ctypes.c_int
            lib.oracle_masked_attention.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_longlong,
                ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_lse_merge.restype = None
            lib.oracle_lse_merge.argtypes = [ctypes.c_int, ctypes.c_longlong, ctypes.c_int,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_tree_visibility.restype = ctypes.c_int
            lib.oracle_tree_visibility.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


@contextlib.contextmanager
def swapped_library(path: str):
    """Test hook: run every wrapper below against another build of verify_oracle.c
    (the mutation tests compile deliberately broken copies to show the pins catch them)."""
    global _lib
    _load()
    saved = _lib
    try:
        with _lock:
            _lib = None
        lib = ctypes.CDLL(path)
        for name in ("oracle_masked_attention", "oracle_lse_merge", "oracle_tree_visibility",
                     "oracle_num_threads", "oracle_set_num_threads"):
            f, g = getattr(lib, name), getattr(saved, name)
            f.restype, f.argtypes = g.restype, g.argtypes
        _lib = lib
        yield
    finally:
        _lib = saved


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def _code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16  # raw bfloat16 bit patterns
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"unsupported array dtype {a.dtype}")


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ----------------------------------------------------------------------------
# primitives (C)
# ----------------------------------------------------------------------------

def masked_attention(q, k, v, visible, scale):
    """Masked softmax attention of one sequence over an explicit key list.

    q [T][Hq][D]; k, v [n][Hkv][D]; visible bool [T][n].  Arrays are float64,
    float32 or uint16 (bf16 bits).  Returns out f64 [T][Hq][D], lse f64 [Hq][T].
    """
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    T, Hq, D = q.shape
    n, Hkv, Dk = k.shape
    assert Dk == D and v.shape == k.shape and k.dtype == v.dtype
    vis = np.ascontiguousarray(visible, dtype=np.uint8)
    assert vis.shape == (T, n)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    lse = np.zeros((Hq, T), dtype=np.float64)
    rc = _load().oracle_masked_attention(T, Hq, Hkv, D, float(scale), n, _ptr(q), _code(q), _ptr(k), _ptr(v),
                                         _code(k), _ptr(vis), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_masked_attention rejected its arguments")
    return out, lse


def lse_merge(o_parts, lse_parts):
    """Exact log-sum-exp merge of partial attentions (LongSpec 2.C, LSE fusion).

    o_parts f64 [S][R][D], lse_parts f64 [S][R] -> out f64 [R][D], lse f64 [R].
    """
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    S, R, D = o_parts.shape
    out = np.zeros((R, D), dtype=np.float64)
    lse = np.zeros(R, dtype=np.float64)
    _load().oracle_lse_merge(S, R, D, _ptr(o_parts), _ptr(lse_parts), _ptr(out), _ptr(lse))
    return out, lse


def tree_visibility(parent):
    """Ancestor-or-self visibility bool [T][T] of a parent-pointer tree (LongSpec 1.3, 2.C)."""
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    T = parent.shape[0]
    vis = np.zeros((T, T), dtype=np.uint8)
    if _load().oracle_tree_visibility(T, _ptr(parent), _ptr(vis)) != 0:
        raise ValueError("parent array is not a topologically ordered forest")
    return vis.astype(bool)


# ----------------------------------------------------------------------------
# bitmask words <-> boolean rows (the draft-mask layout of the library's ABI)
# ----------------------------------------------------------------------------

def words_to_bool(words, T):
    """uint32 words [..., W] -> bool [..., T]; bit j % 32 of word j // 32 is token j."""
    words = np.asarray(words, dtype=np.uint32)
    out = np.zeros(words.shape[:-1] + (T,), dtype=bool)
    for j in range(T):
        out[..., j] = (words[..., j // 32] >> np.uint32(j % 32)) & np.uint32(1) == 1
    return out


def bool_to_words(rows):
    rows = np.asarray(rows, dtype=bool)
    T = rows.shape[-1]
    W = (T + 31) // 32
    out = np.zeros(rows.shape[:-1] + (W,), dtype=np.uint32)
    for j in range(T):
        out[..., j // 32] |= rows[..., j].astype(np.uint32) << np.uint32(j % 32)
    return out


def tree_mask_words(parent):
    """Per-sequence ancestor bitmask words uint32 [B][T][ceil(T/32)] from parent int32 [B][T]."""
    parent = np.asarray(parent, dtype=np.int32)
    return np.stack([bool_to_words(tree_visibility(p)) for p in parent])


# ----------------------------------------------------------------------------
# verification attention per layout
# ----------------------------------------------------------------------------

def _draft_visibility(draft_vis_b, n_prefix_cols, T):
    """Explicit [T][n_prefix + T] matrix: prefix columns all visible, draft columns per mask."""
    vis = np.zeros((T, n_prefix_cols + T), dtype=bool)
    vis[:, :n_prefix_cols] = True
    vis[:, n_prefix_cols:] = draft_vis_b
    return vis


def attention_dense(q, k_cache, v_cache, seqlens, draft_vis, scale):
    """Dense layout.  q [B][T][Hq][D]; caches [B][Lmax][Hkv][D] with the draft
    keys already at slots L_b .. L_b+T-1; draft_vis bool [B][T][T].
    Returns out f64 [B][T][Hq][D], lse f64 [B][Hq][T]."""
    B, T, Hq, D = q.shape
    out = np.zeros((B, T, Hq, D))
    lse = np.zeros((B, Hq, T))
    for b in range(B):
        L = int(seqlens[b])
        vis = _draft_visibility(draft_vis[b], L, T)
        out[b], lse[b] = masked_attention(q[b], k_cache[b, : L + T], v_cache[b, : L + T], vis, scale)
    return out, lse


def gather_pages(pages, page_table_b, n_tokens, page_size):
    """Contiguous copy [n_tokens][Hkv][D] of one sequence held in pages [P][page][Hkv][D]."""
    pos = np.arange(n_tokens)
    page = np.asarray(page_table_b)[pos // page_size]
    if np.any(page < 0) or np.any(page >= pages.shape[0]):
        raise ValueError("page table entry out of range")
    return pages[page, pos % page_size]


def attention_paged(q, k_pages, v_pages, page_table, page_size, seqlens, draft_vis, scale):
    """Paged layout: resolve each sequence's pages into a separate contiguous copy, then dense."""
    B, T, Hq, D = q.shape
    out = np.zeros((B, T, Hq, D))
    lse = np.zeros((B, Hq, T))
    for b in range(B):
        L = int(seqlens[b])
        k = gather_pages(k_pages, page_table[b], L + T, page_size)
        v = gather_pages(v_pages, page_table[b], L + T, page_size)
        vis = _draft_visibility(draft_vis[b], L, T)
        out[b], lse[b] = masked_attention(q[b], k, v, vis, scale)
    return out, lse


def attention_sparse(q, k_cache, v_cache, seqlens, indices, n_indices, draft_vis, scale):
    """Sparse layout: per (b, kv-head) the prefix keys are rows indices[b][h][:n] of
    the full cache (no compaction of the cache itself), then the T draft rows."""
    B, T, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    g = Hq // Hkv
    out = np.zeros((B, T, Hq, D))
    lse = np.zeros((B, Hq, T))
    for b in range(B):
        L = int(seqlens[b])
        for h in range(Hkv):
            n = int(n_indices[b][h])
            idx = np.asarray(indices[b][h][:n], dtype=np.int64)
            if np.any(idx < 0) or np.any(idx >= L):
                raise ValueError("verify index out of range")
            rows = np.concatenate([idx, np.arange(L, L + T)])
            k = k_cache[b][rows][:, h: h + 1]
            v = v_cache[b][rows][:, h: h + 1]
            vis = _draft_visibility(draft_vis[b], n, T)
            o, l = masked_attention(q[b][:, h * g:(h + 1) * g], k, v, vis, scale)
            out[b][:, h * g:(h + 1) * g] = o
            lse[b][h * g:(h + 1) * g] = l
    return out, lse


# ----------------------------------------------------------------------------
# verify index set (Dustin section 1)
# ----------------------------------------------------------------------------

def _top_by_score(cand, score, count):
    """The ``count`` candidates with the largest score; equal scores go to the lower index."""
    if count <= 0 or len(cand) == 0:
        return cand[:0]
    order = np.lexsort((cand, -score[cand]))  # primary key: score descending; then index ascending
    return cand[order[:count]]


def build_verify_index(score_draft, score_target, seqlens, n_sink, window, m_draft, budget):
    """Fixed-size verify set per (sequence, kv-head).

    I = sinks {0..n_sink-1}  U  recent window {L-window .. L-1}
        U  top-m_draft of score_draft among the other positions
        U  top of score_target among those still unchosen, filling up to budget,
    clipped to [0, L) and sorted ascending; |I| = min(budget, L).
    score_* fp32 [B][Hkv][>=L]; returns idx int32 [B][Hkv][budget] (tail -1), n int32 [B][Hkv].
    Requires budget >= n_sink + window; scores must not be NaN.
    """
    if budget < n_sink + window:
        raise ValueError("budget smaller than sinks + window")
    B, Hkv = score_draft.shape[:2]
    idx = np.full((B, Hkv, budget), -1, dtype=np.int32)
    cnt = np.zeros((B, Hkv), dtype=np.int32)
    for b in range(B):
        L = int(seqlens[b])
        fixed = np.zeros(L, dtype=bool)
        fixed[: min(n_sink, L)] = True
        fixed[max(0, L - window):] = True
        cand = np.nonzero(~fixed)[0]
        room = budget - int(fixed.sum())
        for h in range(Hkv):
            sd = np.asarray(score_draft[b, h, :L], dtype=np.float32)
            st = np.asarray(score_target[b, h, :L], dtype=np.float32)
            pick_d = _top_by_score(cand, sd, min(m_draft, room))
            rest = np.setdiff1d(cand, pick_d, assume_unique=True)
            pick_t = _top_by_score(rest, st, room - len(pick_d))
            sel = np.concatenate([np.nonzero(fixed)[0], pick_d, pick_t])
            sel = np.sort(sel)
            cnt[b, h] = len(sel)
            idx[b, h, : len(sel)] = sel
    return idx, cnt


# ----------------------------------------------------------------------------
# after verification: greedy acceptance over the tree, and the KV commit
# (Dustin section 1, step 5: accepted tokens join the cache, rejected ones are
# dropped; HiSpec section 2: the entries of rejected tokens are removed before
# the next phase, and the output equals the target model's own decoding)
# ----------------------------------------------------------------------------

def greedy_accept(parent, draft_tokens, target_next):
    """Greedy acceptance over token trees.

    Reading (the pages fix the guarantee, not the tree rule): a draft node is
    accepted when its parent is accepted -- or it hangs off the committed
    prefix (parent -1) -- and its token equals the target model's greedy
    token after that parent.  The committed path is the accepted root path of
    greatest depth, the one ending at the smallest node index when several
    are equally deep; the bonus token is the target's greedy token after the
    path's last node (after the prefix when nothing is accepted).

    parent [B][T] int32 with -1 <= parent[t] < t; draft_tokens [B][T] int32;
    target_next [B][T+1] int32: column 0 is the target's greedy next token
    after the committed prefix, column t+1 the one after draft node t.
    Returns path [B][T] int32 (node indices from the root down, tail -1),
    n_accept [B] int32 and bonus [B] int32.
    """
    parent = np.asarray(parent)
    draft = np.asarray(draft_tokens)
    tgt = np.asarray(target_next)
    B, T = parent.shape
    path = np.full((B, T), -1, dtype=np.int32)
    n_acc = np.zeros(B, dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int32)
    for b in range(B):
        accepted = [False] * T
        depth = [0] * T
        for t in range(T):  # a parent comes before its children
            p = int(parent[b, t])
            if not -1 <= p < t:
                raise ValueError("parent[%d][%d] = %d is not an earlier node" % (b, t, p))
            up = p < 0 or accepted[p]
            accepted[t] = up and int(draft[b, t]) == int(tgt[b, p + 1])
            depth[t] = 1 if p < 0 else depth[p] + 1
        best = -1
        for t in range(T):
            if accepted[t] and (best < 0 or depth[t] > depth[best]):
                best = t
        if best < 0:
            bonus[b] = tgt[b, 0]
            continue
        nodes = []
        t = best
        while t >= 0:
            nodes.append(t)
            t = int(parent[b, t])
        nodes.reverse()
        path[b, : len(nodes)] = nodes
        n_acc[b] = len(nodes)
        bonus[b] = tgt[b, best + 1]
    return path, n_acc, bonus


def commit_kv_dense(k_cache, v_cache, seqlens, path, n_accept):
    """KV commit after acceptance, contiguous cache [B][len][Hkv][D].

    The draft rows of sequence b sit at slots L_b .. L_b+T-1 (L_b =
    seqlens[b]).  For j < n_accept[b] the row at slot L_b + path[b][j] is
    moved to slot L_b + j, in every kv-head of both caches; every other slot
    keeps its content.  Rows are copied, not computed (any element type).
    Returns new k, v and seqlens + n_accept.
    """
    k = np.array(k_cache, copy=True)
    v = np.array(v_cache, copy=True)
    for b in range(len(seqlens)):
        L = int(seqlens[b])
        a = int(n_accept[b])
        src = [L + int(path[b][j]) for j in range(a)]
        k[b, L:L + a] = np.asarray(k_cache)[b, src]
        v[b, L:L + a] = np.asarray(v_cache)[b, src]
    return k, v, (np.asarray(seqlens) + np.asarray(n_accept)).astype(np.int32)


def commit_kv_paged(k_pages, v_pages, page_table, page_size, seqlens, path, n_accept):
    """The same commit over a paged pool [P][page][Hkv][D]: logical slot s of
    sequence b is row s % page_size of page page_table[b][s // page_size]."""
    k = np.array(k_pages, copy=True)
    v = np.array(v_pages, copy=True)

    def where(b, slot):
        return int(page_table[b][slot // page_size]), slot % page_size

    for b in range(len(seqlens)):
        L = int(seqlens[b])
        for j in range(int(n_accept[b])):
            sp, sr = where(b, L + int(path[b][j]))
            dp, dr = where(b, L + j)
            k[dp, dr] = np.asarray(k_pages)[sp, sr]
            v[dp, dr] = np.asarray(v_pages)[sp, sr]
    return k, v, (np.asarray(seqlens) + np.asarray(n_accept)).astype(np.int32)


# ----------------------------------------------------------------------------
# importance of the cached positions from a few query heads (Dustin section 1:
# the target model's attention scores are one of the two signals of the global
# importance map; section 2: that estimate is computed on a few semantic
# retrieval heads only, instead of every head of every layer)
# ----------------------------------------------------------------------------

def _widen(a):
    """bf16 bit patterns / fp32 / fp64 -> float64, exactly."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def head_importance(q, k_cache, seqlens, heads, scale):
    """Global importance map of the cached prefix from the listed query heads.

    Reading (the pages name the signal -- attention scores of a few heads --
    but not how they are pooled): for sequence b with L = seqlens[b], each
    listed head h and each query token t < T, the attention distribution over
    the L committed keys,
        p[h, t][j] = exp(scale q[b,t,h] . k[b,j,h // group])
                     / sum_{j' < L} exp(scale q[b,t,h] . k[b,j',h // group]),
    and the importance of position j is the sum of p[h, t][j] over the listed
    heads and the T tokens (a head listed twice counts twice).  Only the L
    committed keys are scored: the draft rows after them are no candidates of
    the verify set.

    q [B][T][Hq][D], k_cache [B][Lmax][Hkv][D] (bf16 bits, fp32 or fp64).
    Returns f64 [B][Lmax], zero at j >= L.
    """
    B, T, Hq, D = q.shape
    Lmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    group = Hq // Hkv
    imp = np.zeros((B, Lmax))
    for b in range(B):
        L = int(seqlens[b])
        if L == 0:
            continue
        for h in heads:
            qh = _widen(q[b, :, h])                 # [T][D]
            kh = _widen(k_cache[b, :L, h // group])  # [L][D]
            z = scale * (qh @ kh.T)                 # [T][L]
            z = z - z.max(axis=1, keepdims=True)
            e = np.exp(z)
            imp[b, :L] += (e / e.sum(axis=1, keepdims=True)).sum(axis=0)
    return imp


# ----------------------------------------------------------------------------
# rotary position embedding of the draft block (LongSpec section 1: the target
# model keeps its own RoPE base; position ids may be arbitrary, e.g. the
# anchor-offset indices 0, 1, 2, 3, 8192, 8193, ...)
# ----------------------------------------------------------------------------

def rope_rotate(x, positions, base):
    """Rotary embedding of vectors x [..., D] at integer positions [...].

    Reading (the pages name RoPE and its base, not the layout): the
    rotate-half layout, pairing element i with element i + D/2 for
    i < D/2, at the angle pos * base^(-2i/D):
        out[i]       = x[i] cos(a_i) - x[i + D/2] sin(a_i)
        out[i + D/2] = x[i + D/2] cos(a_i) + x[i] sin(a_i).
    x: bf16 bits / fp32 / fp64; returns f64.
    """
    x = _widen(x)
    D = x.shape[-1]
    half = D // 2
    inv_freq = float(base) ** (-(2.0 * np.arange(half)) / D)
    ang = np.asarray(positions, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def rope_draft_dense(q, k_cache, seqlens, positions, base):
    """q [B][T][Hq][D] rotated at positions[b][t] (every head), and the draft
    key rows of a dense cache [B][Lmax][Hkv][D] -- slots L_b + t for t < T --
    rotated at the same positions; the other cache rows are returned as they
    are (widened).  Returns (q f64, k f64)."""
    pos = np.asarray(positions)
    qr = rope_rotate(q, pos[:, :, None], base)
    k = _widen(k_cache).copy()
    T = pos.shape[1]
    for b in range(len(seqlens)):
        L = int(seqlens[b])
        k[b, L:L + T] = rope_rotate(k_cache[b, L:L + T], pos[b][:, None], base)
    return qr, k


def rope_draft_paged(q, k_pages, page_table, page_size, seqlens, positions, base):
    """The same through a page table: the draft row of token t of sequence b
    is row (L_b + t) % page_size of page page_table[b][(L_b + t) // page_size]."""
    pos = np.asarray(positions)
    qr = rope_rotate(q, pos[:, :, None], base)
    k = _widen(k_pages).copy()
    for b in range(len(seqlens)):
        L = int(seqlens[b])
        for t in range(pos.shape[1]):
            slot = L + t
            pg, row = int(page_table[b][slot // page_size]), slot % page_size
            k[pg, row] = rope_rotate(k_pages[pg, row], pos[b, t], base)
    return qr, k


# ----------------------------------------------------------------------------
# whole verification step for a workload object (duck-typed)
# ----------------------------------------------------------------------------

def _host_array(t):
    """numpy view of a CPU tensor: bf16 -> uint16 bits, fp32 -> float32 (no arithmetic)."""
    import torch  # local: only for reading tensors handed in by the tests

    if isinstance(t, np.ndarray):
        return t
    t = t.detach().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.float64:
        return t.numpy()
    raise TypeError(t.dtype)


def draft_visibility(w):
    """bool [B][T][T]: ancestor-or-self from parents when the workload has a tree,
    else its explicit bitmask words."""
    if w.parent is not None:
        return np.stack([tree_visibility(p) for p in w.parent])
    return words_to_bool(w.mask_words, w.T)


def verify(w, indices=None, n_indices=None):
    """Reference output of one verification step for workload ``w``.

    Returns dict(out f64 [B][T][Hq][D], lse f64 [B][Hq][T], mask_words, and for
    the sparse layout indices/n_indices).
    """
    vis = draft_visibility(w)
    q = _host_array(w.q)
    res = {"mask_words": bool_to_words(vis)}
    if w.layout == "dense":
        res["out"], res["lse"] = attention_dense(q, _host_array(w.k_cache), _host_array(w.v_cache),
                                                 w.seqlens, vis, w.scale)
    elif w.layout == "paged":
        res["out"], res["lse"] = attention_paged(q, _host_array(w.k_pages), _host_array(w.v_pages),
                                                 w.page_table, w.page_size, w.seqlens, vis, w.scale)
    elif w.layout == "sparse":
        if indices is None:
            indices, n_indices = build_verify_index(w.score_draft, w.score_target, w.seqlens, w.n_sink,
                                                    w.window, w.m_draft, w.budget)
        res["indices"], res["n_indices"] = indices, n_indices
        res["out"], res["lse"] = attention_sparse(q, _host_array(w.k_cache), _host_array(w.v_cache),
                                                  w.seqlens, indices, n_indices, vis, w.scale)
    else:
        raise ValueError(w.layout)
    return res
