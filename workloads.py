"""Seeded synthetic inputs for speculative-decoding verification attention.

This module draws the inputs that both the fp64 oracle and the CUDA library
consume: query/key/value tensors, token trees (parent pointers), explicit draft
bitmasks, page tables, cache lengths and importance scores.  It contains none of
the method's arithmetic: it never turns a tree into a mask, never selects an
index set and never computes attention.  Every tensor comes from its own numpy
PCG64 stream keyed by ``(seed, tensor_id, chunk)``, so a workload is identical
bit for bit on every machine and for every thread count.

Workloads follow the shapes of the five measured configurations:

* ``tiny``   -- B1, Hq4, Hkv1, d64, fp32, prefix 512, 8-node random tree
  (parent[i] uniform in [0, i)), dense cache.
* ``chain``  -- B1, Hq32, Hkv8, d128, bf16, prefix 32768, 8-token draft chain,
  dense cache.
* ``tree``   -- B1, Hq32, Hkv8, d128, bf16, prefix 131072, 64-node token tree of
  depth 6, dense cache.
* ``sparse`` -- B16, Hq32, Hkv8, d128, bf16, prefixes uniform in
  [16384, 32768], 5-token chain, per-(sequence, kv-head) verify set of 4 sinks,
  256 recent tokens and top-scored rest (2048 in all), dense cache; query
  heads 9 and 22 (kv-heads 2 and 5) stand in for the profiled retrieval heads
  of the importance pass.
* ``paged``  -- B64, Hq32, Hkv8, d128, bf16, prefixes uniform in [2048, 8192],
  16-token pages behind a random page table, 16 draft tokens under a
  block mask (bidirectional inside 4-token blocks, causal across blocks).

Values are N(0, 1) drawn in fp32; bf16 tensors are the round-to-nearest-even
image of those fp32 draws (torch's float->bfloat16 conversion), so the oracle
widens exactly the bits the GPU reads.  Scores are U(0, 1) fp32.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
from typing import Optional

import numpy as np
import torch

# tensor ids: one independent stream per tensor kind
_ID_Q, _ID_K, _ID_V, _ID_LEN, _ID_TREE, _ID_PAGES, _ID_SD, _ID_ST, _ID_MASK = range(1, 10)
_CHUNK = 1 << 22  # elements per generator chunk (fixed, so results do not depend on threads)


def _rng(seed: int, tensor_id: int, chunk: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(tensor_id), int(chunk)])


def _fill_normal(shape, seed: int, tensor_id: int) -> np.ndarray:
    """fp32 N(0,1) array of ``shape`` drawn chunk by chunk (threaded, deterministic)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    n_chunks = (n + _CHUNK - 1) // _CHUNK

    def work(c):
        lo = c * _CHUNK
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = _rng(seed, tensor_id, c).standard_normal(hi - lo, dtype=np.float32)

    if n_chunks <= 1:
        for c in range(n_chunks):
            work(c)
    else:
        workers = max(1, min(n_chunks, os.cpu_count() or 1))
        with _cf.ThreadPoolExecutor(workers) as ex:
            list(ex.map(work, range(n_chunks)))
    return out.reshape(shape)


def _fill_uniform(shape, seed: int, tensor_id: int) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for c in range((n + _CHUNK - 1) // _CHUNK):
        lo = c * _CHUNK
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = _rng(seed, tensor_id, c).random(hi - lo, dtype=np.float32)
    return out.reshape(shape)


def _as_dtype(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(a)
    if dtype == "bf16":
        return t.to(torch.bfloat16)  # round to nearest even
    if dtype == "fp32":
        return t
    raise ValueError(f"unknown dtype {dtype!r}")


# ----------------------------------------------------------------------------
# token structures (inputs only: parent pointers and explicit bitmasks)
# ----------------------------------------------------------------------------

def chain_parents(T: int) -> np.ndarray:
    """Draft chain: token i's parent is token i-1; the root has parent -1."""
    return np.arange(-1, T - 1, dtype=np.int32)


def random_parents(T: int, rng: np.random.Generator) -> np.ndarray:
    """Random recursive tree: parent[i] uniform in [0, i) for i >= 1, root 0."""
    p = np.empty(T, dtype=np.int32)
    p[0] = -1
    for i in range(1, T):
        p[i] = rng.integers(0, i)
    return p


def depth_tree_parents(T: int, depth: int, rng: np.random.Generator):
    """Token tree of ``T`` nodes whose deepest node sits at ``depth``.

    Nodes 1..depth form a spine so the depth is reached; every other node draws
    a depth uniform in [1, depth] and a parent uniform among the nodes already
    created one level up.  Nodes are then renumbered by (depth, creation order)
    so that parent[i] < i.  Returns (parent int32[T], depth int32[T]).
    """
    if T < depth + 1:
        raise ValueError("tree too small for its depth")
    par = [-1]
    dep = [0]
    by_depth = {0: [0]}
    for k in range(1, depth + 1):
        par.append(k - 1)
        dep.append(k)
        by_depth.setdefault(k, []).append(k)
    for node in range(depth + 1, T):
        d = int(rng.integers(1, depth + 1))
        cands = by_depth[d - 1]
        par.append(int(cands[int(rng.integers(0, len(cands)))]))
        dep.append(d)
        by_depth.setdefault(d, []).append(node)
    order = sorted(range(T), key=lambda n: (dep[n], n))
    new_id = {old: new for new, old in enumerate(order)}
    parent = np.array([-1 if par[o] < 0 else new_id[par[o]] for o in order], dtype=np.int32)
    depths = np.array([dep[o] for o in order], dtype=np.int32)
    return parent, depths


def chain_depths(parent: np.ndarray) -> np.ndarray:
    """Depth of each node of a parent-pointer array (parent[i] < i)."""
    d = np.zeros(len(parent), dtype=np.int32)
    for i in range(1, len(parent)):
        d[i] = d[parent[i]] + 1 if parent[i] >= 0 else 0
    return d


def pack_bits(rows: np.ndarray) -> np.ndarray:
    """Pack a boolean [..., T] array into uint32 words [..., ceil(T/32)], bit j%32 of word j/32."""
    T = rows.shape[-1]
    W = (T + 31) // 32
    out = np.zeros(rows.shape[:-1] + (W,), dtype=np.uint32)
    for j in range(T):
        out[..., j // 32] |= (rows[..., j].astype(np.uint32) << np.uint32(j % 32))
    return out


def block_draft_mask(T: int, block: int, across: str = "causal") -> np.ndarray:
    """Boolean [T, T] visibility for masked draft blocks of ``block`` tokens.

    Inside a block every token sees every other (bidirectional).  Across blocks
    ``across='causal'`` lets block beta see all blocks <= beta; ``'isolated'``
    lets it see its own block only.
    """
    blk = np.arange(T) // block
    if across == "causal":
        return blk[None, :] <= blk[:, None]
    if across == "isolated":
        return blk[None, :] == blk[:, None]
    raise ValueError(across)


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    layout: str                 # "dense" | "paged" | "sparse"
    B: int
    T: int
    Hq: int
    Hkv: int
    D: int
    dtype: str                  # "bf16" | "fp32"
    scale: float
    seqlens: np.ndarray         # int32 [B]   committed prefix length L_b
    q: torch.Tensor             # [B][T][Hq][D]
    parent: Optional[np.ndarray] = None      # int32 [B][T] (tree/chain) or None
    mask_words: Optional[np.ndarray] = None  # uint32 [B][T][W] explicit bitmask when not a tree
    positions: Optional[np.ndarray] = None   # int32 [B][T]
    # dense and sparse layouts
    k_cache: Optional[torch.Tensor] = None   # [B][Lmax][Hkv][D]
    v_cache: Optional[torch.Tensor] = None
    max_cache_len: int = 0
    # paged layout
    k_pages: Optional[torch.Tensor] = None   # [P][page][Hkv][D]
    v_pages: Optional[torch.Tensor] = None
    page_table: Optional[np.ndarray] = None  # int32 [B][max_pages] (-1 = unused)
    page_size: int = 0
    # sparse layout: verify-set selection inputs
    score_draft: Optional[np.ndarray] = None   # fp32 [B][Hkv][Lmax]
    score_target: Optional[np.ndarray] = None  # fp32 [B][Hkv][Lmax]
    n_sink: int = 0
    window: int = 0
    m_draft: int = 0
    budget: int = 0
    score_heads: tuple = ()  # query heads of the importance pass (synthetic retrieval heads)

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one verification call must read.

        Per (sequence, kv-head): the prefix keys it attends (L_b, or the verify
        set size for the sparse layout) plus the T draft keys, times d, times 2
        (K and V), times the element size.
        """
        per_key = self.D * 2 * self.elem_bytes
        if self.layout == "sparse":
            n_prefix = self.Hkv * self.budget_effective_total()
        else:
            n_prefix = int(self.seqlens.astype(np.int64).sum()) * self.Hkv
        return (n_prefix + self.B * self.Hkv * self.T) * per_key

    def budget_effective_total(self) -> int:
        """Sum over sequences of min(budget, L_b) (per kv-head)."""
        return int(np.minimum(self.seqlens.astype(np.int64), self.budget).sum())

    def tokens(self) -> int:
        return self.B * self.T


CONFIG_NAMES = ("tiny", "chain", "tree", "sparse", "paged")


def _dense_cache(B, Lmax, Hkv, D, dtype, seed):
    k = _as_dtype(_fill_normal((B, Lmax, Hkv, D), seed, _ID_K), dtype)
    v = _as_dtype(_fill_normal((B, Lmax, Hkv, D), seed, _ID_V), dtype)
    return k, v


def make_workload(name: str, seed: int = 0, **over) -> Workload:
    """Build a named workload; keyword overrides shrink or vary it for tests.

    Overrides: B, T, Hq, Hkv, D, dtype, L (fixed prefix), L_lo/L_hi (ragged
    range), layout, tree ('random'|'depth'|'chain'|'block'|'block_isolated'|
    'random_mask'), depth, page_size, n_sink, window, budget, m_draft,
    spare_pages.
    """
    base = {
        "tiny": dict(layout="dense", B=1, T=8, Hq=4, Hkv=1, D=64, dtype="fp32", L=512, tree="random"),
        "chain": dict(layout="dense", B=1, T=8, Hq=32, Hkv=8, D=128, dtype="bf16", L=32768, tree="chain"),
        "tree": dict(layout="dense", B=1, T=64, Hq=32, Hkv=8, D=128, dtype="bf16", L=131072, tree="depth", depth=6),
        "sparse": dict(layout="sparse", B=16, T=5, Hq=32, Hkv=8, D=128, dtype="bf16", L_lo=16384, L_hi=32768,
                       tree="chain", n_sink=4, window=256, budget=2048, m_draft=894, score_heads=(9, 22)),
        "paged": dict(layout="paged", B=64, T=16, Hq=32, Hkv=8, D=128, dtype="bf16", L_lo=2048, L_hi=8192,
                      tree="block", page_size=16),
    }
    if name not in base:
        raise ValueError(f"unknown workload {name!r}")
    p = dict(base[name])
    p.update(over)
    B, T, Hq, Hkv, D, dtype = p["B"], p["T"], p["Hq"], p["Hkv"], p["D"], p["dtype"]
    layout = p["layout"]

    # cache lengths
    if "L" in p and "L_lo" not in over:
        seqlens = np.full(B, int(p["L"]), dtype=np.int32)
    else:
        lo, hi = int(p["L_lo"]), int(p["L_hi"])
        seqlens = _rng(seed, _ID_LEN).integers(lo, hi + 1, size=B).astype(np.int32)
    if "seqlens" in over:
        seqlens = np.asarray(over["seqlens"], dtype=np.int32)

    # draft structure
    trng = _rng(seed, _ID_TREE)
    tree = p["tree"]
    parent = None
    mask_words = None
    depths = None
    if tree == "chain":
        parent = np.tile(chain_parents(T), (B, 1))
        depths = np.tile(np.arange(T, dtype=np.int32), (B, 1))
    elif tree == "random":
        parent = np.stack([random_parents(T, trng) for _ in range(B)])
        depths = np.stack([chain_depths(pp) for pp in parent])
    elif tree == "depth":
        pd = [depth_tree_parents(T, int(p.get("depth", 6)), trng) for _ in range(B)]
        parent = np.stack([a for a, _ in pd])
        depths = np.stack([d for _, d in pd])
    elif tree in ("block", "block_isolated"):
        across = "causal" if tree == "block" else "isolated"
        rows = np.broadcast_to(block_draft_mask(T, int(p.get("block", 4)), across), (B, T, T))
        mask_words = pack_bits(rows)
        depths = np.tile(np.arange(T, dtype=np.int32), (B, 1))
    elif tree == "random_mask":
        mrng = _rng(seed, _ID_MASK)
        rows = mrng.random((B, T, T)) < float(p.get("density", 0.5))
        rows |= np.eye(T, dtype=bool)[None]
        mask_words = pack_bits(rows)
        depths = np.tile(np.arange(T, dtype=np.int32), (B, 1))
    else:
        raise ValueError(tree)
    positions = (seqlens[:, None] + depths).astype(np.int32)

    q = _as_dtype(_fill_normal((B, T, Hq, D), seed, _ID_Q), dtype)
    w = Workload(name=name, layout=layout, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype,
                 scale=1.0 / float(np.sqrt(D)), seqlens=seqlens, q=q, parent=parent,
                 mask_words=mask_words, positions=positions)

    if layout in ("dense", "sparse"):
        Lmax = int(seqlens.max()) + T + int(p.get("extra_slots", 0))
        w.k_cache, w.v_cache = _dense_cache(B, Lmax, Hkv, D, dtype, seed)
        w.max_cache_len = Lmax
    elif layout == "paged":
        ps = int(p["page_size"])
        need = (seqlens.astype(np.int64) + T + ps - 1) // ps
        max_pages = int(need.max())
        P = int(need.sum()) + int(p.get("spare_pages", 0))
        perm = _rng(seed, _ID_PAGES).permutation(P).astype(np.int32)
        table = np.full((B, max_pages), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            table[b, : need[b]] = perm[off: off + need[b]]
            off += int(need[b])
        w.page_table = table
        w.page_size = ps
        w.k_pages = _as_dtype(_fill_normal((P, ps, Hkv, D), seed, _ID_K), dtype)
        w.v_pages = _as_dtype(_fill_normal((P, ps, Hkv, D), seed, _ID_V), dtype)
    else:
        raise ValueError(layout)

    if layout == "sparse":
        Lmax = w.max_cache_len
        w.score_draft = _fill_uniform((B, Hkv, Lmax), seed, _ID_SD)
        w.score_target = _fill_uniform((B, Hkv, Lmax), seed, _ID_ST)
        w.n_sink = int(p["n_sink"])
        w.window = int(p["window"])
        w.budget = int(p["budget"])
        w.m_draft = int(p["m_draft"])
        w.score_heads = tuple(int(h) for h in p.get("score_heads", ()))
    return w


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw uint16 bit patterns of a bf16 tensor (no arithmetic)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
