"""GPU parity: the CUDA library against the fp64 oracle on the same seeded inputs.

Bars: bf16 (and fp32) outputs max-abs <= 2e-3, lse max-abs <= 1e-3, masks and
verify index sets bit-exact.  Small cases span several 64-key tiles with a
ragged tail; the full-size workloads are checked on every row the oracle can
afford (all of them for chain / sparse / paged, one kv-head group for tree).
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_masked_gb300 as va
import workloads as W
from tests.gpu_util import compare, dev_i32, dev_words, run_library

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    va.api.lib()


# ----------------------------------------------------------------------------
# a1: tree -> bitmask
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 5, 8, 31, 32, 33, 63, 64])
def test_tree_mask_bit_exact(T):
    rng = np.random.default_rng(T)
    parents = np.stack([W.random_parents(T, rng) for _ in range(7)])
    if T >= 8:
        parents[3] = W.depth_tree_parents(T, 6, rng)[0] if T >= 7 else parents[3]
    parents[0] = W.chain_parents(T)
    got = va.verify_tree_mask_from_parents(dev_i32(parents)).cpu().numpy().view(np.uint32)
    want = oracle.tree_mask_words(parents)
    assert np.array_equal(got, want)


def test_tree_mask_bad_parent_is_reported():
    ws = va.Workspace(256)
    parents = np.array([[-1, 0, 5, 1]], np.int32)  # parent[2] = 5 is not earlier
    va.verify_tree_mask_from_parents(dev_i32(parents), workspace=ws)
    with pytest.raises(va.VerifyAttnError) as ei:
        va.verify_attn_check_status(ws)
    assert ei.value.status == va.api.VA_ERR_DEVICE_BOUNDS
    va.verify_attn_check_status(ws)  # cleared


# ----------------------------------------------------------------------------
# a2-a4: attention, small cases
# ----------------------------------------------------------------------------

def _check(w, mode="parent", **kw):
    ref = oracle.verify(w)
    out, lse = run_library(w, mode=mode, **kw)
    torch.cuda.synchronize()
    return compare(out, lse, ref)


def test_tiny_config_full():
    w = W.make_workload("tiny")
    for mode in ("parent", "mask"):
        eo, el, _ = _check(w, mode)
        assert eo < 1e-4 and el < 1e-4  # fp32 path, no TF32


@pytest.mark.parametrize("L", [0, 1, 63, 64, 120, 125, 128, 1000, 4099])
def test_chain_small(L):
    """Prefix lengths around the 64- and 128-key tile edges: the draft block
    inside one tile, straddling two, or starting a tile of its own."""
    w = W.make_workload("chain", seed=L, L=L)
    for mode in ("parent", "causal", "mask"):
        _check(w, mode)


@pytest.mark.parametrize("case", ["chain", "paged", "shapes", "empty_row"])
def test_small_rows_on_mma_kernel(case, monkeypatch):
    """Segments of at most 64 rows with d128 run on the keys-on-lanes tcgen05
    kernel by default; VA_SMALL_ROWS_KERNEL=mma routes them to the mma.sync
    kernel, which stays held to the same bar."""
    monkeypatch.setenv("VA_SMALL_ROWS_KERNEL", "mma")
    if case == "chain":
        for L in (0, 125, 4099):
            _check(W.make_workload("chain", seed=L, L=L), "parent")
    elif case == "paged":
        _check(W.make_workload("paged", seed=21, B=4, L_lo=40, L_hi=700, page_size=16), "mask")
    elif case == "shapes":
        for Hq, Hkv, T in ((8, 8, 3), (16, 2, 8), (12, 4, 7)):
            _check(W.make_workload("tree", seed=Hq * T, Hq=Hq, Hkv=Hkv, T=T, D=128, L=517, tree="random", B=2),
                   "parent")
    else:
        w0 = W.make_workload("tree", seed=10, B=2, T=12, L=0, tree="random_mask", density=0.3)
        m = w0.mask_words.copy()
        m[0, 5, 0] = 0
        w0.mask_words = m
        out, lse = run_library(w0, "mask")
        compare(out, lse, oracle.verify(w0))


@pytest.mark.parametrize("seed", [0, 1])
def test_tree_small(seed):
    w = W.make_workload("tree", seed=seed, L=3001)
    for mode in ("parent", "mask"):
        _check(w, mode)


@pytest.mark.parametrize("Hq,Hkv,T,D", [(8, 8, 3, 128), (16, 2, 8, 128), (32, 8, 5, 64), (4, 1, 64, 64),
                                        (12, 4, 7, 128), (32, 2, 9, 128), (32, 4, 16, 128), (20, 2, 10, 128),
                                        (32, 8, 64, 128), (16, 1, 40, 128), (2, 2, 40, 128), (6, 2, 11, 128),
                                        (4, 1, 4, 128)])
def test_shapes_and_row_blocks(Hq, Hkv, T, D):
    """group*T from 3 to 640 rows: d64 on the mma.sync kernel with 1, 2, 4 row
    groups; d128 up to 64 rows on the keys-on-lanes tcgen05 kernel (16, 32 and
    64 row columns, padded), above that on the rows-on-lanes tcgen05 kernel with
    one or two 128-row M-tiles and several 256-row blocks."""
    w = W.make_workload("tree", seed=Hq * T, Hq=Hq, Hkv=Hkv, T=T, D=D, L=517, tree="random", B=2)
    _check(w, "parent")


@pytest.mark.parametrize("offset", [0, 4])
def test_whole_segments_and_output_alignment(offset):
    """192 one-tile segments: each is whole inside one CTA, which writes the final
    rows itself (bulk copies when out is 16-byte aligned, plain stores at an
    8-byte offset) with no merge."""
    w = W.make_workload("chain", seed=30 + offset, B=24, L_lo=40, L_hi=110, tree="random")
    ref = oracle.verify(w)
    q = w.q.cuda()
    flat = torch.zeros(q.numel() + offset, dtype=q.dtype, device="cuda")
    out = flat[offset:].view(q.shape)
    assert (out.data_ptr() % 16 == 0) == (offset == 0)
    o, lse = va.verify_attn_dense(q, w.k_cache.cuda(), w.v_cache.cuda(), dev_i32(w.seqlens),
                                  tree_parent=dev_i32(w.parent), out=out)
    torch.cuda.synchronize()
    compare(o, lse, ref)


def test_random_masks_and_empty_rows():
    """Arbitrary bitmasks; with L=0 a row that hides itself sees nothing (out 0, lse -inf)."""
    w = W.make_workload("tree", seed=9, B=3, T=19, L=130, tree="random_mask", density=0.3)
    _check(w, "mask")
    w0 = W.make_workload("tree", seed=10, B=2, T=12, L=0, tree="random_mask", density=0.3)
    m = w0.mask_words.copy()
    m[0, 5, 0] = 0  # row 5 of sequence 0 sees no key at all
    w0.mask_words = m
    ref = oracle.verify(w0)
    assert np.isneginf(ref["lse"][0, :, 5]).all()
    out, lse = run_library(w0, "mask")
    compare(out, lse, ref)
    assert torch.all(out[0, 5] == 0)


@pytest.mark.parametrize("page_size", [1, 4, 8, 16, 64, 128])
def test_paged_small(page_size):
    """Pages below 8 rows are gathered with cp.async; larger ones arrive as
    one TMA box per page (128-row pages as two 64-row boxes)."""
    w = W.make_workload("paged", seed=page_size, B=5, L_lo=3, L_hi=700, page_size=page_size, spare_pages=7)
    _check(w, "mask")
    wb = W.make_workload("paged", seed=page_size + 1, B=4, L_lo=40, L_hi=300, page_size=page_size,
                         tree="block_isolated")
    _check(wb, "mask")
    wt = W.make_workload("paged", seed=page_size + 2, B=3, L_lo=40, L_hi=300, page_size=page_size,
                         tree="depth", T=16, depth=4)
    _check(wt, "parent")


@pytest.mark.parametrize("page_size", [4, 8, 32])
def test_paged_fp32(page_size):
    """fp32 pages (mma.sync kernel): 128-byte boxes hold 32 values."""
    w = W.make_workload("tiny", seed=60 + page_size, layout="paged", B=3, L_lo=5, L_hi=400,
                        page_size=page_size, spare_pages=3)
    eo, el, _ = _check(w, "mask")
    assert eo < 1e-4 and el < 1e-4


def _poison_unread_rows(w):
    """NaN in every cache row no sequence reads: the tail of each sequence's
    last page, spare pages, dense rows past L + T.  Tiles that load whole
    boxes bring such rows into shared memory; they must not reach the output."""
    nan = torch.tensor(float("nan"), dtype=w.q.dtype)
    if w.layout == "paged":
        read = np.zeros(w.k_pages.shape[:2], dtype=bool)
        for b in range(w.B):
            n = int(w.seqlens[b]) + w.T
            for slot in range(n):
                read[w.page_table[b, slot // w.page_size], slot % w.page_size] = True
        m = torch.from_numpy(~read)
        w.k_pages[m] = nan
        w.v_pages[m] = nan
    else:
        for b in range(w.B):
            n = int(w.seqlens[b]) + w.T
            w.k_cache[b, n:] = nan
            w.v_cache[b, n:] = nan
    return w


@pytest.mark.parametrize("case", ["paged8", "paged16", "paged128", "dense", "dense_tree"])
def test_unread_cache_rows_poisoned(case):
    if case.startswith("paged"):
        ps = int(case[5:])
        w = W.make_workload("paged", seed=70 + ps, B=4, L_lo=30, L_hi=500, page_size=ps, spare_pages=5)
    elif case == "dense":
        w = W.make_workload("chain", seed=71, B=3, L_lo=30, L_hi=700, extra_slots=150)
    else:
        w = W.make_workload("tree", seed=72, B=2, Hkv=2, L_lo=30, L_hi=700, extra_slots=150)
    _check(_poison_unread_rows(w), "mask")


@pytest.mark.parametrize("page_size", [8, 16, 64])
@pytest.mark.parametrize("kernel", ["tcp", "tc"])
def test_many_rows_paged_tma(page_size, kernel, monkeypatch):
    """More than 128 packed rows over pages of 8 rows or more: one TMA box
    per page into the two-M-tile kernel of 128-key tiles (VA_MANY_ROWS_KERNEL=tcp)
    or the 64-key rows-on-lanes kernel."""
    monkeypatch.setenv("VA_MANY_ROWS_KERNEL", kernel)
    w = W.make_workload("paged", seed=50 + page_size, B=3, Hkv=2, Hq=8, T=40, L_lo=100, L_hi=2600,
                        page_size=page_size, tree="depth", depth=5, spare_pages=3)
    _check(_poison_unread_rows(w), "parent")


@pytest.mark.parametrize("kernel", ["tcp", "tc"])
def test_many_rows_both_kernels(kernel, monkeypatch):
    """Both kernels for more than 128 dense rows: 144 rows (one row block,
    the second M-tile partly padding), 640 rows (three row blocks), ragged
    lengths with segments whole inside one CTA and cut over many."""
    monkeypatch.setenv("VA_MANY_ROWS_KERNEL", kernel)
    _check(W.make_workload("tree", seed=61, Hq=32, Hkv=2, T=9, D=128, L=5170, tree="random", B=2), "parent")
    _check(W.make_workload("tree", seed=62, Hq=16, Hkv=1, T=40, D=128, L_lo=1, L_hi=3000, tree="random", B=3),
           "parent")
    _check(W.make_workload("tree", seed=63, B=5, Hkv=2, Hq=8, T=64, L_lo=0, L_hi=400, tree="random_mask",
                           density=0.3), "mask")


@pytest.mark.parametrize("layout", ["paged", "sparse"])
def test_many_rows_through_gathers(layout):
    """More than 64 packed rows (rows on the TMEM lanes) with K/V rows gathered
    through a page table or a verify set, ragged lengths, a token tree."""
    if layout == "paged":
        w = W.make_workload("paged", seed=41, B=3, L_lo=100, L_hi=700, page_size=16, T=32, tree="depth", depth=5)
        _check(w, "parent")
    else:
        w = W.make_workload("sparse", seed=42, B=2, L_lo=300, L_hi=900, budget=256, window=32, n_sink=4, m_draft=60,
                            T=24, tree="depth", depth=4)
        ref = oracle.verify(w)
        out, lse = run_library(w, "parent", indices=dev_i32(ref["indices"]), n_indices=dev_i32(ref["n_indices"]))
        torch.cuda.synchronize()
        compare(out, lse, ref)


def test_sparse_small_with_library_indices():
    w = W.make_workload("sparse", seed=3, B=3, L_lo=200, L_hi=900, budget=256, window=32, n_sink=4, m_draft=60)
    ref = oracle.verify(w)
    idx, cnt = va.verify_build_index(dev_i32(w.seqlens), torch.from_numpy(w.score_draft).cuda(),
                                     torch.from_numpy(w.score_target).cuda(), w.n_sink, w.window, w.m_draft,
                                     w.budget)
    assert np.array_equal(cnt.cpu().numpy(), ref["n_indices"])
    assert np.array_equal(idx.cpu().numpy(), ref["indices"])
    out, lse = run_library(w, "parent", indices=idx, n_indices=cnt)
    compare(out, lse, ref)


def test_debug_validation_of_verify_sets(monkeypatch):
    """VA_DEBUG_VALIDATE=1: a verify set with an index listed twice, or out of
    order, is reported on the device (the fast path would attend a duplicate
    twice); the sets the builder writes pass.  The bad rows are made on the host."""
    w = W.make_workload("sparse", seed=3, B=3, L_lo=200, L_hi=900, budget=256, window=32, n_sink=4, m_draft=60)
    ref = oracle.verify(w)
    monkeypatch.setenv("VA_DEBUG_VALIDATE", "1")
    shape = va.make_shape(w.B, w.T, w.Hq, w.Hkv, w.D, 0)

    def call(idx):
        ws = va.Workspace.for_shape(shape)
        run_library(w, "parent", indices=dev_i32(idx), n_indices=dev_i32(ref["n_indices"]), workspace=ws)
        return ws

    out_ws = call(ref["indices"])
    va.verify_attn_check_status(out_ws)  # the builder's sets are valid
    dup = ref["indices"].copy()
    dup[1, 0, 7] = dup[1, 0, 6]  # listed twice
    with pytest.raises(va.VerifyAttnError) as ei:
        va.verify_attn_check_status(call(dup))
    assert ei.value.status == va.api.VA_ERR_DEVICE_INVALID
    swapped = ref["indices"].copy()
    swapped[2, 1, [10, 11]] = swapped[2, 1, [11, 10]]  # out of order
    with pytest.raises(va.VerifyAttnError) as ei:
        va.verify_attn_check_status(call(swapped))
    assert ei.value.status == va.api.VA_ERR_DEVICE_INVALID
    far = ref["indices"].copy()
    far[0, 0, 5] = 10 ** 6  # past the sequence
    with pytest.raises(va.VerifyAttnError) as ei:
        va.verify_attn_check_status(call(far))
    assert ei.value.status == va.api.VA_ERR_DEVICE_BOUNDS


def test_sparse_full_index_equals_dense_on_gpu():
    w = W.make_workload("sparse", seed=4, B=2, L_lo=100, L_hi=300, budget=512, window=8, n_sink=2, m_draft=3)
    Lmax = int(w.seqlens.max())
    idx = np.full((w.B, w.Hkv, Lmax), -1, np.int32)
    cnt = np.zeros((w.B, w.Hkv), np.int32)
    for b in range(w.B):
        idx[b, :, : w.seqlens[b]] = np.arange(w.seqlens[b])
        cnt[b] = w.seqlens[b]
    out_s, lse_s = run_library(w, "parent", indices=dev_i32(idx), n_indices=dev_i32(cnt))
    w.layout = "dense"
    out_d, lse_d = run_library(w, "parent")
    ref = oracle.verify(w)
    compare(out_s, lse_s, ref)
    compare(out_d, lse_d, ref)


# ----------------------------------------------------------------------------
# verify index set (a5)
# ----------------------------------------------------------------------------

@pytest.fixture(params=["sampled", "radix"])
def index_path(request):
    """Runs a test with the builder's default path (the sampled-threshold
    select, falling back to the radix select where the sample cannot decide)
    and with the radix select over all keys only."""
    L = va.api.lib()
    assert L.verify_attn_test_index_path(1 if request.param == "radix" else 0) == 0
    yield request.param
    assert L.verify_attn_test_index_path(0) == 0


@pytest.mark.parametrize("L_lo,L_hi", [(1, 300), (2000, 5000), (40000, 50000)])
def test_build_index_bit_exact(L_lo, L_hi, index_path):
    """Includes L below the budget, ties (coarse scores) and L past the shared-memory cache."""
    rng = np.random.default_rng(L_hi)
    B, Hkv = 4, 3
    seqlens = rng.integers(L_lo, L_hi + 1, size=B).astype(np.int32)
    stride = int(seqlens.max()) + 5
    sd = (rng.integers(0, 50, size=(B, Hkv, stride)) / 49).astype(np.float32)
    st = rng.random((B, Hkv, stride), dtype=np.float32)
    st[0, 0, :10] = -0.0
    st[0, 0, 10:20] = 0.0
    sd[1, 1, :] = np.float32(0.5)  # all ties
    args = (4, 64, 300, 1024)
    ref_idx, ref_n = oracle.build_verify_index(sd, st, seqlens, *args)
    idx, n = va.verify_build_index(dev_i32(seqlens), torch.from_numpy(sd).cuda(), torch.from_numpy(st).cuda(), *args)
    assert np.array_equal(n.cpu().numpy(), ref_n)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)


@pytest.mark.parametrize("dist", ["normal", "negative", "wide", "few_distinct", "step"])
@pytest.mark.parametrize("m_draft", [0, 300])
def test_build_index_score_distributions(dist, m_draft, index_path):
    """Score shapes that move the k-th key across the radix digits: signed and
    negative scores, a wide exponent range, a handful of distinct values (ties
    at every digit), and values spaced so bucket edges fall at the threshold."""
    rng = np.random.default_rng(zlib.crc32(f"{dist}{m_draft}".encode()))
    B, Hkv = 3, 2
    seqlens = rng.integers(9000, 30000, size=B).astype(np.int32)
    stride = int(seqlens.max())

    def draw():
        if dist == "normal":
            return rng.standard_normal((B, Hkv, stride))
        if dist == "negative":
            return -rng.random((B, Hkv, stride)) - 1.0
        if dist == "wide":
            return rng.standard_normal((B, Hkv, stride)) * np.exp2(rng.integers(-60, 60, size=(B, Hkv, stride)))
        if dist == "few_distinct":
            return rng.integers(0, 7, size=(B, Hkv, stride)) * 0.25
        # step: consecutive float32 values, so digits differ only in the low bits
        return np.float32(1.0) + rng.integers(0, 4096, size=(B, Hkv, stride)) * np.float32(2.0 ** -23)

    sd = draw().astype(np.float32)
    st = draw().astype(np.float32)
    args = (4, 200, m_draft, 1500)
    ref_idx, ref_n = oracle.build_verify_index(sd, st, seqlens, *args)
    idx, n = va.verify_build_index(dev_i32(seqlens), torch.from_numpy(sd).cuda(), torch.from_numpy(st).cuda(), *args)
    assert np.array_equal(n.cpu().numpy(), ref_n)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)


@pytest.mark.parametrize("n_tied", [2, 5, 32, 33, 200])
def test_build_index_ties_at_the_threshold(n_tied, index_path):
    """Continuous scores with n_tied copies of the value at the k-th rank of
    each select, spread over positions: the quota ends inside the tied run,
    so the tie rule (lowest positions first) decides -- in the sampled path by
    ranking up to 32 tied keys, beyond that by the radix select."""
    rng = np.random.default_rng(n_tied)
    B, Hkv = 2, 2
    seqlens = np.array([24000, 17000], np.int32)
    stride = int(seqlens.max())
    sd = rng.random((B, Hkv, stride), dtype=np.float32)
    st = rng.random((B, Hkv, stride), dtype=np.float32)
    n_sink, window, m_draft, budget = 4, 256, 894, 2048
    for b in range(B):
        L = int(seqlens[b])
        for h in range(Hkv):
            for arr, k in ((sd, m_draft), (st, budget - n_sink - window - m_draft)):
                row = arr[b, h, :L]
                order = np.argsort(-row[n_sink:L - window], kind="stable") + n_sink
                v = row[order[k - 1]]
                pos = rng.choice(order[k:k + 4 * n_tied], size=n_tied - 1, replace=False)
                row[pos] = v  # n_tied keys equal to the k-th largest
    args = (n_sink, window, m_draft, budget)
    ref_idx, ref_n = oracle.build_verify_index(sd, st, seqlens, *args)
    idx, n = va.verify_build_index(dev_i32(seqlens), torch.from_numpy(sd).cuda(), torch.from_numpy(st).cuda(), *args)
    assert np.array_equal(n.cpu().numpy(), ref_n)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)


# ----------------------------------------------------------------------------
# combine (exposed merge)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("D", [64, 128])
def test_combine_matches_oracle_merge(D):
    rng = np.random.default_rng(D)
    S, R = 7, 33
    o = rng.standard_normal((S, R, D)).astype(np.float32)
    l = (rng.standard_normal((S, R)) * 3).astype(np.float32)
    l[2, :5] = -np.inf
    l[:, 7] = -np.inf  # a row with every part empty
    ro, rl = oracle.lse_merge(o.astype(np.float64), l.astype(np.float64))
    out, lse = va.verify_attn_combine(torch.from_numpy(o).cuda(), torch.from_numpy(l).cuda())
    out = out.cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.isneginf(lse[7]) and np.all(out[7] == 0)
    fin = np.isfinite(rl)
    assert np.abs(out - ro).max() < 1e-5
    assert np.abs(lse[fin] - rl[fin]).max() < 1e-5


# ----------------------------------------------------------------------------
# errors recorded on the device, bounded waits, determinism
# ----------------------------------------------------------------------------

def test_device_bounds_are_reported_not_faulted():
    w = W.make_workload("paged", seed=5, B=3, L_lo=100, L_hi=200)
    table = w.page_table.copy()
    table[1, 2] = 10 ** 6  # page out of range: clamped, recorded
    shape = va.make_shape(w.B, w.T, w.Hq, w.Hkv, w.D, 0)
    ws = va.Workspace.for_shape(shape)
    va.verify_attn_paged(w.q.cuda(), w.k_pages.cuda(), w.v_pages.cuda(), dev_i32(table), dev_i32(w.seqlens),
                         tree_mask=dev_words(w.mask_words), workspace=ws)
    with pytest.raises(va.VerifyAttnError) as ei:
        va.verify_attn_check_status(ws)
    assert ei.value.status == va.api.VA_ERR_DEVICE_BOUNDS
    # a seqlen past the cache is clamped and recorded too
    wd = W.make_workload("chain", seed=6, L=300)
    sl = wd.seqlens.copy()
    sl[0] = wd.max_cache_len
    shape = va.make_shape(1, wd.T, wd.Hq, wd.Hkv, wd.D, 0)
    ws2 = va.Workspace.for_shape(shape)
    va.verify_attn_dense(wd.q.cuda(), wd.k_cache.cuda(), wd.v_cache.cuda(), dev_i32(sl), workspace=ws2)
    with pytest.raises(va.VerifyAttnError):
        va.verify_attn_check_status(ws2)
    # the workspace is usable again afterwards
    out, lse = run_library(wd, "parent", workspace=ws2)
    va.verify_attn_check_status(ws2)
    compare(out, lse, oracle.verify(wd))


def test_bounded_wait_times_out_cleanly():
    ws = va.Workspace(256)
    st = va.api.lib().verify_attn_selftest_wait_timeout(ws.ptr, 2_000_000, va.api._stream())
    assert st == 0
    with pytest.raises(va.VerifyAttnError) as ei:
        va.verify_attn_check_status(ws)
    assert ei.value.status == va.api.VA_ERR_TIMEOUT
    va.verify_attn_check_status(ws)


def test_deterministic_and_workspace_reuse():
    w = W.make_workload("chain", seed=7, L=5000)
    shape = va.make_shape(1, w.T, w.Hq, w.Hkv, w.D, 0)
    ws = va.Workspace.for_shape(shape)
    o1, l1 = run_library(w, "parent", workspace=ws)
    o2, l2 = run_library(w, "parent", workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    va.verify_attn_check_status(ws)


def test_workspace_reused_across_shapes():
    """One workspace, sized for the largest, serves calls of three shapes in a
    row (32, then 64 packed rows; one and two sequences): the merge counters
    sit at the same place for every shape and each call leaves them at zero."""
    cases = [W.make_workload("chain", seed=201, L=4000),
             W.make_workload("chain", seed=202, B=2, L_lo=3000, L_hi=9000),
             W.make_workload("chain", seed=203, T=16, L=7000),
             W.make_workload("chain", seed=204, L=2500)]
    need = max(va.api.workspace_size(va.make_shape(w.B, w.T, w.Hq, w.Hkv, w.D, 0)) for w in cases)
    ws = va.Workspace(need)
    for w in cases:
        out, lse = run_library(w, "parent", workspace=ws)
        va.verify_attn_check_status(ws)
        compare(out, lse, oracle.verify(w), strict=True)


def test_timeout_then_recovery():
    """A real timeout inside the attention kernel, made on the host: one CTA's
    announcement of its segment parts is dropped, so the other parts of those
    segments wait for it until a 2 ms limit runs out.  The call reports
    VA_ERR_TIMEOUT; after verify_attn_workspace_init the same workspace gives
    the oracle's result again."""
    L = va.api.lib()
    w = W.make_workload("chain", seed=205, L=5000)  # 8 segments of 40 tiles: all split over CTAs
    ws = va.Workspace.for_shape(va.make_shape(w.B, w.T, w.Hq, w.Hkv, w.D, 0))
    assert L.verify_attn_test_inject(2_000_000, 0) == 0
    try:
        run_library(w, "parent", workspace=ws)
        with pytest.raises(va.VerifyAttnError) as ei:
            va.verify_attn_check_status(ws)
        assert ei.value.status == va.api.VA_ERR_TIMEOUT
    finally:
        assert L.verify_attn_test_inject(0, -1) == 0
    assert L.verify_attn_workspace_init(ws.ptr, ws.nbytes, va.api._stream()) == 0
    for _ in range(2):
        out, lse = run_library(w, "parent", workspace=ws)
        va.verify_attn_check_status(ws)
        compare(out, lse, oracle.verify(w), strict=True)


@pytest.mark.parametrize("kernel", ["tc", "tcp"])
def test_timeout_then_recovery_many_rows(kernel, monkeypatch):
    """The same injected timeout in the many-row kernels (tree workload shape,
    two kv-heads): every segment is cut over many CTAs."""
    if kernel == "tcp":
        monkeypatch.setenv("VA_MANY_ROWS_KERNEL", "tcp")
    else:
        monkeypatch.delenv("VA_MANY_ROWS_KERNEL", raising=False)
    L = va.api.lib()
    w = W.make_workload("tree", seed=206, Hkv=2, Hq=8, L=20000)
    ws = va.Workspace.for_shape(va.make_shape(w.B, w.T, w.Hq, w.Hkv, w.D, 0))
    assert L.verify_attn_test_inject(2_000_000, 0) == 0
    try:
        run_library(w, "parent", workspace=ws)
        with pytest.raises(va.VerifyAttnError) as ei:
            va.verify_attn_check_status(ws)
        assert ei.value.status == va.api.VA_ERR_TIMEOUT
    finally:
        assert L.verify_attn_test_inject(0, -1) == 0
    assert L.verify_attn_workspace_init(ws.ptr, ws.nbytes, va.api._stream()) == 0
    out, lse = run_library(w, "parent", workspace=ws)
    va.verify_attn_check_status(ws)
    compare(out, lse, oracle.verify(w), strict=True)


def test_workspace_too_small_is_rejected():
    w = W.make_workload("chain", seed=8, L=100)
    small = va.Workspace(1024)
    with pytest.raises(va.VerifyAttnError) as ei:
        run_library(w, "parent", workspace=small)
    assert ei.value.status == va.api.VA_ERR_WORKSPACE


@pytest.mark.parametrize("case", ["sparse", "paged_isolated", "dense_ragged"])
def test_partials_never_read_stale_workspace(case):
    """Ragged lengths with fewer key tiles than CTAs: every partial slot the merge
    reads must have been written by this very call.  The partial slots hold NaN
    bytes first, so reading a stale slot cannot go unnoticed."""
    if case == "sparse":
        w = W.make_workload("sparse", seed=3, B=3, L_lo=200, L_hi=900, budget=256, window=32, n_sink=4, m_draft=60)
    elif case == "paged_isolated":
        w = W.make_workload("paged", seed=17, B=4, L_lo=40, L_hi=300, page_size=16, tree="block_isolated")
    else:
        w = W.make_workload("tree", seed=4, B=5, L_lo=1, L_hi=200, T=9, tree="random")
    ref = oracle.verify(w)
    shape = va.make_shape(w.B, w.T, w.Hq, w.Hkv, w.D, 0)
    ws = va.Workspace.for_shape(shape)
    # initialised (status word and merge counters at zero), then the partial
    # slots, which fill most of the workspace, overwritten with NaN bytes
    assert va.api.lib().verify_attn_workspace_init(ws.ptr, ws.nbytes, va.api._stream()) == 0
    ws.buffer[ws.offset + ws.nbytes // 4: ws.offset + ws.nbytes].fill_(0xFF)
    kw = {}
    if w.layout == "sparse":
        kw = dict(indices=dev_i32(ref["indices"]), n_indices=dev_i32(ref["n_indices"]))
    out, lse = run_library(w, "mask" if w.parent is None else "parent", workspace=ws, **kw)
    va.verify_attn_check_status(ws)
    compare(out, lse, ref)


# ----------------------------------------------------------------------------
# the online softmax's reference maximum has to move
# ----------------------------------------------------------------------------

def _reference_jumps(w):
    """Key 0 of every sequence and kv-head scores far below the draft rows'
    usual scores, and every key of the second half of the sequence is shifted
    along the rows' mean query direction so that its score rises by about 8:
    the first tile's reference (key 0) has to move at once, and the first tile
    of the second half moves it again, so O and l are rescaled.  The weight
    stays spread over the many keys of the second half (a few dominant keys
    would test the precision of a single bf16 P instead, 2^-9 of each weight)."""
    q = w.q.float()
    group = w.Hq // w.Hkv
    for b in range(w.B):
        n = int(w.seqlens[b]) + w.T
        for h in range(w.Hkv):
            rows = q[b, :, h * group:(h + 1) * group].reshape(-1, w.D)
            u = rows.sum(0)
            u = u / u.norm()
            proj = float((rows @ u).mean())
            shift = 8.0 * w.D ** 0.5 / max(proj, 0.5)  # mean score rise of about 8
            slots = [(0, None)] + [(s, 1.0) for s in range(n // 2, n)]
            for slot, sign in slots:
                if w.layout == "paged":
                    ref = w.k_pages[w.page_table[b, slot // w.page_size], slot % w.page_size]
                else:
                    ref = w.k_cache[b, slot]
                if sign is None:
                    ref[h] = (-shift * u).to(w.q.dtype)
                else:
                    ref[h] = (ref[h].float() + shift * u).to(w.q.dtype)
    return w


@pytest.mark.parametrize("case", ["chain", "paged64rows", "tree", "sparse", "tiny_fp32"])
def test_reference_max_moves(case):
    if case == "chain":
        w = W.make_workload("chain", seed=81, B=2, L_lo=1500, L_hi=3000)
    elif case == "paged64rows":
        w = W.make_workload("paged", seed=82, B=3, L_lo=800, L_hi=2500, page_size=16)
    elif case == "tree":
        w = W.make_workload("tree", seed=83, B=1, Hkv=2, L=2500)
    elif case == "sparse":
        w = W.make_workload("sparse", seed=84, B=2, Hkv=2, L_lo=3000, L_hi=5000, budget=600, m_draft=200, window=64)
    else:
        w = W.make_workload("tiny", seed=85, L=2000)
    w = _reference_jumps(w)
    if w.layout == "sparse":  # the oracle's verify sets, handed to the library
        ref = oracle.verify(w)
        out, lse = run_library(w, "parent", indices=dev_i32(ref["indices"]), n_indices=dev_i32(ref["n_indices"]))
        torch.cuda.synchronize()
        compare(out, lse, ref)
    else:
        _check(w, "mask" if case == "paged64rows" else "parent")
