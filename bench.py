"""Benchmark: speculative-decoding verification attention on one GB300 per rank.

One *step* is one verification pass over one batch of the workload: the draft
tree's ancestor mask, the split-KV prefix pass, the masked draft-block pass and
the log-sum-exp merge (the sparse workload adds the verify-index build).  The
headline workload is the long-context token tree: a 64-node tree of depth 6
over a 131072-token bf16 cache (B1, Hq32, Hkv8, d128); every other measured
workload (chain, sparse, paged, tiny) is reported under ``other_configs`` with
the same evidence.

Reported (one JSON line on rank 0):
  value        algorithmic KV bytes of all ranks / max-over-ranks time, GB/s
               (KV bytes = (prefix keys + T) * d * 2 (K, V) * elem per kv-head)
  tokens_per_s verified draft tokens per second
  roofline     the dominant kernel's achieved GB/s (bytes per launch over its
               CUDA-event duration) against the measured HBM copy bandwidth
  sustained    the same step replayed for at least 0.6 s with the SM clocks
               sampled every 20 ms (dozens of samples under load)
  e2e          the same metric through the public API with host buffers:
               per step, H2D of the step's new inputs (q, the draft tokens'
               K/V rows, tree parents, seqlens), the call, D2H of out + lse;
               two input sets used in turn, so the copies of the neighbouring
               steps overlap this step's call on a second stream
  cpu_baseline the fp64 oracle timed on this host's cores (a baseline only)

Timing: W warm-up steps, then exactly K steps replayed from CUDA graphs; each
step reads a different copy of the inputs and the copies together exceed the
L2 cache, so no step is served from L2.  Under torchrun every rank runs its own
replica (no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "verify-attention achieved HBM GB/s (% of GB300 peak) and verified tokens/s"
L2_BYTES = 129 * 1024 * 1024
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------
# device-side workload
# ----------------------------------------------------------------------------

class DeviceCase:
    """One resident copy of a workload's inputs and outputs on the GPU."""

    def __init__(self, w, va):
        self.w = w
        self.va = va
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()  # noqa: E731
        self.q = w.q.cuda()
        self.seqlens = i32(w.seqlens)
        self.parent = i32(w.parent) if w.parent is not None else None
        self.mask = (torch.from_numpy(np.ascontiguousarray(w.mask_words).view(np.int32)).cuda()
                     if w.mask_words is not None else None)
        if w.layout in ("dense", "sparse"):
            self.k = w.k_cache.cuda()
            self.v = w.v_cache.cuda()
        else:
            self.k = w.k_pages.cuda()
            self.v = w.v_pages.cuda()
            self.page_table = i32(w.page_table)
        if w.layout == "sparse":
            self.sd = torch.from_numpy(w.score_draft).cuda()
            self.st = torch.from_numpy(w.score_target).cuda()
            self.idx = torch.empty(w.B, w.Hkv, w.budget, dtype=torch.int32, device="cuda")
            self.nidx = torch.empty(w.B, w.Hkv, dtype=torch.int32, device="cuda")
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(w.B, w.Hq, w.T, dtype=torch.float32, device="cuda")
        shape = va.make_shape(w.B, w.T, w.Hq, w.Hkv, w.D, 0 if w.dtype == "bf16" else 2, w.scale)
        self.ws = va.Workspace.for_shape(shape)

    def step(self):
        """One verification pass (all on the current stream)."""
        va, w = self.va, self.w
        if w.layout == "dense":
            va.verify_attn_dense(self.q, self.k, self.v, self.seqlens, tree_parent=self.parent, tree_mask=self.mask,
                                 out=self.out, lse=self.lse, workspace=self.ws, scale=w.scale)
        elif w.layout == "paged":
            va.verify_attn_paged(self.q, self.k, self.v, self.page_table, self.seqlens, tree_parent=self.parent,
                                 tree_mask=self.mask, out=self.out, lse=self.lse, workspace=self.ws, scale=w.scale)
        else:
            va.verify_build_index(self.seqlens, self.sd, self.st, w.n_sink, w.window, w.m_draft, w.budget,
                                  indices=self.idx, n_indices=self.nidx, workspace=self.ws)
            va.verify_attn_sparse(self.q, self.k, self.v, self.seqlens, self.idx, self.nidx, tree_parent=self.parent,
                                  tree_mask=self.mask, out=self.out, lse=self.lse, workspace=self.ws, scale=w.scale)

    def resident_bytes(self):
        tot = 0
        for t in (self.q, self.k, self.v):
            tot += t.numel() * t.element_size()
        return tot


def n_copies_for(w):
    per_step = w.kv_bytes()
    return int(min(8, max(2, math.ceil(3 * L2_BYTES / max(per_step, 1)))))


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        try:
            idx = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
            phys = idx[device_index] if idx and idx[0] != "" and device_index < len(idx) else str(device_index)
            self.path = f"/tmp/va_clocks_{os.getpid()}.csv"
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", phys, f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[0]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(num(r[1]) for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# measurement
# ----------------------------------------------------------------------------

def time_graph_steps(cases, steps, warmup, graph_steps):
    """Capture ``graph_steps`` consecutive steps (rotating copies) in one CUDA graph;
    replay it to run ``warmup`` + ``steps`` steps; return seconds for the timed steps."""
    stream = torch.cuda.Stream()
    # eager warm-up outside capture (first-call attribute setup)
    with torch.cuda.stream(stream):
        for i in range(max(1, len(cases))):
            cases[i % len(cases)].step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(graph_steps):
            cases[i % len(cases)].step()
    reps_w = max(1, math.ceil(warmup / graph_steps))
    reps = max(1, math.ceil(steps / graph_steps))
    for _ in range(reps_w):
        graph.replay()
    torch.cuda.synchronize()
    return graph, reps


def per_call_durations(cases, n_calls):
    """CUDA-event duration of each verification call, enqueued behind a spin
    kernel so host launch latency never enters an interval."""
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_calls)]
    torch.cuda._sleep(int(50e6))  # ~25 ms of spinning while the host enqueues
    for i in range(n_calls):
        c = cases[i % len(cases)]
        ev[i][0].record(stream)
        c.step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e-3 for a, b in ev]


def measure_next_rows(va, peak, steps=1024):
    """The steps after verification at the paged workload's shape (B64, T16
    random trees, 16-row pages): greedy acceptance, then the KV commit of the
    accepted rows.  Device time per call from CUDA events around graphs of 64
    calls; the commit's bytes are the rows it moves, read once and written once."""
    w = W.make_workload("paged", seed=0, tree="random")
    rng = np.random.default_rng(1)
    # tokens from a 2-symbol alphabet: paths of a few nodes, some rows moved
    tgt = rng.integers(0, 2, size=(w.B, w.T + 1)).astype(np.int32)
    draft = rng.integers(0, 2, size=(w.B, w.T)).astype(np.int32)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()  # noqa: E731
    parent, d_draft, d_tgt = i32(w.parent), i32(draft), i32(tgt)
    k, v, table, seqlens = w.k_pages.cuda(), w.v_pages.cuda(), i32(w.page_table), i32(w.seqlens)
    path, n, bonus = va.verify_accept_greedy(parent, d_draft, d_tgt)
    seq_out = torch.empty_like(seqlens)
    torch.cuda.synchronize()
    p_h, n_h = path.cpu().numpy(), n.cpu().numpy()
    moved = int(sum(int(np.sum(p_h[b, : n_h[b]] != np.arange(n_h[b]))) for b in range(w.B)))
    row_bytes = w.D * 2
    commit_bytes = moved * w.Hkv * 2 * row_bytes * 2
    res = {"workload": f"paged shape: B{w.B} T{w.T} Hkv{w.Hkv} d{w.D} bf16, random trees, 16-row pages",
           "mean_accepted": round(float(n_h.mean()), 2), "rows_moved_per_call": moved * w.Hkv * 2}

    def timed(fn):
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(64):
                fn()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = max(1, steps // 64)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / (reps * 64)

    t_acc = timed(lambda: va.verify_accept_greedy(parent, d_draft, d_tgt, path=path, n_accept=n, bonus=bonus))
    # the same accepted rows are moved every call (the cache content changes, the traffic does not)
    t_com = timed(lambda: va.verify_commit_kv_paged(k, v, table, seqlens, path, n, seqlens_out=seq_out))
    res["accept_us"] = round(t_acc * 1e6, 3)
    res["commit_us"] = round(t_com * 1e6, 3)
    res["commit_GBps"] = round(commit_bytes / t_com / 1e9, 1)
    res["commit_frac_of_measured_hbm"] = round(commit_bytes / t_com / 1e9 / peak, 4)
    res["note"] = "both latency-bound at this size: a few KB per sequence"
    return res


def measure_rope(va, peak, steps=1024):
    """The rotary embedding of the draft block at the paged workload's shape
    (B64, T16, Hq32/Hkv8, d128 bf16, 16-row pages, tree positions L + depth):
    every head of q and the T draft key rows, read and written once.  Device
    time per call from CUDA events around graphs of 64 calls (the rows are
    rotated again each call; the traffic does not change)."""
    w = W.make_workload("paged", seed=0, tree="random")
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()  # noqa: E731
    depth = np.stack([W.chain_depths(p) for p in w.parent])
    pos = i32(w.seqlens[:, None] + depth)
    q, k, table, seqlens = w.q.cuda(), w.k_pages.cuda(), i32(w.page_table), i32(w.seqlens)
    nbytes = 2 * w.B * w.T * (w.Hq + w.Hkv) * w.D * 2

    def fn():
        va.verify_rope_draft_paged(q, k, table, seqlens, pos, 500000.0)

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(64):
            fn()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // 64)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / (reps * 64)
    return {"workload": f"paged shape: B{w.B} T{w.T} Hq{w.Hq} Hkv{w.Hkv} d{w.D} bf16, 16-row pages, "
                        "tree positions",
            "us_per_call": round(t * 1e6, 3), "algorithmic_bytes": nbytes,
            "GBps": round(nbytes / t / 1e9, 1), "frac_of_measured_hbm": round(nbytes / t / 1e9 / peak, 4),
            "launches_per_call": 1, "cpu_baseline": oracle_rate(*rope_oracle_sample()),
            "note": "about 21 MB a call: launch- and latency-bound, the rows mostly served from L2 in the loop"}


def measure_rope_fused(va, peak, steps=512):
    """The rotary embedding inside the attention kernels against the separate
    pass: at the paged and chain workloads' shapes, one step of (rotation pass
    + unrotated attention) against one attention call given the positions
    (tree / chain positions L + depth, base 500000).  Device time per step from
    CUDA events around graphs of 32 steps over resident input copies larger
    than L2."""
    res = {}
    for name in ("paged", "chain"):
        w = W.make_workload(name, seed=0)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()  # noqa: E731
        depth = (np.stack([W.chain_depths(p) for p in w.parent]) if w.parent is not None
                 else np.tile(np.arange(w.T, dtype=np.int32), (w.B, 1)))
        pos = i32(w.seqlens[:, None] + depth)
        cases = [DeviceCase(w, va) for _ in range(n_copies_for(w))]

        def sep(c):
            if w.layout == "paged":
                va.verify_rope_draft_paged(c.q, c.k, c.page_table, c.seqlens, pos, 500000.0)
            else:
                va.verify_rope_draft_dense(c.q, c.k, c.seqlens, pos, 500000.0)
            c.step()

        def fused(c):
            if w.layout == "paged":
                va.verify_attn_paged(c.q, c.k, c.v, c.page_table, c.seqlens, tree_parent=c.parent, tree_mask=c.mask,
                                     positions=pos, rope_base=500000.0, out=c.out, lse=c.lse, workspace=c.ws,
                                     scale=w.scale)
            else:
                va.verify_attn_dense(c.q, c.k, c.v, c.seqlens, tree_parent=c.parent, tree_mask=c.mask,
                                     positions=pos, rope_base=500000.0, out=c.out, lse=c.lse, workspace=c.ws,
                                     scale=w.scale)

        out = {}
        for tag, fn in (("rotation_pass_then_attention_us", sep), ("attention_with_rotation_inside_us", fused),
                        ("attention_without_rotation_us", lambda c: c.step())):
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for c in cases:
                    fn(c)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(32):
                    fn(cases[i % len(cases)])
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            reps = max(1, steps // 32)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            out[tag] = round(e0.elapsed_time(e1) * 1e3 / (reps * 32), 3)
            del g
        for c in cases:
            va.verify_attn_check_status(c.ws)
        res[name] = out
        del cases
        torch.cuda.empty_cache()
    return res


def measure_scoring(va, peak, steps=256):
    """The importance pass of a few query heads at the sparse workload's shape
    (B16, T5, Hq32/Hkv8, prefixes 16K-32K, two synthetic retrieval heads on
    kv-heads 2 and 5).  Device time per call from CUDA events around graphs
    of 16 calls; the algorithmic bytes are the K rows of the listed kv-heads
    (read once), the q rows and the importance rows written (Hkv per position).
    The K rows of one call (about 200 MB) exceed the L2."""
    w = W.make_workload("sparse", seed=0)
    heads = list(w.score_heads)
    group = w.Hq // w.Hkv
    n_kv = len({h // group for h in heads})
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()  # noqa: E731
    q, k, seqlens = w.q.cuda(), w.k_cache.cuda(), i32(w.seqlens)
    score = torch.empty(w.B, w.Hkv, w.max_cache_len, dtype=torch.float32, device="cuda")
    scratch = va.ScoreScratch(w.B, w.T, len(heads), w.max_cache_len)
    total_L = int(w.seqlens.astype(np.int64).sum())
    nbytes = total_L * n_kv * w.D * 2 + w.B * w.T * len(heads) * w.D * 2 + total_L * w.Hkv * 4

    def fn():
        va.verify_head_importance(q, k, seqlens, heads, score=score, scale=w.scale, scratch=scratch)

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(16):
            fn()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // 16)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / (reps * 16)
    return {"workload": f"sparse shape: B{w.B} T{w.T} Hq{w.Hq} Hkv{w.Hkv} d{w.D} bf16, prefixes "
                        f"16K-32K, heads {heads}",
            "us_per_call": round(t * 1e6, 3), "algorithmic_bytes": nbytes,
            "GBps": round(nbytes / t / 1e9, 1), "frac_of_measured_hbm": round(nbytes / t / 1e9 / peak, 4),
            "launches_per_call": 2, "cpu_baseline": oracle_rate(*scoring_oracle_sample(w))}


def measure_sparse_overhead(va, scoring_us, steps=128):
    """At the sparse workload's shape: the verification over the whole cache
    (dense, every committed key) against the sparse path's parts -- the
    verify-set build, the gathered attention -- and the importance pass
    (timed by measure_scoring), each from CUDA events around graphs of 16
    calls.  The full-cache call reads ~1.6 GB of K/V, far beyond L2; the index
    build reads 25 MB of scores, which a serving step would also find in L2
    right after the importance pass wrote them."""
    w = W.make_workload("sparse", seed=0)
    c = DeviceCase(w, va)
    c.step()  # the verify sets, for the sparse-attention timing

    def timed(fn):
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(16):
                fn()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = max(1, steps // 16)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (reps * 16)

    full_us = timed(lambda: va.verify_attn_dense(c.q, c.k, c.v, c.seqlens, tree_parent=c.parent, tree_mask=c.mask,
                                                 out=c.out, lse=c.lse, workspace=c.ws, scale=w.scale))
    index_us = timed(lambda: va.verify_build_index(c.seqlens, c.sd, c.st, w.n_sink, w.window, w.m_draft, w.budget,
                                                   indices=c.idx, n_indices=c.nidx, workspace=c.ws))
    attn_us = timed(lambda: va.verify_attn_sparse(c.q, c.k, c.v, c.seqlens, c.idx, c.nidx, tree_parent=c.parent,
                                                  tree_mask=c.mask, out=c.out, lse=c.lse, workspace=c.ws,
                                                  scale=w.scale))
    res = {"workload": f"sparse shape: B{w.B} T{w.T} Hq{w.Hq} Hkv{w.Hkv} d{w.D} bf16, prefixes 16K-32K, "
                       f"verify sets of {w.budget}",
           "full_cache_attention_us": round(full_us, 2), "index_build_us": round(index_us, 2),
           "sparse_attention_us": round(attn_us, 2)}
    if scoring_us is not None:
        res["importance_pass_us"] = scoring_us
        res["selection_overhead_frac_of_full_cache"] = round((index_us + scoring_us) / full_us, 4)
        res["sparse_path_speedup_vs_full_cache"] = round(full_us / (index_us + scoring_us + attn_us), 3)
    return res


def e2e_measure(w, va, steps):
    """Through the public API with host buffers.  Every step copies its new
    inputs from pinned host memory to the device, runs the call, and copies out
    and lse back to pinned host memory.  Two device input sets are used in
    turn: the uploads of step i+1 and the read-back of step i-1 run on a copy
    stream, ordered by events around step i's call on the compute stream, so
    only the first upload and the last read-back are not hidden; one
    synchronisation at the end.  Returns (seconds per step, H2D bytes, D2H bytes)."""
    cases = [DeviceCase(w, va), DeviceCase(w, va)]
    T, B = w.T, w.B
    pin = lambda t: t.contiguous().pin_memory()  # noqa: E731
    h_q = pin(w.q)
    h_seq = pin(torch.from_numpy(np.asarray(w.seqlens, np.int32)))
    h_par = pin(torch.from_numpy(np.asarray(w.parent, np.int32))) if w.parent is not None else None
    h_mask = (pin(torch.from_numpy(np.ascontiguousarray(w.mask_words).view(np.int32)))
              if w.mask_words is not None else None)
    # the draft tokens' new K/V rows, appended at slots L_b .. L_b+T-1: one copy
    # per (sequence, page) run of slots (dense: one per sequence)
    runs = []  # (b, first slot, n slots, page or -1)
    for b_ in range(B):
        L = int(w.seqlens[b_])
        j = 0
        while j < T:
            if w.layout == "paged":
                slot = L + j
                n = min(T - j, w.page_size - slot % w.page_size)
                runs.append((b_, slot, n, int(w.page_table[b_, slot // w.page_size])))
            else:
                n = T
                runs.append((b_, L + j, n, -1))
            j += n

    def src_rows(kv, b_, slot, n, page):
        if page >= 0:
            pages = w.k_pages if kv == 0 else w.v_pages
            return pin(pages[page, slot % w.page_size: slot % w.page_size + n])
        cache = w.k_cache if kv == 0 else w.v_cache
        return pin(cache[b_, slot: slot + n])

    h_new = [(src_rows(0, *r), src_rows(1, *r)) for r in runs]
    h_out = [torch.empty_like(h_q).pin_memory() for _ in range(2)]
    h_lse = [torch.empty(B, w.Hq, T, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = h_q.numel() * h_q.element_size() + h_seq.numel() * 4
    h2d += (h_par.numel() * 4 if h_par is not None else 0) + (h_mask.numel() * 4 if h_mask is not None else 0)
    h2d += sum(a.numel() * a.element_size() + c.numel() * c.element_size() for a, c in h_new)
    if w.layout == "sparse":
        h_sd = pin(torch.from_numpy(w.score_draft))
        h_st = pin(torch.from_numpy(w.score_target))
        h2d += 2 * h_sd.numel() * 4
    d2h = h_out[0].numel() * h_out[0].element_size() + h_lse[0].numel() * 4

    def upload(case):
        case.q.copy_(h_q, non_blocking=True)
        case.seqlens.copy_(h_seq, non_blocking=True)
        if h_par is not None:
            case.parent.copy_(h_par, non_blocking=True)
        if h_mask is not None:
            case.mask.copy_(h_mask, non_blocking=True)
        for (b_, slot, n, page), (hk, hv) in zip(runs, h_new):
            if page >= 0:
                r0 = slot % w.page_size
                case.k[page, r0: r0 + n].copy_(hk, non_blocking=True)
                case.v[page, r0: r0 + n].copy_(hv, non_blocking=True)
            else:
                case.k[b_, slot: slot + n].copy_(hk, non_blocking=True)
                case.v[b_, slot: slot + n].copy_(hv, non_blocking=True)
        if w.layout == "sparse":
            case.sd.copy_(h_sd, non_blocking=True)
            case.st.copy_(h_st, non_blocking=True)

    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    up_done = [torch.cuda.Event(), torch.cuda.Event()]
    call_done = [torch.cuda.Event(), torch.cuda.Event()]

    def run(n_steps):
        with torch.cuda.stream(copy):
            upload(cases[0])
            up_done[0].record(copy)
        for i in range(n_steps):
            s = i & 1
            if i + 1 < n_steps:  # next step's inputs into the other set, once its last call is done
                with torch.cuda.stream(copy):
                    if i >= 1:
                        copy.wait_event(call_done[s ^ 1])
                    upload(cases[s ^ 1])
                    up_done[s ^ 1].record(copy)
            comp.wait_event(up_done[s])
            cases[s].step()
            call_done[s].record(comp)
            with torch.cuda.stream(copy):  # this step's result back to the host
                copy.wait_event(call_done[s])
                h_out[s].copy_(cases[s].out, non_blocking=True)
                h_lse[s].copy_(cases[s].lse, non_blocking=True)
        torch.cuda.synchronize()

    run(4)
    t0 = time.perf_counter()
    run(steps)
    dt = (time.perf_counter() - t0) / steps
    for c in cases:
        va.verify_attn_check_status(c.ws)
    return dt, h2d, d2h


def cpu_baseline(w, target_s=12.0, max_reps=50):
    """The fp64 oracle as it stands, on this host's cores, over whole kv-head
    groups of the same workload until about ``target_s`` seconds of work."""
    import oracle

    q = W.bf16_bits(w.q) if w.dtype == "bf16" else w.q.numpy()
    vis = oracle.draft_visibility(w)
    g = w.group
    per_key = w.D * 2 * w.elem_bytes
    done_bytes = 0
    groups = 0
    t0 = time.perf_counter()
    if w.layout == "dense":
        k = W.bf16_bits(w.k_cache) if w.dtype == "bf16" else w.k_cache.numpy()
        v = W.bf16_bits(w.v_cache) if w.dtype == "bf16" else w.v_cache.numpy()
        while time.perf_counter() - t0 < target_s and groups < max_reps * w.Hkv:
            h = groups % w.Hkv
            oracle.attention_dense(q[:, :, h * g:(h + 1) * g], k[:, :, h:h + 1], v[:, :, h:h + 1], w.seqlens, vis,
                                   w.scale)
            done_bytes += int((w.seqlens.astype(np.int64) + w.T).sum()) * per_key
            groups += 1
        sample = f"{groups} kv-head groups of the workload (each: all {w.B} sequences x {w.T} draft tokens x {g} heads)"
    else:
        # whole-workload passes (paged / sparse), bounded by time
        reps = 0
        while time.perf_counter() - t0 < target_s and reps < max_reps:
            oracle.verify(w)
            done_bytes += w.kv_bytes()
            reps += 1
        sample = f"{reps} full passes of the workload"
    dt = time.perf_counter() - t0
    return {"value": round(done_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": sample, "seconds": round(dt, 4)}


def oracle_rate(fn, nbytes, sample, target_s=4.0, max_reps=20):
    """Host-side GB/s of one oracle call ``fn`` that covers ``nbytes`` of the
    step's algorithmic bytes, repeated until about ``target_s`` seconds."""
    t0 = time.perf_counter()
    reps = 0
    while reps == 0 or (time.perf_counter() - t0 < target_s and reps < max_reps):
        fn()
        reps += 1
    dt = time.perf_counter() - t0
    return {"value": round(nbytes * reps / dt / 1e9, 4), "unit": "GB/s", "cores": os.cpu_count(),
            "kind": "oracle", "sample": f"{sample}; {reps} runs",
            "seconds": round(dt, 2)}


def scoring_oracle_sample(w, n_seq=2):
    """The importance pass of the oracle on the first ``n_seq`` sequences of
    workload ``w``: (callable, algorithmic bytes it covers, description)."""
    import oracle

    heads = list(w.score_heads)
    n_kv = len({h // w.group for h in heads})
    qb, kb = W.bf16_bits(w.q[:n_seq]), W.bf16_bits(w.k_cache[:n_seq])
    L = w.seqlens[:n_seq]
    nbytes = int(L.astype(np.int64).sum()) * (n_kv * w.D * 2 + w.Hkv * 4) + n_seq * w.T * len(heads) * w.D * 2
    return (lambda: oracle.head_importance(qb, kb, L, heads, w.scale)), nbytes, \
        f"sequences 0..{n_seq - 1} of the workload (numpy fp64, BLAS threads up to the cores)"


def rope_oracle_sample(B=4):
    """The oracle's rotation of the draft block on a B-sequence cut of the paged
    workload (its own page pool): (callable, algorithmic bytes, description)."""
    import oracle

    w = W.make_workload("paged", seed=0, B=B, tree="random")
    pos = (w.seqlens[:, None] + np.stack([W.chain_depths(p) for p in w.parent])).astype(np.int32)
    qb, kb = W.bf16_bits(w.q), W.bf16_bits(w.k_pages)
    nbytes = 2 * w.B * w.T * (w.Hq + w.Hkv) * w.D * 2
    return (lambda: oracle.rope_draft_paged(qb, kb, w.page_table, w.page_size, w.seqlens, pos, 500000.0)), \
        nbytes, f"{B} sequences of the paged workload (numpy fp64, one thread)"


# DRAM traffic per launch of the dominant kernel from one ncu capture of it
# (dram__bytes_read.sum + dram__bytes_write.sum, the --set full capture of
# `bench.py --profile <config>`), valid only while the sources that kernel is
# built from hash to those captured.
_HEADERS = ['va_common.cuh', 'va_pipeline.cuh', 'va_tcgen05.cuh', 'va_kernels.h', 'va_rope_fused.cuh', 'va_merge.cuh']
KERNEL_SOURCES = {"tc": ["va_attn_tc.cu"] + _HEADERS, "tck": ["va_attn_tck.cu"] + _HEADERS}
PROFILED_TRAFFIC = {
    "tree": {"sources": "tc", "sha256": "5f3eb81cd915d48d4d7ded3a3450edc49e011db4a13bdb337279b5b9734ee886",
             "kernel": "verify_attn_tc_kernel<2, TMA>", "bytes": 541492736},
    "chain": {"sources": "tck", "sha256": "82f27a4640fe712ccc1c3bc4dc5d7408724acaa1eecde6bd4dd2565ec887c29c",
              "kernel": "verify_attn_tck_kernel<32, TMA>", "bytes": 138061568},
    "sparse": {"sources": "tck", "sha256": "82f27a4640fe712ccc1c3bc4dc5d7408724acaa1eecde6bd4dd2565ec887c29c",
               "kernel": "verify_attn_tck_kernel<32, gather>", "bytes": 141492480},
    "paged": {"sources": "tck", "sha256": "82f27a4640fe712ccc1c3bc4dc5d7408724acaa1eecde6bd4dd2565ec887c29c",
              "kernel": "verify_attn_tck_kernel<64, TMA>", "bytes": 1470916864},
}


def kernel_sources_sha256(which):
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_masked_gb300", "csrc")
    for name in KERNEL_SOURCES[which]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(config):
    rec = PROFILED_TRAFFIC.get(config)
    if rec is None or rec["sha256"] != kernel_sources_sha256(rec["sources"]):
        return None
    return rec["bytes"]


def attention_path(w):
    """The dominant kernel of one verification call and the launches of one
    step (mirrors the library's row plan)."""
    R = (w.Hq // w.Hkv) * w.T
    small_rows = w.dtype == "bf16" and w.D == 128 and R <= 64 and os.environ.get("VA_SMALL_ROWS_KERNEL") != "mma"
    if small_rows:
        nr = 16 if R <= 16 else (32 if R <= 32 else 64)
        kernel, launches = f"verify_attn_tck_kernel<{nr}> (keys on TMEM lanes, LSE merge inside)", 1
    elif (w.dtype == "bf16" and w.D == 128 and R > 128 and os.environ.get("VA_MANY_ROWS_KERNEL") == "tcp"
          and (w.layout == "dense" or (w.layout == "paged" and w.page_size >= 8))):
        kernel, launches = "verify_attn_tcp_kernel (two M-tiles of rows on TMEM lanes, LSE merge inside)", 1
    elif w.dtype == "bf16" and w.D == 128:
        kernel, launches = "verify_attn_tc_kernel (rows on TMEM lanes, LSE merge inside)", 1
    else:
        kernel, launches = "verify_attn_kernel (mma.sync / fp32 SIMT) + split-segment merge kernel", 2
    if w.layout == "sparse":
        launches += 1  # the verify-index build
    return kernel, launches


def load_peak_hbm():
    try:
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------
# main
# ----------------------------------------------------------------------------

def run_profile(args):
    """A fixed number of eager verification steps of one workload: the
    command the committed ncu summaries are taken from."""
    import speculative_decoding_verification_masked_gb300 as va

    torch.cuda.set_device(0)
    va.api.lib(build_if_missing=False)
    if args.profile == "after":
        w = W.make_workload("paged", seed=0, tree="random")
        rng = np.random.default_rng(1)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()  # noqa: E731
        tgt = i32(rng.integers(0, 2, size=(w.B, w.T + 1)))
        draft = i32(rng.integers(0, 2, size=(w.B, w.T)))
        k, v = w.k_pages.cuda(), w.v_pages.cuda()
        ws = va.Workspace(256)
        for _ in range(args.calls):
            path, n, _ = va.verify_accept_greedy(i32(w.parent), draft, tgt, workspace=ws)
            va.verify_commit_kv_paged(k, v, i32(w.page_table), i32(w.seqlens), path, n, workspace=ws)
        torch.cuda.synchronize()
        va.verify_attn_check_status(ws)
        print(json.dumps({"profile": "after", "calls": args.calls, "status": "ok"}))
        return 0
    if args.profile == "rope":
        w = W.make_workload("paged", seed=0, tree="random")
        depth = np.stack([W.chain_depths(p) for p in w.parent])
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()  # noqa: E731
        q, k, ws = w.q.cuda(), w.k_pages.cuda(), va.Workspace(256)
        for _ in range(args.calls):
            va.verify_rope_draft_paged(q, k, i32(w.page_table), i32(w.seqlens), i32(w.seqlens[:, None] + depth),
                                       500000.0, workspace=ws)
        torch.cuda.synchronize()
        va.verify_attn_check_status(ws)
        print(json.dumps({"profile": "rope", "calls": args.calls, "status": "ok"}))
        return 0
    if args.profile == "score":
        w = W.make_workload("sparse", seed=0)
        q, k = w.q.cuda(), w.k_cache.cuda()
        seqlens = torch.from_numpy(w.seqlens).cuda()
        score = torch.empty(w.B, w.Hkv, w.max_cache_len, dtype=torch.float32, device="cuda")
        scratch = va.ScoreScratch(w.B, w.T, len(w.score_heads), w.max_cache_len)
        ws = va.Workspace(256)
        for _ in range(args.calls):
            va.verify_head_importance(q, k, seqlens, list(w.score_heads), score=score, scale=w.scale,
                                      scratch=scratch, workspace=ws)
        torch.cuda.synchronize()
        va.verify_attn_check_status(ws)
        print(json.dumps({"profile": "score", "calls": args.calls, "status": "ok"}))
        return 0
    case = DeviceCase(W.make_workload(args.profile, seed=0), va)
    for _ in range(args.calls):
        case.step()
    torch.cuda.synchronize()
    va.verify_attn_check_status(case.ws)
    print(json.dumps({"profile": args.profile, "calls": args.calls, "status": "ok"}))
    return 0


def dist_setup(n):
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return rank, world, local, dist
    torch.cuda.set_device(0)
    return 0, 1, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x, dist):
    """The slowest rank's value (NCCL reduces device tensors, gloo host ones)."""
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, seconds, dist):
    """Units every rank processed, over the slowest rank's time (weak scaling:
    each rank runs its own replica of the workload)."""
    world = dist.get_world_size() if dist is not None else 1
    return units_per_rank * world / max_over_ranks(seconds, dist)


def run_reference(args):
    """The oracle as the reference arm: bounded samples of the workload per step."""
    rank = int(os.environ.get("RANK", 0))
    if rank != 0:
        return 0
    w = W.make_workload(args.config, seed=0)
    secs = []
    cb = None
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(w, target_s=max(1.0, 30.0 / max(1, args.steps + args.warmup)), max_reps=4)
        if i >= args.warmup:
            secs.append(r["seconds"])
            cb = r
    line = {"impl": "reference", "metric": METRIC,
            "value": cb["value"], "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * sum(secs) / len(secs), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, None),
            "cpu_baseline": {"kind": "oracle", "cores": cb["cores"], "sample": cb["sample"], "value": cb["value"],
                             "unit": "GB/s"},
            "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def config_dict(w, n_copies):
    d = {"workload": f"{w.name}: B{w.B} T{w.T} Hq{w.Hq} Hkv{w.Hkv} d{w.D} {w.dtype} {w.layout}",
         "batch": w.B, "draft_tokens": w.T, "prefix_len": (int(w.seqlens.min()), int(w.seqlens.max())),
         "kv_bytes_per_step": w.kv_bytes()}
    if n_copies is not None:
        d["l2"] = f"inputs rotated over {n_copies} resident copies ({n_copies} x {w.kv_bytes() / 1e6:.0f} MB read) > L2"
    return d


def nvtx(name):
    """An NVTX range around a bench phase (visible in a profiler timeline)."""
    class _R:
        def __enter__(self):
            torch.cuda.nvtx.range_push(name)

        def __exit__(self, *a):
            torch.cuda.nvtx.range_pop()
    return _R()


def replay_timed(graph, reps, rank, dist, sample_clocks):
    """CUDA-event seconds of ``reps`` graph replays on the current stream,
    bracketed by barrier + synchronize; optionally with the SM clocks sampled."""
    clocks = ClockSampler(torch.cuda.current_device()) if (sample_clocks and rank == 0) else None
    if clocks:
        time.sleep(0.1)
    barrier(dist)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(dist)
    clk = clocks.stop() if clocks else None
    return e0.elapsed_time(e1) * 1e-3, clk


class AttentionOnly:
    """The attention call of a sparse step alone (the verify sets built once
    beforehand), to time the dominant kernel without the index build."""

    def __init__(self, case):
        self.case = case
        case.va.verify_build_index(case.seqlens, case.sd, case.st, case.w.n_sink, case.w.window, case.w.m_draft,
                                   case.w.budget, indices=case.idx, n_indices=case.nidx, workspace=case.ws)

    def step(self):
        c, w = self.case, self.case.w
        c.va.verify_attn_sparse(c.q, c.k, c.v, c.seqlens, c.idx, c.nidx, tree_parent=c.parent, tree_mask=c.mask,
                                out=c.out, lse=c.lse, workspace=c.ws, scale=w.scale)


def measure_config(name, va, args, peak, peak_kind, want_e2e, want_cpu, rank, dist, cpu_s):
    """Everything reported for one workload: exactly K timed steps (after W
    warm-up steps), a sustained region of at least 0.6 s with clocks, the
    dominant kernel's roofline, per-call percentiles, e2e and the oracle."""
    w = W.make_workload(name, seed=0)
    world = dist.get_world_size() if dist is not None else 1
    n_copies = n_copies_for(w)
    cases = [DeviceCase(w, va) for _ in range(n_copies)]
    bytes_step = w.kv_bytes()
    kernel, launches = attention_path(w)
    res = {"w": w, "n_copies": n_copies, "kernel": kernel, "launches": launches}
    with nvtx(f"{name}: warm-up"):
        graph_steps = min(max(args.steps, 1), 64)
        graph, _ = time_graph_steps(cases, 0, 0, graph_steps)
        # W warm-up steps, then exactly K steps: graphs of `graph_steps` steps,
        # and a remainder graph for K not a multiple of it
        full, rem = divmod(args.steps, graph_steps)
        g_rem = time_graph_steps(cases, 0, 0, rem)[0] if rem else None
        g_w, _ = time_graph_steps(cases, 0, 0, 1)
        for _ in range(args.warmup):
            g_w.replay()
        torch.cuda.synchronize()
    with nvtx(f"{name}: timed K steps"):
        clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
        barrier(dist)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(full):
            graph.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record()
        torch.cuda.synchronize()
        barrier(dist)
        dt = e0.elapsed_time(e1) * 1e-3 / args.steps
    with nvtx(f"{name}: sustained"):
        reps = max(1, math.ceil(0.6 / max(dt * graph_steps, 1e-6)))
        sus_t, _ = replay_timed(graph, reps, rank, dist, sample_clocks=False)
        clk = clocks.stop() if clocks else None
    sus_dt = sus_t / (reps * graph_steps)
    for c in cases:
        va.verify_attn_check_status(c.ws)
    dt_max = max_over_ranks(dt, dist)
    sus_max = max_over_ranks(sus_dt, dist)
    res.update(dt=dt_max, gbs=whole_job_rate(bytes_step, dt, dist) / 1e9, tok_s=w.tokens() * world / dt_max,
               steps=args.steps, clocks=clk,
               sustained={"us_per_step": round(sus_max * 1e6, 3), "steps": reps * graph_steps,
                          "seconds": round(sus_t, 3), "GBps": round(bytes_step / sus_max / 1e9, 1),
                          "frac_of_measured_hbm": round(bytes_step / sus_max / 1e9 / peak, 4)})
    # the dominant kernel: the step itself when it is one launch; the sparse
    # attention timed alone; otherwise the whole call (its launches together)
    with nvtx(f"{name}: kernel"):
        if w.layout == "sparse":
            kcases = [AttentionOnly(c) for c in cases]
            kg, kreps = time_graph_steps(kcases, 64 * max(1, math.ceil(0.1 / max(sus_dt * 64, 1e-6))), 3, 64)
            kt, _ = replay_timed(kg, kreps, rank, dist, sample_clocks=False)
            kern_s, kern_from = kt / (kreps * 64), "attention calls alone, CUDA events over graph replays"
            del kg
        else:
            kern_s = dt_max
            kern_from = "timed region / steps" + ("" if launches == 1 else " (all launches of the call)")
    with nvtx(f"{name}: per-call"):
        durs = per_call_durations(cases, 200)
    call_pct = [float(x) for x in np.percentile(np.asarray(durs, dtype=np.float64), [10, 50, 90])]
    traffic = profiled_traffic(name)
    res["roofline"] = {"bound": "hbm", "achieved": round(bytes_step / kern_s / 1e9, 1), "peak": peak, "unit": "GB/s",
                       "frac": round(bytes_step / kern_s / 1e9 / peak, 4), "traffic": traffic,
                       "kernel": kernel, "kernel_us": round(kern_s * 1e6, 3), "kernel_us_from": kern_from,
                       "call_us": round(statistics.mean(durs) * 1e6, 3),
                       "call_us_p10_p50_p90": [round(x * 1e6, 3) for x in call_pct], "peak_kind": peak_kind}
    del graph, g_w, g_rem, cases
    torch.cuda.empty_cache()
    if want_e2e:
        with nvtx(f"{name}: e2e"):
            e_dt, h2d, d2h = e2e_measure(w, va, max(50, min(args.steps * 10, 400)))
        e_dt = max_over_ranks(e_dt, dist)
        res["e2e"] = {"value": round(bytes_step * world / e_dt / 1e9, 2), "unit": "GB/s",
                      "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                      "ms_per_step": round(e_dt * 1e3, 4)}
        torch.cuda.empty_cache()
    if want_cpu and rank == 0:
        with nvtx(f"{name}: oracle on the host"):
            res["cpu"] = cpu_baseline(w, target_s=cpu_s)
    return res


def config_entry(r, world, peak):
    """The other_configs entry of one measured workload."""
    d = {"workload": config_dict(r["w"], r["n_copies"])["workload"],
         "GBps": round(r["gbs"] / world, 1), "frac_of_measured_hbm": round(r["gbs"] / world / peak, 4),
         "us_per_step": round(r["dt"] * 1e6, 3), "steps": r["steps"], "tokens_per_s": round(r["tok_s"] / world, 1),
         "kv_bytes_per_step": r["w"].kv_bytes(), "gpu_launches_per_step": r["launches"],
         "roofline": r["roofline"], "sustained": r["sustained"], "clocks": r["clocks"]}
    if "cpu" in r:
        d["cpu_baseline"] = r["cpu"]
    return d


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="tree", choices=list(W.CONFIG_NAMES))
    ap.add_argument("--only", action="store_true", help="measure the --config workload alone")
    ap.add_argument("--all-configs", action="store_true",
                    help="also the steps before and after verification (rotation, importance, acceptance, commit)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--profile", choices=list(W.CONFIG_NAMES) + ["after", "score", "rope"], default=None,
                    help="run --calls plain verification steps of one workload (for ncu) and exit; "
                         "'after': --calls acceptance + KV commit pairs at the paged shape; "
                         "'score': --calls importance passes at the sparse shape; "
                         "'rope': --calls draft-block rotations at the paged shape")
    ap.add_argument("--calls", type=int, default=4)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.steps < 1:
        args.steps = 1
    if args.impl == "reference":
        return run_reference(args)
    if args.profile is not None:
        return run_profile(args)

    rank, world, local, dist = dist_setup(args.gpus)
    import speculative_decoding_verification_masked_gb300 as va

    va.api.lib(build_if_missing=(rank == 0))
    barrier(dist)
    peak, peak_kind = load_peak_hbm()
    want_cpu = not args.no_cpu
    main_res = measure_config(args.config, va, args, peak, peak_kind, want_e2e=True, want_cpu=want_cpu, rank=rank,
                              dist=dist, cpu_s=12.0)
    others = {}
    if not args.only:
        for name in W.CONFIG_NAMES:
            if name == args.config:
                continue
            r = measure_config(name, va, args, peak, peak_kind, want_e2e=False, want_cpu=want_cpu, rank=rank,
                               dist=dist, cpu_s=5.0)
            others[name] = config_entry(r, world, peak)
    next_rows = measure_next_rows(va, peak) if args.all_configs and rank == 0 else None
    scoring = measure_scoring(va, peak) if args.all_configs and rank == 0 else None
    sparse_overhead = (measure_sparse_overhead(va, scoring["us_per_call"] if scoring else None)
                       if args.all_configs and rank == 0 else None)
    rope = measure_rope(va, peak) if args.all_configs and rank == 0 else None
    rope_fused = measure_rope_fused(va, peak) if args.all_configs and rank == 0 else None
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    w = main_res["w"]
    line = {
        "metric": METRIC,
        "value": round(main_res["gbs"], 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": main_res["steps"],
        "warmup": args.warmup,
        "ms_per_step": round(main_res["dt"] * 1e3, 5),
        "tokens_per_s": round(main_res["tok_s"], 1),
        "frac_of_hbm_peak": round(main_res["gbs"] / world / peak, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) q/k/v, seeded trees/page tables/scores)",
        "config": config_dict(w, main_res["n_copies"]),
        "roofline": main_res["roofline"],
        "sustained": main_res["sustained"],
        "e2e": main_res.get("e2e"),
        "gpu_launches": main_res["steps"] * main_res["launches"],
        "clocks": main_res["clocks"],
    }
    if "cpu" in main_res:
        line["cpu_baseline"] = main_res["cpu"]
    if others:
        line["other_configs"] = others
    if next_rows is not None:
        line["after_verification"] = next_rows
    if scoring is not None:
        line["scoring_pass"] = scoring
    if sparse_overhead is not None:
        line["sparse_vs_full_cache"] = sparse_overhead
    if rope is not None:
        line["rope_draft"] = rope
    if rope_fused is not None:
        line["rope_inside_attention"] = rope_fused
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
