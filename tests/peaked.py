"""Attention-sink inputs for the GPU parity tests: a few keys of every
(sequence, kv-head) -- key 0 among them -- score 8 to 12 above the rest for
every query row, and their values are large multiples of one shared vector,
weighted so that they cancel in the exact output.

Why this shape.  The online softmax turns each score into a weight P that the
PV product multiplies; rounded to bf16, a weight keeps only 8 significant bits
(up to 2^-8 of itself).  With the weight spread over thousands of keys those
errors average out, but when a handful of keys carry the row, each of their
weights moves the output by up to 2^-8 x weight x |v|.  Here |v| is up to 8 and
the sinks carry ~95% of the weight, so a kernel that multiplies a single bf16 P
misses the exact result by ~1e-2, while |out| itself stays far below 0.5 -- so
the bf16 rounding of the output (half an ulp, < 1e-3 there) leaves the 2e-3 bar
meaningful without any allowance.

Construction (all values exactly representable in bf16):
  * element 0 of every query row of the kv-head's group is set to 4.0;
  * a sink key row is zero except element 0 = kappa_j and element 1 =
    t_j = (j - (n-1)/2) / (2(n-1)), a tilt in [-1/4, 1/4], so its score is
    scale * (4 kappa_j + q_1 t_j):
    the same base for every row, and a small row-dependent tilt (q_1 is the
    row's own N(0, 1) element) that moves the sinks' weight ratios by a few
    percent from row to row -- enough that each row rounds its weights
    differently, little enough that the values still cancel;
  * the sink values are bf16(c_j * r) for one vector r in U(-1, 1)^D, with
    c_0 .. c_{n-2} from a fixed signed pattern and c_{n-1} chosen so that
    sum_j exp(z_j) c_j = 0 for the realised sink scores z_j.
The other keys and values stay N(0, 1) draws.  This module only shapes inputs;
the expected results come from the oracle.
"""
import numpy as np
import torch

BETA = 4.0
C_PATTERN = (8.0, -7.0, 7.5, -8.0, 6.5, -6.0, 7.0)


def _bf16(x):
    return float(torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).float())


def sink_scores(w, n_sinks):
    """The realised sink scores z_j = scale * BETA * kappa_j (natural-log units):
    spread over [10, 11] for the first n-1 sinks, the last one at 11.3, so that
    every sink carries a sizeable share of the weight."""
    targets = list(np.linspace(10.0, 11.0, n_sinks - 1)) + [11.3]
    unit = w.scale * BETA
    kappas = [_bf16(t / unit) for t in targets]
    return kappas, [unit * k for k in kappas]


def _slot_row(w, b, slot):
    """The cache row (k, v views over [Hkv][D]) of logical slot `slot` of sequence b."""
    if w.layout == "paged":
        page = int(w.page_table[b, slot // w.page_size])
        return w.k_pages[page, slot % w.page_size], w.v_pages[page, slot % w.page_size]
    return w.k_cache[b, slot], w.v_cache[b, slot]


def make_peaked(w, n_sinks=5, seed=0):
    """Reshape workload ``w`` in place into the attention-sink form above.

    Returns {(b, h): [sink positions]} (prefix positions, key 0 first).  For a
    sparse workload the sink positions get a target score above every other,
    so the oracle's verify set (handed to the library) holds them all."""
    rng = np.random.default_rng(seed)
    kappas, z = sink_scores(w, n_sinks)
    e = np.exp(np.array(z) - max(z))
    c = [C_PATTERN[j % len(C_PATTERN)] for j in range(n_sinks - 1)]
    c.append(-float(np.dot(e[:-1], c)) / e[-1])
    group = w.Hq // w.Hkv
    dt = w.q.dtype
    w.q[..., 0] = BETA
    sinks = {}
    for b in range(w.B):
        L = int(w.seqlens[b])
        assert L >= 4 * n_sinks, "prefix too short for the sinks"
        for h in range(w.Hkv):
            others = rng.choice(np.arange(1, L), size=n_sinks - 1, replace=False)
            pos = [0] + sorted(int(x) for x in others)
            r = torch.from_numpy(rng.uniform(-1.0, 1.0, size=w.D).astype(np.float32))
            # which sink sits at key 0 is drawn too
            order = list(rng.permutation(n_sinks))
            for j, slot in zip(order, pos):
                k_row, v_row = _slot_row(w, b, slot)
                k_row[h] = 0
                k_row[h, 0] = kappas[j]
                k_row[h, 1] = (j - (n_sinks - 1) / 2) / (2 * max(n_sinks - 1, 1))
                v_row[h] = (c[j] * r).to(dt)
            sinks[(b, h)] = pos
            if w.layout == "sparse":
                w.score_target[b, h, pos] = 2.0  # U(0,1) elsewhere: the sinks are always selected
    del group
    return sinks
