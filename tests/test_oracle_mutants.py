"""The oracle's pins catch plausible mistakes.

Each case copies oracle/verify_oracle.c, plants one mistake (a dropped term, a
wrong sign, index or operand), builds the copy with gcc and checks that the pin
set used in test_oracle_pins.py rejects it, while the pristine source passes.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import twin
from tests.test_oracle_pins import _f64, _rand_case, _sdpa, _prefix_tree_split

SRC = os.path.join(os.path.dirname(oracle.__file__), "verify_oracle.c")

MUTANTS = {
    "gqa_mapping": ("const int kvh = h / group;", "const int kvh = h % Hkv;"),
    "dropped_scale": ("z[n] = scale * s;", "z[n] = s;"),
    "lse_without_max": ("const double l = zmax + log(sum);", "const double l = log(sum);"),
    "mask_ignored_in_pv": ("if (!vis[n]) continue;\n          const double p", "const double p"),
    "transposed_q_index": ("s += widen(q, q_dtype, ((size_t)i * Hq + h) * D + d)",
                           "s += widen(q, q_dtype, ((size_t)h * T + i) * D + d)"),
    "bf16_widening_shift": ("<< 16;", "<< 15;"),
    "merge_weight_sign": ("const double w = exp(lse_parts[(size_t)s * n_rows + r] - l);",
                          "const double w = exp(l - lse_parts[(size_t)s * n_rows + r]);"),
    "merge_drops_a_part": ("for (int s = 0; s < n_parts; ++s) {\n      const double w",
                           "for (int s = 1; s < n_parts; ++s) {\n      const double w"),
    "tree_excludes_self": ("int j = i;", "int j = parent[i];"),
    "tree_parent_only": ("j = parent[j];", "j = (j == i) ? parent[j] : -1;"),
}


def _pins_pass():
    """A compact run of the pins; False at the first disagreement."""
    try:
        for dtype in ("fp32", "bf16"):
            q, k, v, vis = _rand_case(1, T=5, Hq=4, Hkv=2, D=8, n=12, dtype=dtype)
            vis[:, 0] = True
            out, lse = oracle.masked_attention(q, k, v, vis, 0.35)
            tout, tlse = twin.attention(_f64(q).tolist(), _f64(k).tolist(), _f64(v).tolist(), vis.tolist(), 0.35)
            if not (np.allclose(out, tout, atol=1e-10) and np.allclose(lse, tlse, atol=1e-10)):
                return False
            ref, ref_lse = _sdpa(q, k, v, vis, 0.35)
            if not (np.allclose(out, ref, atol=1e-10) and np.allclose(lse, ref_lse, atol=1e-10)):
                return False
        # divide-and-aggregate exactness
        q, k, v, vis = _rand_case(2, T=4, Hq=2, Hkv=1, D=8, n=14)
        vis[:, :6] = True
        full = oracle.masked_attention(q, k, v, vis, 0.5)
        for cuts in ([0, 6, 14], [0, 3, 9, 14]):
            part = _prefix_tree_split(q, k, v, vis, 0.5, cuts)
            if not (np.allclose(part[0], full[0], atol=1e-10) and np.allclose(part[1], full[1], atol=1e-10)):
                return False
        # tree visibility against an independent ancestor walk
        rng = np.random.default_rng(0)
        for T in (5, 17):
            p = W.random_parents(T, rng)
            vis = oracle.tree_visibility(p)
            for i in range(T):
                if set(np.nonzero(vis[i])[0].tolist()) != twin.ancestors(p, i):
                    return False
        return True
    except Exception:
        return False


def _build_variant(tmp_path, name, edit):
    src = open(SRC).read()
    if edit is not None:
        old, new = edit
        assert src.count(old) >= 1, f"mutant {name}: pattern not found"
        src = src.replace(old, new, 1)
    c = tmp_path / f"{name}.c"
    c.write_text(src)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-std=c11", str(c), "-o", str(so), "-lm"],
                   check=True)
    return str(so)


def test_pristine_oracle_passes_the_pins(tmp_path):
    with oracle.swapped_library(_build_variant(tmp_path, "pristine", None)):
        assert _pins_pass()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    with oracle.swapped_library(_build_variant(tmp_path, name, MUTANTS[name])):
        assert not _pins_pass(), f"pins did not catch mutant {name}"


# ----------------------------------------------------------------------------
# the Python-side oracle functions (greedy acceptance, KV commit): the planted
# mistake is applied to the function's source and the function swapped in
# ----------------------------------------------------------------------------

PY_MUTANTS = {
    "accept_ignores_parent": ("greedy_accept", "up = p < 0 or accepted[p]", "up = True"),
    "accept_target_column": ("greedy_accept", "int(tgt[b, p + 1])", "int(tgt[b, p])"),
    "accept_ties_to_larger_end": ("greedy_accept", "depth[t] > depth[best]", "depth[t] >= depth[best]"),
    "accept_bonus_column": ("greedy_accept", "bonus[b] = tgt[b, best + 1]", "bonus[b] = tgt[b, best]"),
    "commit_no_move": ("commit_kv_dense", "src = [L + int(path[b][j]) for j in range(a)]",
                       "src = [L + j for j in range(a)]"),
    "commit_paged_row": ("commit_kv_paged", "return int(page_table[b][slot // page_size]), slot % page_size",
                         "return int(page_table[b][slot // page_size]), (slot + 1) % page_size"),
    "importance_gqa_mapping": ("head_importance", "k_cache[b, :L, h // group]", "k_cache[b, :L, h % Hkv]"),
    "importance_shifted_rows": ("head_importance", "k_cache[b, :L, h // group]", "k_cache[b, 1:L + 1, h // group]"),
    "importance_dropped_scale": ("head_importance", "z = scale * (qh @ kh.T)", "z = qh @ kh.T"),
    "importance_unnormalised": ("head_importance", "(e / e.sum(axis=1, keepdims=True))", "e"),
    "importance_normalised_over_tokens": ("head_importance", "e / e.sum(axis=1, keepdims=True)",
                                          "e / e.sum(axis=0, keepdims=True)"),
    "importance_max_over_tokens": ("head_importance", "z.max(axis=1, keepdims=True)", "z.max(axis=0, keepdims=True)"),
    "rope_sign": ("rope_rotate", "lo * c - hi * s", "lo * c + hi * s"),
    "rope_interleaved_pairs": ("rope_rotate", "lo, hi = x[..., :half], x[..., half:]",
                               "lo, hi = x[..., 0::2], x[..., 1::2]"),
    "rope_frequency_exponent": ("rope_rotate", "(-(2.0 * np.arange(half)) / D)", "(-(1.0 * np.arange(half)) / D)"),
    "rope_draft_slot": ("rope_draft_dense", "rope_rotate(k_cache[b, L:L + T], pos[b][:, None], base)",
                        "rope_rotate(k_cache[b, L + 1:L + T + 1], pos[b][:, None], base)"),
    "rope_paged_row": ("rope_draft_paged", "slot % page_size", "(slot + 1) % page_size"),
}


def _py_pins_pass():
    from tests import test_oracle_pins as pins
    try:
        pins.test_greedy_accept_hand()
        for seed in range(12):
            pins.test_greedy_accept_brute_force(seed)
        pins.test_greedy_accept_chain_is_prefix_match()
        pins.test_commit_kv_hand()
        pins.test_commit_kv_paged_equals_dense()
        pins.test_commit_kv_identity_and_untouched_rows()
        pins.test_head_importance_hand()
        for seed in range(2):
            pins.test_head_importance_matches_torch_softmax(seed)
        pins.test_head_importance_mass_and_equal_keys()
        pins.test_head_importance_follows_the_prefix_rows_only()
        pins.test_rope_hand()
        pins.test_rope_matches_complex_rotation(0)
        pins.test_rope_invariants()
        pins.test_rope_draft_rows_only()
        return True
    except (AssertionError, IndexError, ValueError):
        return False


def test_pristine_python_oracle_passes_the_pins():
    assert _py_pins_pass()


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_planted_python_mistake_is_caught(monkeypatch, name):
    import inspect
    import textwrap

    fn_name, old, new = PY_MUTANTS[name]
    src = inspect.getsource(getattr(oracle, fn_name))
    assert src.count(old) == 1, f"mutant {name}: pattern not found"
    ns = dict(vars(oracle))
    exec(textwrap.dedent(src.replace(old, new)), ns)
    monkeypatch.setattr(oracle, fn_name, ns[fn_name])
    assert not _py_pins_pass(), f"pins did not catch mutant {name}"
