"""Pins of the oracle's router: top-k selection, keys and gates.

Each check compares the oracle with something other than itself: a selection
by repeated arg-max written as a pure-Python loop, exhaustive search over all
k-subsets, torch.topk / scipy's softmax (library routines), and closed forms.
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe_oracle as O


def _select_by_repeated_argmax(keys_row, k):
    """Textbook selection: k passes, each taking the largest remaining key,
    the lower id on ties."""
    chosen = []
    for _ in range(k):
        best = None
        for e, v in enumerate(keys_row):
            if e in chosen:
                continue
            if best is None or v > keys_row[best] or (v == keys_row[best] and e < best):
                best = e
        chosen.append(best)
    return chosen


@pytest.mark.parametrize("E,k", [(8, 2), (8, 1), (8, 8), (16, 4), (5, 3)])
def test_topk_matches_repeated_argmax_with_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    # a coarse grid makes many exact ties
    keys = rng.integers(-3, 4, size=(200, E)).astype(np.float64) * 0.5
    sel = O.topk_select(keys, k)
    for t in range(keys.shape[0]):
        assert list(sel[t]) == _select_by_repeated_argmax(list(keys[t]), k)


def test_topk_is_the_best_subset_tiny():
    """Exhaustive search over all C(8,2)=28 subsets (Tiny workload shape): the
    chosen set has the largest key sum; among equal sums the lexicographically
    smallest sorted id tuple wins when keys tie."""
    rng = np.random.default_rng(3)
    E, k = 8, 2
    keys = rng.integers(-4, 5, size=(300, E)).astype(np.float64)
    sel = O.topk_select(keys, k)
    for t in range(keys.shape[0]):
        best = None
        for sub in itertools.combinations(range(E), k):
            s = sum(keys[t, e] for e in sub)
            # among equal sums prefer the subset whose keys, sorted by (key desc, id asc),
            # come first; equivalently the subset picked by the tie rule
            order = tuple(sorted(sub, key=lambda e: (-keys[t, e], e)))
            cand = (s, tuple((-keys[t, e], e) for e in order))
            if best is None or cand[0] > best[0] or (cand[0] == best[0] and cand[1] < best[1]):
                best = cand
        want = [e for _, e in best[1]]
        assert list(sel[t]) == want


def test_topk_matches_torch_on_tie_free_inputs():
    rng = np.random.default_rng(7)
    keys = rng.standard_normal((500, 64))
    for k in (1, 2, 8):
        sel = O.topk_select(keys, k)
        tv, ti = torch.topk(torch.from_numpy(keys), k, dim=-1, largest=True, sorted=True)
        np.testing.assert_array_equal(sel, ti.numpy())


def test_softmax_gates_equal_renormalised_full_softmax():
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((64, 16)) * 2
    sel, g = O.route(logits, 4, O.SOFTMAX)
    full = scipy.special.softmax(logits, axis=-1)
    p = np.take_along_axis(full, sel.astype(np.int64), axis=-1)
    np.testing.assert_allclose(g, p / p.sum(-1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(g.sum(-1), 1.0, rtol=0, atol=1e-14)
    # order of gates follows the selection order (descending logit)
    assert np.all(np.diff(g, axis=-1) <= 1e-15)


def test_sigmoid_gates_closed_form():
    rng = np.random.default_rng(12)
    logits = rng.standard_normal((64, 16))
    bias = rng.standard_normal(16) * 0.1
    sel, g = O.route(logits, 3, O.SIGMOID, bias)
    np.testing.assert_allclose(g.sum(-1), 1.0, atol=1e-14)
    for t in range(4):
        s = [1.0 / (1.0 + math.exp(-logits[t, e])) for e in sel[t]]
        for i in range(3):
            assert abs(g[t, i] - s[i] / sum(s)) < 1e-14
    # the bias moves the selection: a large bias on expert 5 puts it in every set
    b2 = np.zeros(16)
    b2[5] = 10.0
    sel2, _ = O.route(logits, 3, O.SIGMOID, b2)
    assert np.all(sel2[:, 0] == 5)


def test_k1_gate_is_one():
    rng = np.random.default_rng(13)
    logits = rng.standard_normal((32, 8))
    for score in (O.SOFTMAX, O.SIGMOID):
        _, g = O.route(logits, 1, score, np.zeros(8))
        np.testing.assert_array_equal(g, np.ones((32, 1)))


def test_router_logits_against_python_dot():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((5, 7))
    w = rng.standard_normal((3, 7))
    lg = O.router_logits(x, w)
    for t in range(5):
        for e in range(3):
            assert abs(lg[t, e] - math.fsum(x[t, h] * w[e, h] for h in range(7))) < 1e-13


def test_selection_keys_f32_close_to_f64():
    rng = np.random.default_rng(15)
    l32 = (rng.standard_normal((100, 32)) * 3).astype(np.float32)
    b = (rng.standard_normal(32) * 0.1).astype(np.float32)
    k64 = O.selection_keys(l32.astype(np.float64), O.SIGMOID, b.astype(np.float64))
    k32 = O.selection_keys_f32(l32, O.SIGMOID, b)
    assert k32.dtype == np.float32
    np.testing.assert_allclose(k32, k64, atol=3e-7)
    np.testing.assert_array_equal(O.selection_keys_f32(l32, O.SOFTMAX), l32)


def test_topk_gap():
    keys = np.array([[3.0, 1.0, 2.0, 2.5]])
    # sorted: 3, 2.5, 2, 1 ; k=2: gap between 2nd and 3rd = 0.5, inner gap 0.5
    assert O.topk_gap(keys, 2)[0] == pytest.approx(0.5)
    assert O.topk_gap(keys, 1)[0] == pytest.approx(0.5)
    assert O.topk_gap(keys, 4)[0] == np.inf
