"""Pins of the oracle's permutation maps: invariants, a library stable sort,
and the unpermute(permute(x)) identities."""
import numpy as np
import pytest

from moe_expert_layer_05_gb300.inputs import random_topk_indices
from oracle import moe_oracle as O


CASES = [
    # T, E, k, skew
    (256, 8, 2, 0.0),
    (300, 16, 4, 1.5),     # hot experts, some empty
    (64, 8, 8, 0.0),       # k == E: every token visits every expert
    (1, 8, 2, 0.0),
    (0, 8, 2, 0.0),
    (129, 4, 1, 3.0),
]


@pytest.mark.parametrize("T,E,k,skew", CASES)
@pytest.mark.parametrize("pad", [1, 32, 128])
def test_maps_invariants(T, E, k, skew, pad):
    idx = random_topk_indices(T, E, k, seed=T + E, skew=skew)
    m = O.permutation_maps(idx, E, pad)
    counts, offsets, poffsets = m["counts"], m["offsets"], m["poffsets"]
    assert counts.sum() == T * k
    assert offsets[0] == 0 and np.all(np.diff(offsets) == counts)
    seg = np.diff(poffsets)
    assert np.all(seg % pad == 0) and np.all(seg >= counts) and np.all(seg - counts < pad)
    # every (t,i) has its own row; rows map back
    rows = m["slot_row"].ravel()
    assert len(np.unique(rows)) == rows.size
    for t in range(T):
        for i in range(k):
            r = m["slot_row"][t, i]
            assert m["row_src"][r] == t and m["row_slot"][r] == i
            e = idx[t, i]
            assert poffsets[e] <= r < poffsets[e] + counts[e]
    # each token appears exactly k times
    src = m["row_src"]
    assert np.all(np.bincount(src[src >= 0], minlength=T) == k)
    assert (src < 0).sum() == poffsets[-1] - T * k


@pytest.mark.parametrize("T,E,k,skew", CASES)
def test_order_equals_library_stable_sort(T, E, k, skew):
    """Compact order = Python's stable sorted() of pairs keyed by expert id,
    pairs enumerated in token order."""
    idx = random_topk_indices(T, E, k, seed=T * 3 + E, skew=skew)
    m = O.permutation_maps(idx, E, 1)
    pairs = [(t, i) for t in range(T) for i in range(k)]
    order = sorted(pairs, key=lambda p: idx[p[0], p[1]])
    compact = O.compact_rows(m)
    for pos, (t, i) in enumerate(order):
        assert compact[t, i] == pos
    # with pad=1 compact and padded layouts coincide
    np.testing.assert_array_equal(compact, m["slot_row"])


def test_unpermute_of_permute():
    rng = np.random.default_rng(0)
    T, E, H = 50, 8, 6
    x = rng.standard_normal((T, H))
    for k in (1, 2, 4):
        idx = random_topk_indices(T, E, k, seed=k)
        m = O.permutation_maps(idx, E, 32)
        xp = O.permute(x, m)
        assert np.all(xp[m["row_src"] < 0] == 0)
        y = O.unpermute_sum(xp, m)
        np.testing.assert_array_equal(y, k * x)
        sh = rng.standard_normal((T, H))
        np.testing.assert_allclose(O.unpermute_sum(xp, m, sh), k * x + sh, rtol=0, atol=1e-15)


def test_bad_index_rejected():
    with pytest.raises(ValueError):
        O.permutation_maps(np.array([[0, 9]]), 8)
