"""Pins of the oracle's MXFP8 layer: with the quantiser replaced by the
identity it is exactly the unquantised layer (pinned by closed forms and finite
differences); with the real quantiser each GEMM sees MX-representable
operands, and the deviation from the unquantised layer stays at the size the
format predicts."""
import numpy as np
import pytest

from oracle import moe_oracle as O


def _case(seed, T=64, H=64, E=4, k=2, F=64, S=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) * 0.2
    w1 = rng.standard_normal((E, 2 * F, H)) * 0.1
    w2 = rng.standard_normal((E, H, F)) * 0.1
    w1s = rng.standard_normal((2 * S, H)) * 0.1 if S else None
    w2s = rng.standard_normal((H, S)) * 0.1 if S else None
    dy = rng.standard_normal((T, H))
    return x, wr, w1, w2, w1s, w2s, dy


def ident(v, axis):
    return np.asarray(v, np.float64)


@pytest.mark.parametrize("score,S", [(O.SOFTMAX, 0), (O.SIGMOID, 64)])
def test_identity_quantiser_gives_the_unquantised_layer(score, S):
    x, wr, w1, w2, w1s, w2s, dy = _case(1, S=S)
    kw = dict(w1_shared=w1s, w2_shared=w2s)
    ref = O.moe_forward(x, wr, w1, w2, k=2, score=score, **kw)
    got = O.moe_forward_mx(x, wr, w1, w2, k=2, score=score, quant=ident, **kw)
    np.testing.assert_allclose(got["y"], ref["y"], rtol=1e-12, atol=1e-12)
    rb = O.moe_backward(x, wr, w1, w2, ref, dy, score=score, **kw)
    gb = O.moe_backward_mx(x, wr, w1, w2, got, dy, score=score, quant=ident, **kw)
    for n in ["dx", "dW1", "dW2", "dgate", "dWr"] + (["dW1_shared", "dW2_shared"] if S else []):
        np.testing.assert_allclose(gb[n], rb[n], rtol=1e-11, atol=1e-11, err_msg=n)


def test_quantised_layer_deviation_matches_the_format():
    """E4M3 keeps 3 mantissa bits: each quantised operand carries ~2-3 % rms
    relative error, so a chain of two quantised GEMMs lands a few percent
    from the unquantised layer — not less than 1 %, not more than 15 %."""
    x, wr, w1, w2, _, _, dy = _case(2, T=256, H=256, F=128)
    ref = O.moe_forward(x, wr, w1, w2, k=2)
    got = O.moe_forward_mx(x, wr, w1, w2, k=2)
    r = np.linalg.norm(got["y"] - ref["y"]) / np.linalg.norm(ref["y"])
    assert 0.01 < r < 0.15


def test_quantised_operands_are_representable():
    calls = []

    def spy(v, axis):
        out = O.mxfp8_roundtrip(v, axis)
        # idempotent: an MX-representable tensor quantises to itself
        np.testing.assert_array_equal(O.mxfp8_roundtrip(out, axis), out)
        calls.append(axis)
        return out

    x, wr, w1, w2, _, _, dy = _case(3, T=64)
    fwd = O.moe_forward_mx(x, wr, w1, w2, k=2, quant=spy)
    O.moe_backward_mx(x, wr, w1, w2, fwd, dy, quant=spy)
    assert set(calls) == {-1, 0}


def test_weight_cache_changes_nothing():
    x, wr, w1, w2, w1s, w2s, dy = _case(4, S=64)
    kw = dict(w1_shared=w1s, w2_shared=w2s)
    cache = {}
    a = O.moe_forward_mx(x, wr, w1, w2, k=2, **kw)
    b = O.moe_forward_mx(x, wr, w1, w2, k=2, weight_cache=cache, **kw)
    c = O.moe_forward_mx(x, wr, w1, w2, k=2, weight_cache=cache, **kw)     # served from the cache
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["y"], c["y"])
    ga = O.moe_backward_mx(x, wr, w1, w2, a, dy, **kw)
    gb = O.moe_backward_mx(x, wr, w1, w2, a, dy, weight_cache=cache, **kw)
    for n in ("dx", "dW1", "dW2", "dW1_shared", "dW2_shared"):
        np.testing.assert_array_equal(ga[n], gb[n])
