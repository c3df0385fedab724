"""Pins of the oracle's layer forward and backward: closed forms, a pure-Python
dense SwiGLU, the identity expert, the gate association, and central finite
differences for every gradient."""
import math

import numpy as np
import pytest

from oracle import moe_oracle as O


def _py_swiglu(xrow, w1, w2):
    """Dense SwiGLU MLP with Python loops: z = W1 x; h = silu(z_gate)*z_up; W2 h."""
    F = len(w1) // 2
    H = len(xrow)
    z = [math.fsum(w1[j][c] * xrow[c] for c in range(H)) for j in range(2 * F)]
    h = [(z[j] / (1.0 + math.exp(-z[j]))) * z[F + j] for j in range(F)]
    return [math.fsum(w2[c][j] * h[j] for j in range(F)) for c in range(H)]


def _tiny(seed, T=6, H=8, E=4, F=4, S=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) * 0.5
    w1 = rng.standard_normal((E, 2 * F, H)) * 0.5
    w2 = rng.standard_normal((E, H, F)) * 0.5
    w1s = rng.standard_normal((2 * S, H)) * 0.5 if S else None
    w2s = rng.standard_normal((H, S)) * 0.5 if S else None
    return x, wr, w1, w2, w1s, w2s


def test_single_expert_is_dense_swiglu():
    x, wr, w1, w2, _, _ = _tiny(1, T=5, H=6, E=1, F=3)
    out = O.moe_forward(x, wr, w1, w2, k=1)
    assert np.all(out["topk_idx"] == 0) and np.all(out["gates"] == 1.0)
    for t in range(5):
        want = _py_swiglu(list(x[t]), w1[0].tolist(), w2[0].tolist())
        np.testing.assert_allclose(out["y"][t], want, rtol=1e-12, atol=1e-13)


def test_shared_expert_only_adds_dense_swiglu():
    x, wr, w1, w2, w1s, w2s = _tiny(2, S=5)
    a = O.moe_forward(x, wr, w1, w2, k=2)["y"]
    b = O.moe_forward(x, wr, w1, w2, k=2, w1_shared=w1s, w2_shared=w2s)["y"]
    for t in range(x.shape[0]):
        np.testing.assert_allclose(b[t] - a[t], _py_swiglu(list(x[t]), w1s.tolist(), w2s.tolist()),
                                   rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("score", [O.SOFTMAX, O.SIGMOID])
def test_identity_expert_reproduces_input(score):
    """With every expert replaced by the identity, y_t = sum_i g_i x_t = x_t
    because the normalised gates sum to one."""
    x, wr, w1, w2, _, _ = _tiny(3, T=20, E=8)
    out = O.moe_forward(x, wr, w1, w2, k=3, score=score, bias=np.linspace(-0.2, 0.2, 8),
                        expert_fn=lambda e, rows: rows)
    np.testing.assert_allclose(out["y"], x, rtol=1e-14, atol=1e-14)


def test_worked_example_closed_form():
    """T=1, H=2, E=2, k=1, F=1, softmax.  x = (1, 0).
    Router rows (2,0) and (1,0): logits (2,1) -> expert 0, gate 1.
    W1_0 = [[ln 3, 0], [2, 0]]: a = ln 3, b = 2; silu(ln 3) = ln 3 * 3/4.
    W2_0 = [[1], [-1]]: y = (1.5 ln 3, -1.5 ln 3)."""
    x = np.array([[1.0, 0.0]])
    wr = np.array([[2.0, 0.0], [1.0, 0.0]])
    w1 = np.array([[[math.log(3.0), 0.0], [2.0, 0.0]], [[5.0, 5.0], [5.0, 5.0]]])
    w2 = np.array([[[1.0], [-1.0]], [[7.0], [7.0]]])
    out = O.moe_forward(x, wr, w1, w2, k=1)
    v = 1.5 * math.log(3.0)
    np.testing.assert_allclose(out["y"][0], [v, -v], rtol=1e-15)
    # k=2: gates softmax(2,1) = (e/(e+1), 1/(e+1)); expert 1: a=b=5, h=5*5*sig(5)
    out2 = O.moe_forward(x, wr, w1, w2, k=2)
    g0 = math.e / (math.e + 1.0)
    h1 = 25.0 / (1.0 + math.exp(-5.0))
    np.testing.assert_allclose(out2["y"][0], [g0 * v + (1 - g0) * 7 * h1, -g0 * v + (1 - g0) * 7 * h1],
                               rtol=1e-14)


def test_gate_before_fc2_equals_gate_after():
    """The layer applies g to the SwiGLU output before fc2 (memory-efficient
    permutation); fc2 is linear, so g*W2 h = W2 (g h)."""
    x, wr, w1, w2, _, _ = _tiny(4, T=10, E=4)
    out = O.moe_forward(x, wr, w1, w2, k=2)
    idx, g = out["topk_idx"], out["gates"]
    F = w1.shape[1] // 2
    y2 = np.zeros_like(x)
    for t in range(10):
        for i in range(2):
            e = idx[t, i]
            z = w1[e] @ x[t]
            hp = g[t, i] * O.silu(z[:F]) * z[F:]
            y2[t] += w2[e] @ hp
    np.testing.assert_allclose(out["y"], y2, rtol=1e-12, atol=1e-13)


def _loss(x, wr, w1, w2, w1s, w2s, dy, k, score, bias, routing):
    y = O.moe_forward(x, wr, w1, w2, k=k, score=score, bias=bias, w1_shared=w1s, w2_shared=w2s)
    assert np.array_equal(y["topk_idx"], routing), "perturbation changed the routing"
    return float((dy * y["y"]).sum())


@pytest.mark.parametrize("score,S", [(O.SOFTMAX, 0), (O.SIGMOID, 3)])
def test_backward_matches_finite_differences(score, S):
    x, wr, w1, w2, w1s, w2s = _tiny(5, T=6, H=5, E=4, F=3, S=S)
    rng = np.random.default_rng(9)
    dy = rng.standard_normal(x.shape)
    bias = np.array([0.1, -0.05, 0.0, 0.2]) if score == O.SIGMOID else None
    k = 2
    fwd = O.moe_forward(x, wr, w1, w2, k=k, score=score, bias=bias, w1_shared=w1s, w2_shared=w2s)
    keys = O.selection_keys(fwd["logits"], score, bias)
    assert O.topk_gap(keys, k).min() > 1e-3     # routing is stable under eps perturbations
    g = O.moe_backward(x, wr, w1, w2, fwd, dy, score=score, w1_shared=w1s, w2_shared=w2s)
    routing = fwd["topk_idx"]
    eps = 1e-6
    params = {"x": x, "wr": wr, "w1": w1, "w2": w2}
    grads = {"x": g["dx"], "wr": g["dWr"], "w1": g["dW1"], "w2": g["dW2"]}
    if S:
        params.update({"w1s": w1s, "w2s": w2s})
        grads.update({"w1s": g["dW1_shared"], "w2s": g["dW2_shared"]})
    for name, p in params.items():
        num = np.zeros_like(p)
        it = np.nditer(p, flags=["multi_index"])
        for _ in it:
            ix = it.multi_index
            old = p[ix]
            p[ix] = old + eps
            lp = _loss(x, wr, w1, w2, w1s, w2s, dy, k, score, bias, routing)
            p[ix] = old - eps
            lm = _loss(x, wr, w1, w2, w1s, w2s, dy, k, score, bias, routing)
            p[ix] = old
            num[ix] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grads[name], num, rtol=1e-6, atol=1e-7, err_msg=name)


@pytest.mark.parametrize("score", [O.SOFTMAX, O.SIGMOID])
def test_gate_gradient_matches_finite_differences(score):
    """dgate: derivative of <dy, y> w.r.t. each gate value, routing fixed."""
    x, wr, w1, w2, _, _ = _tiny(6, T=4, H=5, E=4, F=3)
    dy = np.random.default_rng(1).standard_normal(x.shape)
    fwd = O.moe_forward(x, wr, w1, w2, k=2, score=score)
    g = O.moe_backward(x, wr, w1, w2, fwd, dy, score=score)
    eps = 1e-6
    for t in range(4):
        for i in range(2):
            gp = fwd["gates"].copy(); gp[t, i] += eps
            gm = fwd["gates"].copy(); gm[t, i] -= eps
            yp = O.moe_forward(x, None, w1, w2, 2, routing=(fwd["topk_idx"], gp))["y"]
            ym = O.moe_forward(x, None, w1, w2, 2, routing=(fwd["topk_idx"], gm))["y"]
            num = float((dy * (yp - ym)).sum()) / (2 * eps)
            assert abs(num - g["dgate"][t, i]) < 1e-6 * max(1.0, abs(num))


def test_router_backward_zero_outside_selection():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((10, 8))
    sel, g = O.route(logits, 2, O.SOFTMAX)
    dl = O.router_backward(logits, sel, g, rng.standard_normal((10, 2)), O.SOFTMAX)
    mask = np.zeros_like(dl, bool)
    np.put_along_axis(mask, sel.astype(np.int64), True, axis=-1)
    assert np.all(dl[~mask] == 0)
    # softmax Jacobian rows sum to zero: a uniform shift of the logits does not move the gates
    np.testing.assert_allclose(dl.sum(-1), 0.0, atol=1e-15)
