"""Pins of the oracle's MXFP8 layer: with the quantiser replaced by the
identity it is exactly the unquantised layer (pinned by closed forms and finite
differences); with the real quantiser each GEMM sees MX-representable
operands, and the deviation from the unquantised layer stays at the size the
format predicts; and every GEMM of the recipe, forward and backward, equals the
MX block-scaled dot product taken along that GEMM's contraction axis (which
pins the axis each operand is quantised along)."""
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


# ------------------------------------------------------------------ the quantisation axes
def _mx_dot(A, B):
    """C = A B^T as an MX block-scaled GEMM: both operands quantised in blocks
    of 32 along their shared (contraction) axis, each block contributing
    X_A X_B sum_i P_A,i P_B,i (the OCP MX v1.0 dot product of two MX vectors:
    scales multiply once per block pair, elements are the decoded E4M3 codes).
    The contraction axis is zero-padded to whole blocks.  A [M,K], B [N,K]."""
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    K = A.shape[1]
    pad = (-K) % O.MX_BLOCK
    A = np.concatenate([A, np.zeros((A.shape[0], pad))], axis=1)
    B = np.concatenate([B, np.zeros((B.shape[0], pad))], axis=1)
    qa, sa = O.mxfp8_quantize(A, axis=-1)
    qb, sb = O.mxfp8_quantize(B, axis=-1)
    pa, pb = O.e4m3_decode(qa), O.e4m3_decode(qb)
    out = np.zeros((A.shape[0], B.shape[0]))
    for j in range(A.shape[1] // O.MX_BLOCK):
        cols = slice(j * O.MX_BLOCK, (j + 1) * O.MX_BLOCK)
        xa = np.exp2(sa[:, j].astype(np.float64) - 127.0)
        xb = np.exp2(sb[:, j].astype(np.float64) - 127.0)
        out += (xa[:, None] * xb[None, :]) * (pa[:, cols] @ pb[:, cols].T)
    return out


def _skewed(rng, shape, std):
    """Gaussian values whose magnitude varies by powers of two along both axes,
    so blocks taken along rows and along columns get different scales."""
    r = np.exp2(rng.integers(-3, 4, size=shape[0]))[:, None]
    c = np.exp2(rng.integers(-3, 4, size=shape[1]))[None, :]
    return rng.standard_normal(shape) * std * r * c


@pytest.mark.parametrize("score", [O.SOFTMAX, O.SIGMOID])
def test_mx_recipe_equals_block_scaled_gemms_on_contraction_axes(score):
    """The MXFP8 layer, forward and backward, recomputed GEMM by GEMM as block
    scaled dot products whose blocks run along each GEMM's contraction axis:
    fc1 over H, fc2 over F, the fc2 data gradient over H, the fc1 data
    gradient over 2F, the weight gradients over the expert's tokens.  E = 2 and
    k = 2 route every token to both experts (rows in ascending token order), so
    the gates are not 1 and enter fc2's operand before it is quantised; a
    shared expert rides along.  Dimensions all differ (T=72 pads to three token
    blocks, H=64, F=96, 2F=192, S=160), so a block taken along any other axis
    changes the result."""
    rng = np.random.default_rng(11)
    T, H, E, k, F, S = 72, 64, 2, 2, 96, 160
    x = _skewed(rng, (T, H), 1.0)
    wr = rng.standard_normal((E, H)) * 0.05
    w1 = np.stack([_skewed(rng, (2 * F, H), 0.1) for _ in range(E)])
    w2 = np.stack([_skewed(rng, (H, F), 0.1) for _ in range(E)])
    w1s = _skewed(rng, (2 * S, H), 0.1)
    w2s = _skewed(rng, (H, S), 0.1)
    dy = _skewed(rng, (T, H), 1.0)
    kw = dict(w1_shared=w1s, w2_shared=w2s)
    fwd = O.moe_forward_mx(x, wr, w1, w2, k=k, score=score, **kw)
    bwd = O.moe_backward_mx(x, wr, w1, w2, fwd, dy, score=score, **kw)

    idx, gate = fwd["topk_idx"], fwd["gates"]
    assert sorted(idx[0]) == [0, 1]
    y = np.zeros((T, H))
    dx = np.zeros((T, H))
    dgate = np.zeros((T, k))
    for e in range(E):
        slot = np.nonzero(idx == e)[1]                      # one slot per token, tokens ascending
        g = gate[np.arange(T), slot][:, None]
        z = _mx_dot(x, w1[e])                               # contraction over H
        a, b = z[:, :F], z[:, F:]
        hp = g * O.silu(a) * b
        y += _mx_dot(hp, w2[e])                             # over F
        dhp = _mx_dot(dy, w2[e].T)                          # over H
        dgate[np.arange(T), slot] = (dhp * O.silu(a) * b).sum(axis=1)
        dz = np.concatenate([g * dhp * b * O.silu_grad(a), g * dhp * O.silu(a)], axis=1)
        dx += _mx_dot(dz, w1[e].T)                          # over 2F
        np.testing.assert_allclose(bwd["dW1"][e], _mx_dot(dz.T, x.T), rtol=1e-9, atol=1e-12)   # over tokens
        np.testing.assert_allclose(bwd["dW2"][e], _mx_dot(dy.T, hp.T), rtol=1e-9, atol=1e-12)
    zs = _mx_dot(x, w1s)
    a, b = zs[:, :S], zs[:, S:]
    hs = O.silu(a) * b
    y += _mx_dot(hs, w2s)
    dhs = _mx_dot(dy, w2s.T)
    dzs = np.concatenate([dhs * b * O.silu_grad(a), dhs * O.silu(a)], axis=1)
    dx += _mx_dot(dzs, w1s.T)
    np.testing.assert_allclose(bwd["dW1_shared"], _mx_dot(dzs.T, x.T), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(bwd["dW2_shared"], _mx_dot(dy.T, hs.T), rtol=1e-9, atol=1e-12)
    # the router stays unquantised: its term is the plain chain rule through the gates
    dl = O.router_backward(fwd["logits"], idx, gate, dgate, score)
    dx += dl @ wr
    np.testing.assert_allclose(fwd["y"], y, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(bwd["dgate"], dgate, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(bwd["dx"], dx, rtol=1e-9, atol=1e-12)
    # and the quantisation is not a no-op here: the unquantised layer is several percent away
    plain = O.moe_forward(x, wr, w1, w2, k=k, score=score, **kw)
    assert np.linalg.norm(plain["y"] - y) > 1e-3 * np.linalg.norm(y)


@pytest.mark.parametrize("mx", [False, True])
def test_backward_without_weight_grads_changes_nothing_else(mx):
    """weight_grads=False only leaves outputs out: dx, dgate and dlogits are
    bit-identical to the full backward's."""
    x, wr, w1, w2, w1s, w2s, dy = _case(5, S=64)
    kw = dict(w1_shared=w1s, w2_shared=w2s)
    fwd_fn, bwd_fn = (O.moe_forward_mx, O.moe_backward_mx) if mx else (O.moe_forward, O.moe_backward)
    fwd = fwd_fn(x, wr, w1, w2, k=2, score=O.SIGMOID, **kw)
    full = bwd_fn(x, wr, w1, w2, fwd, dy, score=O.SIGMOID, **kw)
    part = bwd_fn(x, wr, w1, w2, fwd, dy, score=O.SIGMOID, weight_grads=False, **kw)
    for n in ("dx", "dgate", "dlogits"):
        np.testing.assert_array_equal(part[n], full[n])
    assert not {"dW1", "dW2", "dWr", "dW1_shared", "dW2_shared"} & set(part)
