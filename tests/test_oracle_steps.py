"""Pins of the oracle's step-level definitions: composed in the layer's order
they reproduce moe_forward and moe_backward, which are pinned independently
(closed forms, finite differences)."""
import numpy as np
import pytest

from oracle import moe_oracle as O


def _case(seed, T=40, H=8, E=6, k=2, F=4, S=0, score=O.SOFTMAX):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H))
    w1 = rng.standard_normal((E, 2 * F, H)) * 0.5
    w2 = rng.standard_normal((E, H, F)) * 0.5
    w1s = rng.standard_normal((2 * S, H)) * 0.5 if S else None
    w2s = rng.standard_normal((H, S)) * 0.5 if S else None
    dy = rng.standard_normal((T, H))
    return x, wr, w1, w2, w1s, w2s, dy


@pytest.mark.parametrize("score,S,pad", [(O.SOFTMAX, 0, 128), (O.SIGMOID, 4, 32), (O.SOFTMAX, 4, 1)])
def test_steps_compose_to_forward_and_backward(score, S, pad):
    x, wr, w1, w2, w1s, w2s, dy = _case(3, S=S, score=score)
    k = 2
    fwd = O.moe_forward(x, wr, w1, w2, k=k, score=score, w1_shared=w1s, w2_shared=w2s)
    bwd = O.moe_backward(x, wr, w1, w2, fwd, dy, score=score, w1_shared=w1s, w2_shared=w2s)
    idx, gate = fwd["topk_idx"], fwd["gates"]
    m = O.permutation_maps(idx, w1.shape[0], pad)
    po = m["poffsets"]
    row_gate = np.zeros(len(m["row_src"]))
    valid = m["row_src"] >= 0
    row_gate[valid] = gate[m["row_src"][valid], m["row_slot"][valid]]
    xp = O.permute(x, m)
    z, h = O.expert_fc1(xp, w1, po, row_gate)
    o = O.expert_fc2(h, w2, po)
    shared = None
    if S:
        zs, hs = O.expert_fc1(x, w1s[None], O.dense_rows_of(len(x)))
        shared = O.expert_fc2(hs, w2s[None], O.dense_rows_of(len(x)))
    y = O.unpermute_sum(o, m, shared)
    np.testing.assert_allclose(y, fwd["y"], rtol=1e-12, atol=1e-12)
    # backward
    dyp = O.permute(dy, m)
    dz, dg_rows = O.expert_dgrad_fc2(dyp, w2, z, po, row_gate)
    dxp = O.expert_dgrad_fc1(dz, w1, po)
    dgate = dg_rows[m["slot_row"]]
    np.testing.assert_allclose(dgate, bwd["dgate"], rtol=1e-11, atol=1e-12)
    dl = O.router_backward(fwd["logits"], idx, gate, dgate, score)
    dx = O.unpermute_sum(dxp, m) + dl @ wr
    if S:
        dzs, _ = O.expert_dgrad_fc2(dy, w2s[None], zs, O.dense_rows_of(len(x)))
        dx += O.expert_dgrad_fc1(dzs, w1s[None], O.dense_rows_of(len(x)))
        np.testing.assert_allclose(O.expert_wgrad(dzs, x, O.dense_rows_of(len(x)))[0], bwd["dW1_shared"],
                                   rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(O.expert_wgrad(dy, hs, O.dense_rows_of(len(x)))[0], bwd["dW2_shared"],
                                   rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dx, bwd["dx"], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(O.expert_wgrad(dz, xp, po), bwd["dW1"], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(O.expert_wgrad(dyp, h, po), bwd["dW2"], rtol=1e-11, atol=1e-11)
    # router weight gradient as a per-expert sum over the expert's rows
    row_dl = np.zeros(len(m["row_src"]))
    row_dl[valid] = dl[m["row_src"][valid], idx[m["row_src"][valid], m["row_slot"][valid]]]
    dwr = np.stack([(row_dl[a:b, None] * xp[a:b]).sum(0) for _, a, b in O._segments(po)])
    np.testing.assert_allclose(dwr, bwd["dWr"], rtol=1e-11, atol=1e-11)


def test_empty_expert_gets_zero_weight_gradient():
    rng = np.random.default_rng(0)
    po = np.array([0, 128, 128, 256])
    a = rng.standard_normal((256, 3))
    b = rng.standard_normal((256, 5))
    dw = O.expert_wgrad(a, b, po)
    assert np.all(dw[1] == 0)
    np.testing.assert_allclose(dw[0], a[:128].T @ b[:128])
