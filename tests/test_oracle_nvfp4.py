"""Pins of the oracle's NVFP4 quantiser and layer: the E2M1 code points the
OCP MX specification lists (tests/golden/e2m1_points.txt), round-to-nearest-
even against a brute-force nearest search over the grid, the per-element
error bound the block scale implies, invariance under power-of-two scaling,
lossless blocks, and the layer with identity quantiser and storage equal to
the unquantised layer."""
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_points.txt")
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def test_golden_points():
    n = 0
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            val, code = line.split()
            v, c = float(val), int(code, 16)
            assert O.e2m1_encode(np.array([v]))[0] == c, line
            assert O.e2m1_decode(np.array([c]))[0] == v, line
            n += 1
    assert n >= 8


def test_decode_encode_roundtrip_all_codes():
    codes = np.arange(16, dtype=np.uint8)
    np.testing.assert_array_equal(O.e2m1_encode(O.e2m1_decode(codes)), codes)
    assert sorted(set(np.abs(O.e2m1_decode(codes)))) == list(GRID)


def _brute_nearest_even(a):
    """Nearest grid magnitude by exhaustive search; ties to the even code
    (the pattern with mantissa bit 0, i.e. even index in GRID)."""
    out = np.empty_like(a)
    for i, v in enumerate(np.minimum(a, 6.0)):
        d = np.abs(GRID - v)
        best = np.flatnonzero(d == d.min())
        out[i] = GRID[best[0]] if len(best) == 1 else GRID[[b for b in best if b % 2 == 0][0]]
    return out


def test_encode_is_nearest_even_by_brute_force():
    mids = (GRID[:-1] + GRID[1:]) / 2
    rng = np.random.default_rng(3)
    a = np.concatenate([GRID, mids, np.nextafter(mids, 0), np.nextafter(mids, 10), rng.uniform(0, 8, 4000)])
    got = O.e2m1_decode(O.e2m1_encode(a))
    np.testing.assert_array_equal(got, _brute_nearest_even(a))
    neg = O.e2m1_encode(-a[a > 0])
    assert np.all(neg & 0x8) and np.array_equal(O.e2m1_decode(neg), -_brute_nearest_even(a[a > 0]))


def _f32_bf16(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return O.bf16_round(rng.standard_normal(shape) * scale)


def test_error_bound_per_element():
    """|v - dq(v)| <= half an E2M1 step of v*S/s, times s/S; where the scale
    rounded down, values past 6 saturate and the error is their excess over 6
    (at most 6/16 for a normal E4M3 scale, which is within 1/16 relative; the
    rows scaled far down get subnormal scales)."""
    v = _f32_bf16((32, 256), 5) * np.exp2(np.random.default_rng(6).integers(-8, 8, size=(32, 1)))
    c, s, S = O.nvfp4_quantize(v)
    dq = O.nvfp4_dequantize(c, s, S)
    sv = np.repeat(O.e4m3_decode(s), 16, axis=-1)
    u = np.abs(v) * S / np.where(sv > 0, sv, 1)
    half = np.where(u < 2, 0.25, np.where(u < 4, 0.5, 1.0))
    bound = np.where(u <= 6.0, half, u - 6.0 + 1e-12) * sv / S
    assert np.all(np.abs(v - dq) <= bound * (1 + 1e-6) + 1e-30)
    normal = sv >= 2.0 ** -6                         # E4M3 normal scales: within 1/16 relative
    assert normal.any() and (~normal).any()
    assert np.all(u[normal] <= 6.0 * (1 + 1 / 16) + 1e-6)


def test_block_with_the_tensor_amax_gets_the_top_scale():
    v = _f32_bf16((8, 64), 7)
    c, s, S = O.nvfp4_quantize(v)
    i, j = np.unravel_index(np.argmax(np.abs(v)), v.shape)
    assert s[i, j // 16] == 0x7E                  # E4M3 448
    assert O.e2m1_decode(c[i, j]) == np.sign(v[i, j]) * 6.0
    assert np.float32(S) == np.float32(2688.0) / np.float32(np.abs(v).max())


def test_power_of_two_scaling_changes_no_code():
    v = _f32_bf16((16, 128), 8)
    c0, s0, S0 = O.nvfp4_quantize(v)
    for j in (-20, -3, 5, 30):
        c, s, S = O.nvfp4_quantize(v * 2.0 ** j)
        np.testing.assert_array_equal(c, c0)
        np.testing.assert_array_equal(s, s0)
        assert S == np.float32(S0 * 2.0 ** -j)


def test_representable_blocks_are_lossless_and_zero_tensor():
    """Blocks of grid values times amax_b / 6 with amax_b in {6, 3, 1.5, 0.75}
    and a tensor amax of 6 (S = 448): every block scale and code is exact."""
    rng = np.random.default_rng(9)
    v = rng.choice(np.concatenate([GRID, -GRID]), size=(4, 64))
    for b in range(4):
        v[:, 16 * b] = 6.0                          # every block reaches 6 before scaling
        v[:, 16 * b:16 * b + 16] *= 2.0 ** -b
    v[0, 0] = 6.0
    np.testing.assert_array_equal(O.nvfp4_roundtrip(v), v)
    c, s, S = O.nvfp4_quantize(np.zeros((2, 32)))
    assert S == 1.0 and not c.any() and not s.any()
    np.testing.assert_array_equal(O.nvfp4_roundtrip(np.zeros((2, 32))), 0.0)


def test_axis_and_explicit_amax():
    v = _f32_bf16((64, 32), 10)
    a = O.nvfp4_roundtrip(v, axis=0)
    b = O.nvfp4_roundtrip(v.T, axis=-1).T
    np.testing.assert_array_equal(a, b)
    # a larger tensor amax than the data's own: the scale follows the given amax
    c1, s1, S1 = O.nvfp4_quantize(v, amax=2 * np.abs(v).max())
    assert S1 == np.float32(2688.0) / np.float32(2 * np.abs(v).max())


def _case(seed, T=64, H=64, E=4, k=2, F=64, S=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) * 0.2
    w1 = rng.standard_normal((E, 2 * F, H)) * 0.1
    w2 = rng.standard_normal((E, H, F)) * 0.1
    w1s = rng.standard_normal((2 * S, H)) * 0.1 if S else None
    w2s = rng.standard_normal((H, S)) * 0.1 if S else None
    return x, wr, w1, w2, w1s, w2s


@pytest.mark.parametrize("score,S", [(O.SOFTMAX, 0), (O.SIGMOID, 64)])
def test_identity_quantiser_gives_the_unquantised_layer(score, S):
    x, wr, w1, w2, w1s, w2s = _case(1, S=S)
    kw = dict(w1_shared=w1s, w2_shared=w2s)
    ref = O.moe_forward(x, wr, w1, w2, k=2, score=score, **kw)
    got = O.moe_forward_nvfp4(x, wr, w1, w2, k=2, score=score, quant=lambda v, a, ax: np.asarray(v, np.float64),
                              store=lambda v: v, **kw)
    np.testing.assert_allclose(got["y"], ref["y"], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(got["topk_idx"], ref["topk_idx"])


def test_quantised_layer_deviation_matches_the_format():
    """E2M1 keeps one mantissa bit: each quantised operand carries ~8-10 % rms
    relative error, so two quantised GEMMs land 5-30 % from the unquantised
    layer, several times the MXFP8 deviation."""
    x, wr, w1, w2, _, _ = _case(2, T=256, H=256, F=128)
    ref = O.moe_forward(x, wr, w1, w2, k=2)
    got = O.moe_forward_nvfp4(x, wr, w1, w2, k=2)
    mx = O.moe_forward_mx(x, wr, w1, w2, k=2)
    r = np.linalg.norm(got["y"] - ref["y"]) / np.linalg.norm(ref["y"])
    rmx = np.linalg.norm(mx["y"] - ref["y"]) / np.linalg.norm(ref["y"])
    assert 0.05 < r < 0.3 and r > 2 * rmx


def test_h_scale_is_shared_by_all_experts():
    """The h' quantiser calls (one per expert with rows) all get the same
    tensor amax, the largest |h'| over every expert's rows; each weight is
    quantised with the amax of the whole tensor (all experts), x with its own."""
    x, wr, w1, w2, _, _ = _case(4, T=128, H=128, F=64)
    calls = []

    def rec(v, amax, axis):
        calls.append((np.array(v), amax))
        return O.nvfp4_roundtrip(v, amax, axis)

    O.moe_forward_nvfp4(x, wr, w1, w2, k=2, quant=rec)
    used = sorted({int(e) for e in O.route(O.router_logits(x, wr), 2, O.SOFTMAX)[0].ravel()})

    def is_expert_of(v, W):
        return any(v.shape == W[e].shape and np.array_equal(v, W[e]) for e in range(W.shape[0]))

    w1_calls = [a for v, a in calls if is_expert_of(v, w1)]
    w2_calls = [a for v, a in calls if is_expert_of(v, w2)]
    x_calls = [a for v, a in calls if v.shape == x.shape and np.array_equal(v, x)]
    h_calls = [(v, a) for v, a in calls if not (is_expert_of(v, w1) or is_expert_of(v, w2) or
                                                (v.shape == x.shape and np.array_equal(v, x)))]
    assert len(w1_calls) == len(w2_calls) == len(h_calls) == len(used)
    assert set(w1_calls) == {float(np.abs(w1).astype(np.float32).max())}
    assert set(w2_calls) == {float(np.abs(w2).astype(np.float32).max())}
    assert x_calls == [None]
    amaxes = {float(a) for _, a in h_calls}
    assert len(amaxes) == 1
    assert amaxes.pop() == max(np.abs(v).max() for v, _ in h_calls)


def test_sampled_tokens_with_full_tensor_amaxes_match_the_full_forward():
    """Rows of a token sample, given the full tensors' amaxes of x and h',
    equal those rows of the forward over all tokens (everything else is
    row-local) -- the form the full-size GPU test uses."""
    x, wr, w1, w2, _, _ = _case(6, T=96, H=64, F=64)
    full = O.moe_forward_nvfp4(x, wr, w1, w2, k=2)
    h_amaxes = set()

    def rec(v, amax, axis):
        v = np.asarray(v)
        weight = any(v.shape == W[e].shape and np.array_equal(v, W[e]) for W in (w1, w2) for e in range(4))
        if amax is not None and not weight:
            h_amaxes.add(float(amax))                   # h' calls: the shared tensor amax
        return O.nvfp4_roundtrip(v, amax, axis)

    O.moe_forward_nvfp4(x, wr, w1, w2, k=2, quant=rec)
    assert len(h_amaxes) == 1
    h_amax = h_amaxes.pop()
    tokens = np.array([3, 17, 40, 41, 95])
    part = O.moe_forward_nvfp4(x[tokens], wr, w1, w2, k=2, x_amax=np.abs(x).max(), h_amax=h_amax)
    # equal up to the fp64 summation order of the matmuls (a code flip would be ~1e-2)
    np.testing.assert_allclose(part["y"], full["y"][tokens], rtol=1e-12, atol=1e-13)
    wrong = O.moe_forward_nvfp4(x[tokens], wr, w1, w2, k=2)  # the sample's own amaxes: other codes
    assert np.abs(wrong["y"] - full["y"][tokens]).max() > 1e-4


def test_bf16_round_matches_torch_cast():
    """The oracle's bf16 storage rounding equals torch's round-to-nearest-even
    cast (a library routine), ties included."""
    import torch
    rng = np.random.default_rng(12)
    v = np.concatenate([rng.standard_normal(100000) * np.exp2(rng.integers(-30, 30, 100000)),
                        1.0 + np.arange(-64, 64) * 2.0 ** -8,          # exact ties between bf16 neighbours
                        [0.0, -0.0, 65504.0, -3.0e38]])
    want = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.bf16_round(v), want)
