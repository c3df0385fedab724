"""GPU parity of each step of the layer, called through the C ABI, against the
fp64 oracle on the same seeded inputs.

Tolerances: integer and index outputs (top-k indices, counts, offsets, maps,
permuted rows) are bit-exact.  bf16 outputs of a fp32-accumulated GEMM or sum:
see gpu_helpers.assert_bf16_close.  fp32 outputs: bounds stated per test.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_bf16_close, f64, i64, rel_l2
from moe_expert_layer_05_gb300 import api
from moe_expert_layer_05_gb300.inputs import random_topk_indices, to_bf16
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape, dtype=np.float32) * np.float32(std)


def _ws(cfg):
    ws = torch.zeros(max(api.moe_workspace_bytes(cfg), 256), dtype=torch.uint8, device=DEV)
    api.moe_workspace_init(ws)
    return ws


def _status(ws):
    return api.moe_read_device_status(ws)


# ------------------------------------------------------------------ router
@pytest.mark.parametrize("T,H,E", [(256, 128, 8), (300, 512, 128), (1000, 1024, 256), (1, 128, 8),
                                   (129, 256, 16), (4096, 4096, 8)])
def test_router_logits(lib, T, H, E):
    x = to_bf16(_rand((T, H), 1))
    wr = to_bf16(_rand((E, H), 2, 0.02))
    cfg = api.make_config(T, H, E, min(2, E), 128)
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    idx = torch.empty((T, cfg.k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, cfg.k), dtype=torch.float32, device=DEV)
    ws = _ws(cfg)
    api.moe_router_topk(cfg, x.to(DEV), wr.to(DEV), None, logits, idx, gate, ws)
    torch.cuda.synchronize()
    assert _status(ws) == 0
    ref = O.router_logits(f64(x), f64(wr))
    scale = np.abs(f64(x)) @ np.abs(f64(wr)).T
    err = np.abs(f64(logits) - ref)
    # fp32 accumulation of H exact bf16 products: |err| <= 2^-12 * sum |x w|
    assert np.all(err <= 2.0 ** -12 * scale + 1e-6), float((err / (scale + 1e-30)).max())


def _tie_logits(T, E, seed, grid):
    v = _rand((T, E), seed, 2.0)
    if grid:
        v = np.round(v * 4) / 4          # many exact ties
    return v.astype(np.float32)


@pytest.mark.parametrize("score", ["softmax", "sigmoid"])
@pytest.mark.parametrize("T,E,k,grid", [(256, 8, 2, False), (256, 8, 2, True), (500, 128, 8, True),
                                        (333, 256, 8, False), (64, 8, 8, True), (100, 32, 1, True),
                                        (70, 64, 32, False)])
def test_topk_gating(lib, score, T, E, k, grid):
    lg = _tie_logits(T, E, T + E + k, grid)
    bias = (_rand((E,), 5, 0.05) if score == "sigmoid" else None)
    cfg = api.make_config(T, 128, E, k, 128, score=score)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    api.moe_topk_gating(cfg, torch.from_numpy(lg).to(DEV),
                        None if bias is None else torch.from_numpy(bias).to(DEV), idx, gate)
    torch.cuda.synchronize()
    keys32 = O.selection_keys_f32(lg, score, bias)
    want = O.topk_select(keys32, k)
    got = i64(idx)
    if score == "softmax":
        np.testing.assert_array_equal(got, want)       # same fp32 keys: bit-exact, ties included
    else:
        # sigmoid keys round differently on each side: exact where the fp32 keys are 1e-6 apart
        gap = O.topk_gap(keys32.astype(np.float64), k)
        ok = gap > 1e-6
        np.testing.assert_array_equal(got[ok], want[ok])
        assert (~ok).sum() <= max(2, T // 50)
    g_ref = O.gates_from_logits(lg.astype(np.float64), got, score)
    np.testing.assert_allclose(f64(gate), g_ref, rtol=2e-6, atol=2e-7)
    np.testing.assert_allclose(f64(gate).sum(1), 1.0, atol=2e-6)


@pytest.mark.parametrize("E", [8, 64, 256])
def test_topk_signed_zero_keys_tie(lib, E):
    """Softmax keys are the logits: -0.0 and +0.0 are equal keys, so they tie
    and the lower expert id comes first whichever of the two carries the sign
    (the warp path ranks integer images of the keys, with -0 folded into +0)."""
    T, k = 64, 4
    lg = np.full((T, E), -1.0, np.float32)
    rng = np.random.default_rng(E)
    for t in range(T):
        a, b, c = rng.choice(E, 3, replace=False)
        lg[t, a], lg[t, b] = (-0.0, 0.0) if t % 2 else (0.0, -0.0)
        lg[t, c] = -0.0 if t % 3 else 0.5
    cfg = api.make_config(T, 128, E, k, 128, score="softmax")
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    api.moe_topk_gating(cfg, torch.from_numpy(lg).to(DEV), None, idx, gate)
    torch.cuda.synchronize()
    want = O.topk_select(O.selection_keys_f32(lg, "softmax", None), k)
    np.testing.assert_array_equal(i64(idx), want)


@pytest.mark.parametrize("score", ["softmax", "sigmoid"])
@pytest.mark.parametrize("T,E,k", [(96, 8, 2), (96, 64, 8), (40, 16, 16)])
def test_topk_nan_logits_rank_last(lib, score, T, E, k):
    """A NaN key ranks after every finite key (ties among them by lower id),
    as numpy's sort orders NaN: the order stays total, so every lane of the
    warp agrees and no expert is picked twice."""
    lg = _rand((T, E), T + E, 1.0)
    rng = np.random.default_rng(E + k)
    lg[rng.random((T, E)) < 0.2] = np.nan
    lg[7] = np.nan                              # a token with no finite logit
    bias = (_rand((E,), 6, 0.05) if score == "sigmoid" else None)
    cfg = api.make_config(T, 128, E, k, 128, score=score)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    api.moe_topk_gating(cfg, torch.from_numpy(lg).to(DEV),
                        None if bias is None else torch.from_numpy(bias).to(DEV), idx, gate)
    torch.cuda.synchronize()
    got = i64(idx)
    want = O.topk_select(O.selection_keys_f32(lg, score, bias), k)
    for t in range(T):
        assert len(set(got[t])) == k, t
    if score == "softmax":
        np.testing.assert_array_equal(got, want)
    else:
        keys32 = O.selection_keys_f32(lg, score, bias).astype(np.float64)
        fin = np.where(np.isnan(keys32), -np.inf, keys32)
        ok = O.topk_gap(np.nan_to_num(fin, neginf=-1e30), k) > 1e-6
        np.testing.assert_array_equal(got[ok], want[ok])
    np.testing.assert_array_equal(got[7], np.arange(k))
    finite_rows = np.isfinite(np.take_along_axis(lg, got, axis=1)).all(1)
    g_ref = O.gates_from_logits(lg.astype(np.float64), got, score)
    np.testing.assert_allclose(f64(gate)[finite_rows], g_ref[finite_rows], rtol=2e-6, atol=2e-7)


# ------------------------------------------------------------------ permutation
PERM_CASES = [
    # T, E, k, skew, H
    (256, 8, 2, 0.0, 128),
    (300, 16, 4, 1.5, 256),
    (64, 8, 8, 0.0, 128),       # k == E
    (1, 8, 2, 0.0, 128),
    (1000, 128, 8, 1.2, 128),
    (517, 256, 8, 2.0, 256),    # many empty experts, a few hot
    (2000, 8, 1, 4.0, 128),     # one expert takes almost everything
    (0, 8, 2, 0.0, 128),
    (500, 16, 3, 0.5, 128),     # k does not divide the 256-pair chunk
    (300, 32, 6, 1.0, 128),
    (300, 33, 2, 0.5, 128),     # one expert past the row copy's own column sums (last-block scan)
    (2100, 128, 8, 1.0, 128),   # histograms past the last-block scan (scan launch between)
]


def _perm_buffers(cfg):
    cap = api.moe_capacity_rows(cfg)
    T, E, k, H = cfg.T, cfg.E, cfg.k, cfg.H
    b = {
        "counts": torch.full((E,), -7, dtype=torch.int32, device=DEV),
        "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
        "poffsets": torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
        "slot_row": torch.full((max(T, 1), k), -7, dtype=torch.int32, device=DEV),
        "row_src": torch.full((cap,), -7, dtype=torch.int32, device=DEV),
        "row_gate": torch.full((cap,), -7.0, dtype=torch.float32, device=DEV),
        # 0xFFFF is a NaN pattern: unwritten rows are visible
        "x_perm": torch.full((cap, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16),
    }
    return cap, b


@pytest.mark.parametrize("T,E,k,skew,H", PERM_CASES)
def test_permute_bit_exact(lib, T, E, k, skew, H):
    idx = random_topk_indices(T, E, k, seed=T + E, skew=skew)
    gate = np.abs(_rand((T, k), 3)).astype(np.float32)
    x = to_bf16(_rand((T, H), 4))
    cfg = api.make_config(T, H, E, k, 128)
    cap, b = _perm_buffers(cfg)
    ws = _ws(cfg)
    api.moe_permute(cfg, x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(gate).to(DEV),
                    b["counts"], b["offsets"], b["poffsets"], b["slot_row"], b["row_src"], b["row_gate"],
                    b["x_perm"], 1, ws)
    torch.cuda.synchronize()
    assert _status(ws) == 0
    m = O.permutation_maps(idx, E, 128)
    np.testing.assert_array_equal(i64(b["counts"]), m["counts"])
    np.testing.assert_array_equal(i64(b["offsets"]), m["offsets"])
    np.testing.assert_array_equal(i64(b["poffsets"]), m["poffsets"])
    used = int(m["poffsets"][-1])
    if T:
        np.testing.assert_array_equal(i64(b["slot_row"]), m["slot_row"])
    np.testing.assert_array_equal(i64(b["row_src"])[:used], m["row_src"])
    rg = np.zeros(used, np.float32)
    v = m["row_src"] >= 0
    rg[v] = gate[m["row_src"][v], m["row_slot"][v]]
    np.testing.assert_array_equal(b["row_gate"].cpu().numpy()[:used], rg)
    want = O.permute(f64(x), m) if T else np.zeros((used, H))
    got_bits = b["x_perm"][:used].view(torch.int16).cpu().numpy()
    want_bits = to_bf16(want.astype(np.float32)).view(torch.int16).numpy()
    np.testing.assert_array_equal(got_bits, want_bits)


@pytest.mark.parametrize("T,E", [(1024, 8), (4096, 64), (4096, 128)])
def test_permute_is_deterministic(lib, T, E):
    """Three calls on one workspace give the same bits (32 chunks of 8
    experts: the row copy sums the raw histograms; 128 chunks of 64: the
    histogram launch's last block scans them and puts its counter back to
    zero; 128 of 128: a scan launch between)."""
    k, H = 8, 128
    idx = torch.from_numpy(random_topk_indices(T, E, k, seed=1, skew=1.0)).to(DEV)
    x = to_bf16(_rand((T, H), 9)).to(DEV)
    cfg = api.make_config(T, H, E, k, 128)
    ws = _ws(cfg)
    outs = []
    for _ in range(3):
        cap, b = _perm_buffers(cfg)
        api.moe_permute(cfg, x, idx, None, b["counts"], b["offsets"], b["poffsets"], b["slot_row"],
                        b["row_src"], None, b["x_perm"], 1, ws)
        outs.append((b["slot_row"].cpu(), b["x_perm"].view(torch.int16).cpu(), b["counts"].cpu()))
    assert _status(ws) == 0
    m = O.permutation_maps(idx.cpu().numpy(), E, 128)
    np.testing.assert_array_equal(outs[0][0].numpy(), m["slot_row"])
    np.testing.assert_array_equal(outs[0][2].numpy(), m["counts"])
    for o in outs[1:]:
        assert torch.equal(o[0], outs[0][0]) and torch.equal(o[1], outs[0][1]) and torch.equal(o[2], outs[0][2])


def test_launch_chaining_orders_around_other_kernels(lib):
    """Every library kernel waits for the kernel before it in the stream
    (griddepcontrol.wait) and torch's kernels after it wait for it: a torch
    write of x just before moe_permute is seen, one just after is not."""
    T, E, k, H = 2048, 8, 2, 512
    idx = torch.from_numpy(random_topk_indices(T, E, k, seed=5)).to(DEV)
    cfg = api.make_config(T, H, E, k, 128)
    ws = _ws(cfg)
    x = torch.zeros((T, H), dtype=torch.bfloat16, device=DEV)
    for rep in range(3):
        cap, b = _perm_buffers(cfg)
        x.fill_(float(rep + 1))                                   # a torch kernel right before
        api.moe_permute(cfg, x, idx, None, b["counts"], b["offsets"], b["poffsets"], b["slot_row"],
                        b["row_src"], None, b["x_perm"], 1, ws)
        x.fill_(-5.0)                                             # and one right after
        torch.cuda.synchronize()
        used = int(b["poffsets"][-1])
        rows = b["x_perm"][:used][b["row_src"][:used] >= 0].float()
        assert rows.numel() == T * k * H and torch.all(rows == float(rep + 1)), rep
    assert _status(ws) == 0


def test_permute_bad_index_sets_status(lib):
    """An out-of-range expert id is an input error the kernel bounds-checks:
    the pair is dropped, nothing out of range is written, the status word says so."""
    T, E, k, H = 64, 8, 2, 128
    idx = random_topk_indices(T, E, k, seed=2)
    idx[5, 1] = 9
    idx[7, 0] = -3
    x = to_bf16(_rand((T, H), 4))
    cfg = api.make_config(T, H, E, k, 128)
    cap, b = _perm_buffers(cfg)
    ws = _ws(cfg)
    api.moe_permute(cfg, x.to(DEV), torch.from_numpy(idx).to(DEV), None, b["counts"], b["offsets"],
                    b["poffsets"], b["slot_row"], b["row_src"], None, b["x_perm"], 0, ws)
    assert _status(ws) == -5
    assert int(b["counts"].sum()) == T * k - 2
    assert int(b["slot_row"][5, 1]) == -1 and int(b["slot_row"][7, 0]) == -1
    api.moe_workspace_init(ws)
    assert _status(ws) == 0


# ------------------------------------------------------------------ grouped GEMMs
def _routed_case(T, H, E, k, F, skew, seed):
    idx = random_topk_indices(T, E, k, seed=seed, skew=skew)
    m = O.permutation_maps(idx, E, 128)
    cfg = api.make_config(T, H, E, k, F)
    cap = api.moe_capacity_rows(cfg)
    used = int(m["poffsets"][-1])
    valid = np.zeros(cap, bool)
    valid[:used] = m["row_src"] >= 0
    return cfg, m, cap, used, valid


def _rows(cap, K, valid, seed, std=1.0):
    a = _rand((cap, K), seed, std)
    a[~valid] = 0.0          # padding rows are zero, as the permutation leaves them
    return to_bf16(a)


GEMM_CASES = [
    # T, H, E, k, F, skew
    (256, 128, 8, 2, 256, 0.0),       # tiny workload shape
    (700, 256, 16, 4, 384, 1.5),      # hot and empty experts, several tiles
    (300, 512, 128, 8, 128, 1.0),     # fine-grained experts
    (256, 256, 8, 2, 2048, 0.0),      # few tiles, long K
]


@pytest.mark.parametrize("T,H,E,k,F,skew", GEMM_CASES)
def test_gemm_fc1_fc2(lib, T, H, E, k, F, skew):
    cfg, m, cap, used, valid = _routed_case(T, H, E, k, F, skew, 11)
    a = _rows(cap, H, valid, 12)
    w1 = to_bf16(_rand((E, 2 * F, H), 13, 0.05))
    w2 = to_bf16(_rand((E, H, F), 14, 0.05))
    rg = np.where(valid, np.abs(_rand((cap,), 15)), 0).astype(np.float32)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    z = torch.zeros((cap, 2 * F), dtype=torch.bfloat16, device=DEV)
    h = torch.zeros((cap, F), dtype=torch.bfloat16, device=DEV)
    o = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg)
    api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, a.to(DEV), w1.to(DEV), h, ws, c2=z,
                         row_gate=torch.from_numpy(rg).to(DEV), poffsets=po)
    api.moe_grouped_gemm(cfg, api.GG_FC2, h, w2.to(DEV), o, ws, poffsets=po)
    torch.cuda.synchronize()
    assert _status(ws) == 0
    zr, hr = O.expert_fc1(f64(a)[:used], LazyW(w1), m["poffsets"], rg[:used])
    assert_bf16_close(f64(z)[:used], zr, "z")
    assert_bf16_close(f64(h)[:used], hr, "h")
    # Chained check: the oracle's fc2 runs on its own h rounded to bf16, the GPU's on its h; the
    # two h differ by one bf16 ulp wherever fp32 and fp64 z straddle a rounding boundary, so the
    # bound carries an absolute term for those.  (test_gemm_fc2_alone checks fc2 on identical h.)
    or_ = O.expert_fc2(f64(to_bf16(hr.astype(np.float32))), LazyW(w2), m["poffsets"])
    assert_bf16_close(f64(o)[:used], or_, "o", rel_l2_tol=8e-3, elem_rel=2.0 ** -6, elem_abs_frac=2e-2)


@pytest.mark.parametrize("T,H,E,k,F,skew", GEMM_CASES)
def test_gemm_fc1_gathered(lib, T, H, E, k, F, skew):
    """fc1 with the permutation fused into its A load (rows gathered from x in
    token order by row_src, zero rows for padding) gives z and h bit-identical
    to fc1 on the explicitly permuted x_perm (same operand bytes, same MMA
    order), and both match the oracle.  Rows past the last segment of row_src
    hold garbage that no tile may read."""
    cfg, m, cap, used, valid = _routed_case(T, H, E, k, F, skew, 31)
    x = to_bf16(_rand((T, H), 32))
    w1 = to_bf16(_rand((E, 2 * F, H), 33, 0.05)).to(DEV)
    rg = np.where(valid, np.abs(_rand((cap,), 34)), 0).astype(np.float32)
    rs = np.full(cap, 0x7F7F7F7F, np.int32)
    rs[:used] = m["row_src"]
    xp = np.zeros((cap, H), np.float32)
    xp[:used][m["row_src"] >= 0] = x.float().numpy()[m["row_src"][m["row_src"] >= 0]]
    x_perm = to_bf16(xp).to(DEV)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    rgd = torch.from_numpy(rg).to(DEV)
    ws = _ws(cfg)
    outs = []
    for op, a, extra in ((api.GG_FC1_SWIGLU, x_perm, {}),
                         (api.GG_FC1_SWIGLU_GATHERED, x.to(DEV), {"a_rows": torch.from_numpy(rs).to(DEV)})):
        z = torch.zeros((cap, 2 * F), dtype=torch.bfloat16, device=DEV)
        h = torch.zeros((cap, F), dtype=torch.bfloat16, device=DEV)
        api.moe_grouped_gemm(cfg, op, a, w1, h, ws, c2=z, row_gate=rgd, poffsets=po, **extra)
        outs.append((z, h))
    torch.cuda.synchronize()
    assert _status(ws) == 0
    (z0, h0), (z1, h1) = outs
    assert torch.equal(z0[:used].view(torch.int16), z1[:used].view(torch.int16))
    assert torch.equal(h0[:used].view(torch.int16), h1[:used].view(torch.int16))
    zr, hr = O.expert_fc1(f64(x_perm)[:used], LazyW(w1), m["poffsets"], rg[:used])
    assert_bf16_close(f64(h1)[:used], hr, "h (gathered)")


class LazyW:
    def __init__(self, t):
        self.t, self.shape, self.c = t, tuple(t.shape), {}

    def __getitem__(self, e):
        if e not in self.c:
            self.c[e] = f64(self.t[e])
        return self.c[e]


@pytest.mark.parametrize("T,H,E,k,F,skew", GEMM_CASES)
def test_gemm_fc2_alone(lib, T, H, E, k, F, skew):
    cfg, m, cap, used, valid = _routed_case(T, H, E, k, F, skew, 21)
    hin = _rows(cap, F, valid, 22)
    w2 = to_bf16(_rand((E, H, F), 23, 0.05))
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    o = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg)
    api.moe_grouped_gemm(cfg, api.GG_FC2, hin.to(DEV), w2.to(DEV), o, ws, poffsets=po)
    torch.cuda.synchronize()
    assert_bf16_close(f64(o)[:used], O.expert_fc2(f64(hin)[:used], LazyW(w2), m["poffsets"]), "o")


@pytest.mark.parametrize("shared,dropped", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("T,H,E,k,F,skew", [(700, 256, 16, 4, 384, 1.5), (300, 512, 128, 8, 128, 1.0),
                                            (256, 768, 8, 2, 256, 0.0)])
def test_gemm_fc2_combine(lib, T, H, E, k, F, skew, shared, dropped):
    """fc2 with the combine fused into its epilogue: o bit-identical to the
    plain fc2, y bit-identical to moe_unpermute of that o (same slot-order fp32
    sum, one rounding) and within the oracle's combine bound; two calls in a
    row (the counters go back to zero).  With dropped: some pairs have
    slot_row -1 (and their rows row_src -1), as after an out-of-range id."""
    cfg, m, cap, used, valid = _routed_case(T, H, E, k, F, skew, 41)
    hin = _rows(cap, F, valid, 42)
    w2 = to_bf16(_rand((E, H, F), 43, 0.05)).to(DEV)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    slot = m["slot_row"].astype(np.int32).copy()
    src = np.full(cap, -1, np.int32)
    src[:used] = m["row_src"]
    if dropped:
        rng = np.random.default_rng(44)
        for t in rng.choice(T, size=max(1, T // 20), replace=False):
            i = int(rng.integers(k))
            src[slot[t, i]] = -1
            slot[t, i] = -1
    slot_t, src_t = torch.from_numpy(slot).to(DEV), torch.from_numpy(src).to(DEV)
    sh = to_bf16(_rand((T, H), 45)).to(DEV) if shared else None
    ws = _ws(cfg)
    o_ref = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
    api.moe_grouped_gemm(cfg, api.GG_FC2, hin.to(DEV), w2, o_ref, ws, poffsets=po)
    y_ref = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    api.moe_unpermute(cfg, o_ref, slot_t, sh, y_ref)
    for rep in range(2):
        o = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
        y = torch.full((T, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        api.moe_grouped_gemm(cfg, api.GG_FC2_COMBINE, hin.to(DEV), w2, o, ws, c2=y, aux=sh, poffsets=po,
                             a_rows=src_t, slot_row=slot_t)
        torch.cuda.synchronize()
        assert _status(ws) == 0
        assert torch.equal(o[:used].view(torch.int16), o_ref[:used].view(torch.int16)), rep
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), rep
    # and against the oracle's combine of the same o (the plain fc2 is pinned by test_gemm_fc2_alone);
    # dropped pairs leave the sum, as moe_unpermute skips them
    o64 = f64(o_ref)
    if not dropped:
        ref = O.unpermute_sum(o64, m, None if sh is None else f64(sh))
    else:
        ref = np.where((slot >= 0)[..., None], o64[np.where(slot >= 0, slot, 0)], 0.0).sum(1)
        ref = ref + (f64(sh) if shared else 0.0)
    absum = np.where((slot >= 0)[..., None], np.abs(o64)[np.where(slot >= 0, slot, 0)], 0.0).sum(1)
    absum = absum + (np.abs(f64(sh)) if shared else 0.0)
    assert np.all(np.abs(f64(y) - ref) <= 2.0 ** -8 * np.abs(ref) + 2.0 ** -19 * absum + 1e-30)


@pytest.mark.parametrize("T,H,E,k,F,skew", GEMM_CASES)
def test_gemm_dgrad(lib, T, H, E, k, F, skew):
    cfg, m, cap, used, valid = _routed_case(T, H, E, k, F, skew, 31)
    dyp = _rows(cap, H, valid, 32)
    z = _rows(cap, 2 * F, valid, 33)
    w1 = to_bf16(_rand((E, 2 * F, H), 34, 0.05))
    w2 = to_bf16(_rand((E, H, F), 35, 0.05))
    rg = np.where(valid, np.abs(_rand((cap,), 36)), 0).astype(np.float32)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    dz = torch.zeros((cap, 2 * F), dtype=torch.bfloat16, device=DEV)
    dpart = torch.zeros((cap, F // 128), dtype=torch.float32, device=DEV)
    dx = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg)
    api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC2, dyp.to(DEV), w2.to(DEV), dz, ws, aux=z.to(DEV),
                         row_gate=torch.from_numpy(rg).to(DEV), dgate_part=dpart, poffsets=po)
    dz_in = _rows(cap, 2 * F, valid, 37)
    api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC1, dz_in.to(DEV), w1.to(DEV), dx, ws, poffsets=po)
    torch.cuda.synchronize()
    assert _status(ws) == 0
    dzr, dgr = O.expert_dgrad_fc2(f64(dyp)[:used], LazyW(w2), f64(z)[:used], m["poffsets"], rg[:used])
    assert_bf16_close(f64(dz)[:used], dzr, "dz", rel_l2_tol=6e-3)
    dg = f64(dpart)[:used].sum(1)
    scale = np.sqrt(np.mean(dgr ** 2)) + 1e-30
    assert np.max(np.abs(dg - dgr)) <= 2e-3 * scale + 1e-3 * np.abs(dgr).max(), "dgate partial sums"
    dxr = O.expert_dgrad_fc1(f64(dz_in)[:used], LazyW(w1), m["poffsets"])
    assert_bf16_close(f64(dx)[:used], dxr, "dx_perm")


@pytest.mark.parametrize("T,H,E,k,F,skew", GEMM_CASES)
def test_gemm_wgrad(lib, T, H, E, k, F, skew):
    cfg, m, cap, used, valid = _routed_case(T, H, E, k, F, skew, 41)
    dz = _rows(cap, 2 * F, valid, 42)
    xp = _rows(cap, H, valid, 43)
    dyp = _rows(cap, H, valid, 44)
    hh = _rows(cap, F, valid, 45)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    dw1 = torch.full((E, 2 * F, H), 7.0, dtype=torch.float32, device=DEV)
    dw2 = torch.full((E, H, F), 7.0, dtype=torch.float32, device=DEV)
    ws = _ws(cfg)
    api.moe_grouped_gemm(cfg, api.GG_WGRAD_FC1, dz.to(DEV), xp.to(DEV), dw1, ws, poffsets=po)
    api.moe_grouped_gemm(cfg, api.GG_WGRAD_FC2, dyp.to(DEV), hh.to(DEV), dw2, ws, poffsets=po)
    torch.cuda.synchronize()
    assert _status(ws) == 0
    for got, a_, b_, nm in ((dw1, dz, xp, "dW1"), (dw2, dyp, hh, "dW2")):
        ref = O.expert_wgrad(f64(a_)[:used], f64(b_)[:used], m["poffsets"])
        scale = np.einsum("rm,rn->mn", np.abs(f64(a_)[:used]), np.abs(f64(b_)[:used]))
        err = np.abs(f64(got) - ref)
        # fp32 output of an fp32-accumulated sum of exact bf16 products
        assert np.all(err <= 2.0 ** -14 * scale[None] + 1e-6), nm
        empty = m["counts"] == 0
        assert np.all(f64(got)[empty] == 0), nm + " of empty experts"


@pytest.mark.parametrize("T,H,S", [(256, 128, 256), (300, 256, 128), (77, 128, 128)])
def test_gemm_dense_shared_expert(lib, T, H, S):
    """The shared expert: one dense group of T rows (ragged T: the TMA box
    reads zeros past the end; stores are masked)."""
    cfg = api.make_config(T, H, 8, 2, 128, S)
    x = to_bf16(_rand((T, H), 51))
    w1 = to_bf16(_rand((2 * S, H), 52, 0.05))
    w2 = to_bf16(_rand((H, S), 53, 0.05))
    dy = to_bf16(_rand((T, H), 54))
    z = torch.zeros((T, 2 * S), dtype=torch.bfloat16, device=DEV)
    h = torch.zeros((T, S), dtype=torch.bfloat16, device=DEV)
    o = torch.zeros((T, H), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg)
    api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, x.to(DEV), w1.to(DEV), h, ws, c2=z, dense_rows=T)
    api.moe_grouped_gemm(cfg, api.GG_FC2, h, w2.to(DEV), o, ws, dense_rows=T)
    dz = torch.zeros((T, 2 * S), dtype=torch.bfloat16, device=DEV)
    api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC2, dy.to(DEV), w2.to(DEV), dz, ws, aux=z, dense_rows=T)
    dw1 = torch.zeros((2 * S, H), dtype=torch.float32, device=DEV)
    api.moe_grouped_gemm(cfg, api.GG_WGRAD_FC1, dz, x.to(DEV), dw1, ws, dense_rows=T)
    torch.cuda.synchronize()
    assert _status(ws) == 0
    po = O.dense_rows_of(T)
    zr, hr = O.expert_fc1(f64(x), f64(w1)[None], po)
    assert_bf16_close(f64(z), zr, "z shared")
    assert_bf16_close(f64(h), hr, "h shared")
    assert_bf16_close(f64(o), O.expert_fc2(f64(to_bf16(hr.astype(np.float32))), f64(w2)[None], po), "o shared",
                      rel_l2_tol=8e-3, elem_rel=2.0 ** -6, elem_abs_frac=6e-3)
    # backward through the shared expert, fed with the oracle's own z rounded to bf16
    dzr, _ = O.expert_dgrad_fc2(f64(dy), f64(w2)[None], f64(to_bf16(zr.astype(np.float32))), po)
    assert_bf16_close(f64(dz), dzr, "dz shared", rel_l2_tol=1e-2, elem_rel=2.0 ** -5, elem_abs_frac=1e-2)
    ref = O.expert_wgrad(f64(dz), f64(x), po)[0]
    assert rel_l2(f64(dw1), ref) < 1e-5


# ------------------------------------------------------------------ combine
@pytest.mark.parametrize("T,E,k,H,shared", [(256, 8, 2, 128, False), (300, 64, 8, 256, True),
                                            (1, 8, 2, 128, True), (999, 16, 1, 128, False)])
def test_unpermute(lib, T, E, k, H, shared):
    idx = random_topk_indices(T, E, k, seed=3)
    m = O.permutation_maps(idx, E, 128)
    cfg = api.make_config(T, H, E, k, 128)
    cap = api.moe_capacity_rows(cfg)
    o = to_bf16(_rand((cap, H), 61))
    sh = to_bf16(_rand((T, H), 62)) if shared else None
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    api.moe_unpermute(cfg, o.to(DEV), torch.from_numpy(m["slot_row"].astype(np.int32)).to(DEV),
                      None if sh is None else sh.to(DEV), y)
    torch.cuda.synchronize()
    ref = O.unpermute_sum(f64(o), m, None if sh is None else f64(sh))
    # fp32 sum of k+1 bf16 values, one rounding to bf16 (unit roundoff 2^-8) of the exact sum,
    # plus the fp32 sum's own rounding (k+1 <= 33 terms: |fp32 err| <= 2^-19 sum |terms|)
    got = f64(y)
    absum = np.abs(f64(o))[m["slot_row"]].sum(1) + (np.abs(f64(sh)) if shared else 0)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 2.0 ** -19 * absum + 1e-30)
