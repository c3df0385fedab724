"""GPU parity of the MXFP8 path through the C ABI.

* the quantiser is bit-exact against the oracle's (codes and E8M0 scales),
  over every finite bf16 value and in all three modes;
* each MXFP8 grouped GEMM matches the oracle's fp64 GEMM on the same quantised
  operands (the GPU quantises with its own kernel, the oracle with its own;
  both are bit-exact, so the operands are identical);
* the MXFP8 layer (forward, dgrad, wgrad) is within rel-L2 3e-2 of the fp64
  oracle of the same recipe (operands quantised along the same axes), and
  within the format's own error of the unquantised layer.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_bf16_close, f64, rel_l2
from moe_expert_layer_05_gb300 import api
from moe_expert_layer_05_gb300.inputs import Workload, make_inputs, random_topk_indices, to_bf16
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def untile(sf: torch.Tensor, R: int, C: int) -> np.ndarray:
    """Scale tiles (512 B per 128 rows x 4 blocks) -> plain [R, C/32]."""
    t = sf.cpu().numpy()[: R * C // 32].reshape(R // 128, C // 128, 512)
    r = np.arange(128)[:, None]
    b = np.arange(4)[None, :]
    idx = (r % 32) * 16 + (r // 32) * 4 + b
    return t[:, :, idx].transpose(0, 2, 1, 3).reshape(R, C // 32)


def untile_g224(sf: torch.Tensor, R: int, C: int) -> np.ndarray:
    """Scale tiles with the rows in groups of 224 (rows 0..127 of group g in
    tile row 2g, rows 128..223 in the first 96 rows of tile row 2g+1) -> [R, C/32]."""
    t = sf.cpu().numpy()[: (R // 224) * 2 * (C // 128) * 512].reshape(R // 224 * 2, C // 128, 512)
    r = np.arange(R)
    g, i = r // 224, r % 224
    tr, rr = 2 * g + i // 128, i % 128
    b = np.arange(C // 32)
    return t[tr[:, None], (b // 4)[None, :], ((rr % 32) * 16 + (rr // 32) * 4)[:, None] + (b % 4)[None, :]]


def quantize_gpu(x: torch.Tensor, mode: int, batch=1):
    n = x.numel()
    codes = torch.empty(n, dtype=torch.uint8, device=DEV)
    if mode in (api.MX_ROWS, api.MX_ROWS_G224):
        rows, cols = x.numel() // x.shape[-1], x.shape[-1]
        nsf = n // 32 if mode == api.MX_ROWS else rows // 224 * 2 * (cols // 128) * 512
        sf = torch.empty(nsf, dtype=torch.uint8, device=DEV)
        api.moe_quantize_mxfp8(x, 1, rows, cols, mode, codes, sf)
    else:
        rows, cols = x.shape[-2], x.shape[-1]
        nsf = n // 32 if mode != api.MX_COLS_T_G224 else batch * (cols // 224) * 2 * (rows // 128) * 512
        sf = torch.empty(nsf, dtype=torch.uint8, device=DEV)
        api.moe_quantize_mxfp8(x, batch, rows, cols, mode, codes, sf)
    return codes, sf


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape, dtype=np.float32) * np.float32(std)


def test_quantize_every_finite_bf16_value(lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    vals = vals[np.isfinite(vals)]
    vals = vals[np.argsort(np.abs(vals), kind="stable")]          # blocks of similar magnitude
    n = int(np.ceil(len(vals) / (128 * 128))) * 128 * 128
    full = np.zeros(n, np.float32)
    full[:len(vals)] = vals
    x = to_bf16(full.reshape(-1, 128))
    codes, sf = quantize_gpu(x.to(DEV), api.MX_ROWS)
    torch.cuda.synchronize()
    oc, os_ = O.mxfp8_quantize(f64(x), axis=-1)
    np.testing.assert_array_equal(codes.cpu().numpy().reshape(oc.shape), oc)
    np.testing.assert_array_equal(untile(sf, *x.shape), os_)


@pytest.mark.parametrize("R,C,scale", [(256, 512, 1.0), (128, 128, 1e-30), (384, 256, 1e30), (128, 7168, 3.0)])
def test_quantize_rows(lib, R, C, scale):
    v = _rand((R, C), R + C) * np.float32(scale)
    v[5, 64:96] = 0.0                                               # an all-zero block
    v[7, :32] *= np.float32(1e-3)
    x = to_bf16(v)
    codes, sf = quantize_gpu(x.to(DEV), api.MX_ROWS)
    torch.cuda.synchronize()
    oc, os_ = O.mxfp8_quantize(f64(x), axis=-1)
    np.testing.assert_array_equal(codes.cpu().numpy().reshape(R, C), oc)
    np.testing.assert_array_equal(untile(sf, R, C), os_)


@pytest.mark.parametrize("B,R,C,scale", [(1, 256, 384, 1.0), (3, 128, 256, 1.0), (2, 512, 128, 1.0),
                                         (1, 128, 640, 1e-30), (1, 256, 128, 1e30)])
def test_quantize_cols_transposed(lib, B, R, C, scale):
    x = to_bf16(_rand((B, R, C), 7 + B) * np.float32(scale))
    codes, sf = quantize_gpu(x.to(DEV), api.MX_COLS_T, batch=B)
    torch.cuda.synchronize()
    codes = codes.cpu().numpy().reshape(B, C, R)
    sfn = sf.reshape(B, -1)
    for b in range(B):
        oc, os_ = O.mxfp8_quantize(f64(x[b]).T, axis=-1)          # [C, R], blocks along R
        np.testing.assert_array_equal(codes[b], oc)
        np.testing.assert_array_equal(untile(sfn[b], C, R), os_)


def test_quantize_gate_up_interleave(lib):
    E, F, H = 2, 256, 128
    x = to_bf16(_rand((E, 2 * F, H), 9))
    codes, sf = quantize_gpu(x.to(DEV), api.MX_ROWS_GATE_UP, batch=E)
    torch.cuda.synchronize()
    got = codes.cpu().numpy().reshape(E, 2 * F, H)
    gsf = untile(sf, E * 2 * F, H).reshape(E, 2 * F, H // 32)
    oc, os_ = O.mxfp8_quantize(f64(x), axis=-1)
    for e in range(E):
        for j in range(2 * F):
            up, jj = divmod(j, F)
            r = (jj // 128) * 256 + up * 128 + jj % 128
            np.testing.assert_array_equal(got[e, r], oc[e, j])
            np.testing.assert_array_equal(gsf[e, r], os_[e, j])


def test_quantize_g224_scale_layout(lib):
    """The 224-row grouping changes where each scale byte sits, nothing else:
    codes identical, scales equal after both layouts are undone (row and
    transposed-column modes, several matrices)."""
    E, R, C = 2, 896, 1792          # rows (E*R) and output rows (C) multiples of 128 and 224
    x = to_bf16(_rand((E, R, C), 71) * np.float32(3.0)).to(DEV)
    c0, s0 = quantize_gpu(x.reshape(E * R, C), api.MX_ROWS)
    c1, s1 = quantize_gpu(x.reshape(E * R, C), api.MX_ROWS_G224)
    assert torch.equal(c0, c1)
    np.testing.assert_array_equal(untile(s0[: E * R * C // 32], E * R, C), untile_g224(s1, E * R, C))
    t0, u0 = quantize_gpu(x, api.MX_COLS_T, batch=E)             # [E, C, R], blocks along R
    t1, u1 = quantize_gpu(x, api.MX_COLS_T_G224, batch=E)
    assert torch.equal(t0, t1)
    per0, per1 = C * R // 32, (C // 224) * 2 * (R // 128) * 512
    for e in range(E):
        np.testing.assert_array_equal(untile(u0[e * per0:(e + 1) * per0], C, R),
                                      untile_g224(u1[e * per1:(e + 1) * per1], C, R))


# ------------------------------------------------------------------ grouped GEMMs
def _routed(T, H, E, k, F, skew, seed):
    idx = random_topk_indices(T, E, k, seed=seed, skew=skew)
    m = O.permutation_maps(idx, E, 128)
    cfg = api.make_config(T, H, E, k, F, dtype="mxfp8")
    cap = api.moe_capacity_rows(cfg)
    used = int(m["poffsets"][-1])
    valid = np.zeros(cap, bool)
    valid[:used] = m["row_src"] >= 0
    return cfg, m, cap, used, valid


def _rows(cap, K, valid, seed, std=1.0):
    a = _rand((cap, K), seed, std)
    a[~valid] = 0.0
    return to_bf16(a)


def _ws(cfg):
    ws = torch.zeros(api.moe_workspace_bytes(cfg), dtype=torch.uint8, device=DEV)
    api.moe_workspace_init(ws)
    return ws


def deq(t_bf16, axis):
    return O.mxfp8_roundtrip(f64(t_bf16), axis=axis)


MX_CASES = [
    # T, H, E, k, F, skew
    (256, 256, 8, 2, 256, 0.0),
    (640, 512, 16, 4, 384, 1.5),
    (384, 256, 64, 8, 128, 1.0),
]


@pytest.mark.parametrize("T,H,E,k,F,skew", MX_CASES)
def test_mx_gemm_forward(lib, T, H, E, k, F, skew):
    cfg, m, cap, used, valid = _routed(T, H, E, k, F, skew, 3)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    x = _rows(cap, H, valid, 4)
    w1 = to_bf16(_rand((E, 2 * F, H), 5, 0.05))
    w2 = to_bf16(_rand((E, H, F), 6, 0.05))
    rg = np.where(valid, np.abs(_rand((cap,), 7)), 0).astype(np.float32)
    xq, xsf = quantize_gpu(x.to(DEV), api.MX_ROWS)
    w1q, w1sf = quantize_gpu(w1.to(DEV), api.MX_ROWS_GATE_UP, batch=E)
    h_in = _rows(cap, F, valid, 8)
    hq, hsf = quantize_gpu(h_in.to(DEV), api.MX_ROWS)
    w2q, w2sf = quantize_gpu(w2.to(DEV).reshape(E * H, F), api.MX_ROWS)
    z = torch.zeros((cap, 2 * F), dtype=torch.bfloat16, device=DEV)
    h = torch.zeros((cap, F), dtype=torch.bfloat16, device=DEV)
    o = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg)
    api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, xq, w1q, h, ws, c2=z, row_gate=torch.from_numpy(rg).to(DEV),
                         poffsets=po, a_scales=xsf, b_scales=w1sf)
    api.moe_grouped_gemm(cfg, api.GG_FC2, hq, w2q, o, ws, poffsets=po, a_scales=hsf, b_scales=w2sf)
    torch.cuda.synchronize()
    assert api.moe_read_device_status(ws) == 0
    zr, hr = O.expert_fc1(deq(x, -1)[:used], deq(w1, -1), m["poffsets"], rg[:used])
    assert_bf16_close(f64(z)[:used], zr, "z (mxfp8)")
    assert_bf16_close(f64(h)[:used], hr, "h (mxfp8)")
    assert_bf16_close(f64(o)[:used], O.expert_fc2(deq(h_in, -1)[:used], deq(w2, -1), m["poffsets"]), "o (mxfp8)")


@pytest.mark.parametrize("T,H,E,k,F,skew", [(256, 256, 8, 2, 256, 0.0), (640, 512, 16, 4, 384, 1.5)])
def test_mx_gemm_fc2_combine(lib, T, H, E, k, F, skew):
    """MXFP8 fc2 with the combine fused into its epilogue: o bit-identical to
    the plain MXFP8 fc2 and y to moe_unpermute of it, two calls in a row."""
    cfg, m, cap, used, valid = _routed(T, H, E, k, F, skew, 51)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    h_in = _rows(cap, F, valid, 52)
    w2 = to_bf16(_rand((E, H, F), 53, 0.05))
    hq, hsf = quantize_gpu(h_in.to(DEV), api.MX_ROWS)
    w2q, w2sf = quantize_gpu(w2.to(DEV).reshape(E * H, F), api.MX_ROWS)
    slot = torch.from_numpy(m["slot_row"].astype(np.int32)).to(DEV)
    src = torch.full((cap,), -1, dtype=torch.int32, device=DEV)
    src[:used] = torch.from_numpy(m["row_src"].astype(np.int32)).to(DEV)
    sh = to_bf16(_rand((T, H), 54)).to(DEV)
    ws = _ws(cfg)
    o_ref = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
    api.moe_grouped_gemm(cfg, api.GG_FC2, hq, w2q, o_ref, ws, poffsets=po, a_scales=hsf, b_scales=w2sf)
    y_ref = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    api.moe_unpermute(cfg, o_ref, slot, sh, y_ref)
    for rep in range(2):
        o = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
        y = torch.full((T, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        api.moe_grouped_gemm(cfg, api.GG_FC2_COMBINE, hq, w2q, o, ws, c2=y, aux=sh, poffsets=po, a_scales=hsf,
                             b_scales=w2sf, a_rows=src, slot_row=slot)
        torch.cuda.synchronize()
        assert api.moe_read_device_status(ws) == 0
        assert torch.equal(o[:used].view(torch.int16), o_ref[:used].view(torch.int16)), rep
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), rep


@pytest.mark.parametrize("T,H,E,k,F,skew", MX_CASES)
def test_mx_gemm_dgrad(lib, T, H, E, k, F, skew):
    cfg, m, cap, used, valid = _routed(T, H, E, k, F, skew, 13)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    dy = _rows(cap, H, valid, 14)
    z = _rows(cap, 2 * F, valid, 15)
    dz_in = _rows(cap, 2 * F, valid, 16)
    w1 = to_bf16(_rand((E, 2 * F, H), 17, 0.05))
    w2 = to_bf16(_rand((E, H, F), 18, 0.05))
    rg = np.where(valid, np.abs(_rand((cap,), 19)), 0).astype(np.float32)
    dyq, dysf = quantize_gpu(dy.to(DEV), api.MX_ROWS)
    w2tq, w2tsf = quantize_gpu(w2.to(DEV), api.MX_COLS_T, batch=E)        # [E, F, H]
    dzq, dzsf = quantize_gpu(dz_in.to(DEV), api.MX_ROWS)
    w1tq, w1tsf = quantize_gpu(w1.to(DEV), api.MX_COLS_T, batch=E)        # [E, H, 2F]
    dz = torch.zeros((cap, 2 * F), dtype=torch.bfloat16, device=DEV)
    dpart = torch.zeros((cap, F // 128), dtype=torch.float32, device=DEV)
    dx = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg)
    api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC2, dyq, w2tq, dz, ws, aux=z.to(DEV),
                         row_gate=torch.from_numpy(rg).to(DEV), dgate_part=dpart, poffsets=po, a_scales=dysf,
                         b_scales=w2tsf)
    api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC1, dzq, w1tq, dx, ws, poffsets=po, a_scales=dzsf, b_scales=w1tsf)
    torch.cuda.synchronize()
    assert api.moe_read_device_status(ws) == 0
    # W2 quantised along H (its rows), W1 along 2F (its rows): blocks run along each weight's axis 1 of [E, ., .]
    w2_deq = O.mxfp8_roundtrip(f64(w2), axis=1)
    w1_deq = O.mxfp8_roundtrip(f64(w1), axis=1)
    dzr, dgr = O.expert_dgrad_fc2(deq(dy, -1)[:used], w2_deq, f64(z)[:used], m["poffsets"], rg[:used])
    assert_bf16_close(f64(dz)[:used], dzr, "dz (mxfp8)", rel_l2_tol=6e-3)
    dg = f64(dpart)[:used].sum(1)
    assert rel_l2(dg, dgr) < 2e-3
    assert_bf16_close(f64(dx)[:used], O.expert_dgrad_fc1(deq(dz_in, -1)[:used], w1_deq, m["poffsets"]), "dx (mxfp8)")


@pytest.mark.parametrize("T,H,E,k,F,skew", [(512, 896, 8, 2, 256, 0.0), (640, 896, 16, 4, 384, 1.5),
                                             (384, 1792, 64, 8, 128, 1.0)])
def test_mx_gemm_256x224_tiles(lib, T, H, E, k, F, skew):
    """fc2 and the fc1 data gradient on 256 x 224 tiles (B's scale tiles grouped
    by 224 rows): against the oracle on the same quantised operands, and bit
    for bit against the 128 x 256 tiles (same products, same K order), with
    experts whose last 256-row tile is half empty."""
    cfg, m, cap, used, valid = _routed(T, H, E, k, F, skew, 81)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    h_in = _rows(cap, F, valid, 82)
    dz_in = _rows(cap, 2 * F, valid, 83)
    w1 = to_bf16(_rand((E, 2 * F, H), 84, 0.05))
    w2 = to_bf16(_rand((E, H, F), 85, 0.05))
    hq, hsf = quantize_gpu(h_in.to(DEV), api.MX_ROWS)
    dzq, dzsf = quantize_gpu(dz_in.to(DEV), api.MX_ROWS)
    w2q, w2sf = quantize_gpu(w2.to(DEV).reshape(E * H, F), api.MX_ROWS)
    w2g, w2gsf = quantize_gpu(w2.to(DEV).reshape(E * H, F), api.MX_ROWS_G224)
    w1tq, w1tsf = quantize_gpu(w1.to(DEV), api.MX_COLS_T, batch=E)
    w1tg, w1tgsf = quantize_gpu(w1.to(DEV), api.MX_COLS_T_G224, batch=E)
    ws = _ws(cfg)
    out = {}
    for tag, (b2, s2, b1, s1, g) in {"128": (w2q, w2sf, w1tq, w1tsf, 0), "224": (w2g, w2gsf, w1tg, w1tgsf, 224)}.items():
        o = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
        dx = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
        api.moe_grouped_gemm(cfg, api.GG_FC2, hq, b2, o, ws, poffsets=po, a_scales=hsf, b_scales=s2,
                             b_scale_group=g)
        api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC1, dzq, b1, dx, ws, poffsets=po, a_scales=dzsf, b_scales=s1,
                             b_scale_group=g)
        torch.cuda.synchronize()
        assert api.moe_read_device_status(ws) == 0
        out[tag] = (o, dx)
    o, dx = out["224"]
    assert_bf16_close(f64(o)[:used], O.expert_fc2(deq(h_in, -1)[:used], deq(w2, -1), m["poffsets"]), "o (224)")
    w1_deq = O.mxfp8_roundtrip(f64(w1), axis=1)
    assert_bf16_close(f64(dx)[:used], O.expert_dgrad_fc1(deq(dz_in, -1)[:used], w1_deq, m["poffsets"]), "dx (224)")
    for a, b in zip(out["224"], out["128"]):
        assert torch.equal(a[:used].view(torch.int16), b[:used].view(torch.int16))


@pytest.mark.parametrize("T,H,E,k,F,skew", [(512, 256, 8, 2, 256, 0.0), (640, 512, 16, 4, 512, 1.5),
                                             (384, 256, 64, 8, 256, 1.0)])
def test_mx_gemm_dgrad_fc2_mxfp8_copies(lib, T, H, E, k, F, skew):
    """The fc2 data gradient's epilogue also writing dz in MXFP8 (F % 256 ==
    0): the row copy equals the row quantiser applied to the bf16 dz of the
    same call, the transposed copy the column quantiser, codes and scales bit
    for bit over every expert's padded rows; dz and the gate partials are the
    same as without the copies."""
    cfg, m, cap, used, valid = _routed(T, H, E, k, F, skew, 101)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    dy = _rows(cap, H, valid, 102)
    z = _rows(cap, 2 * F, valid, 103).to(DEV)
    w2 = to_bf16(_rand((E, H, F), 104, 0.05))
    rg = torch.from_numpy(np.where(valid, np.abs(_rand((cap,), 105)), 0).astype(np.float32)).to(DEV)
    dyq, dysf = quantize_gpu(dy.to(DEV), api.MX_ROWS)
    w2tq, w2tsf = quantize_gpu(w2.to(DEV), api.MX_COLS_T, batch=E)
    ws = _ws(cfg)
    outs = []
    for with_q in (False, True):
        dz = torch.zeros((cap, 2 * F), dtype=torch.bfloat16, device=DEV)
        dpart = torch.zeros((cap, F // 128), dtype=torch.float32, device=DEV)
        q = dict(q_codes=torch.full((cap * 2 * F,), 0xAB, dtype=torch.uint8, device=DEV),
                 q_scales=torch.full((cap * 2 * F // 32,), 0xAB, dtype=torch.uint8, device=DEV),
                 qt_codes=torch.full((cap * 2 * F,), 0xAB, dtype=torch.uint8, device=DEV),
                 qt_scales=torch.full((cap * 2 * F // 32,), 0xAB, dtype=torch.uint8, device=DEV)) if with_q else {}
        api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC2, dyq, w2tq, dz, ws, aux=z, row_gate=rg, dgate_part=dpart,
                             poffsets=po, a_scales=dysf, b_scales=w2tsf, **q)
        torch.cuda.synchronize()
        assert api.moe_read_device_status(ws) == 0
        outs.append((dz, dpart, q))
    (dz0, dp0, _), (dz1, dp1, q) = outs
    assert torch.equal(dz0[:used].view(torch.int16), dz1[:used].view(torch.int16))
    assert torch.equal(dp0[:used], dp1[:used])
    rc, rs = quantize_gpu(dz1[:used].contiguous(), api.MX_ROWS)
    assert torch.equal(q["q_codes"][: used * 2 * F], rc)
    np.testing.assert_array_equal(untile(q["q_scales"], cap, 2 * F)[:used], untile(rs, used, 2 * F))
    tc, ts = quantize_gpu(dz1[:used].contiguous(), api.MX_COLS_T)          # [2F, used]
    got_t = q["qt_codes"].view(2 * F, cap)[:, :used].contiguous().view(-1)
    assert torch.equal(got_t, tc)
    np.testing.assert_array_equal(untile(q["qt_scales"], 2 * F, cap)[:, : used // 32], untile(ts, 2 * F, used))
    # without the bf16 dz (c = NULL), as the layer runs it: the same copies
    q2 = {k_: torch.zeros_like(v) for k_, v in q.items()}
    dpart2 = torch.zeros_like(dp1)
    api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC2, dyq, w2tq, None, ws, aux=z, row_gate=rg, dgate_part=dpart2,
                         poffsets=po, a_scales=dysf, b_scales=w2tsf, **q2)
    torch.cuda.synchronize()
    assert api.moe_read_device_status(ws) == 0
    assert torch.equal(dpart2[:used], dp1[:used])
    assert torch.equal(q2["q_codes"][: used * 2 * F], q["q_codes"][: used * 2 * F])
    assert torch.equal(q2["qt_codes"].view(2 * F, cap)[:, :used], q["qt_codes"].view(2 * F, cap)[:, :used])


@pytest.mark.parametrize("T,H,E,k,F,skew", [(512, 256, 8, 2, 256, 0.0), (640, 512, 16, 4, 384, 1.5)])
def test_mx_gemm_fc1_mxfp8_copies(lib, T, H, E, k, F, skew):
    """fc1's epilogue also writing h' in MXFP8: the row copy equals the row
    quantiser applied to the bf16 h' of the same call, the transposed copy the
    column quantiser, codes and scales bit for bit over every expert's padded
    rows; z and h' are the same as without the copies, and the copies are the
    same without the bf16 h' (c = NULL)."""
    cfg, m, cap, used, valid = _routed(T, H, E, k, F, skew, 111)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    x = _rows(cap, H, valid, 112)
    w1 = to_bf16(_rand((E, 2 * F, H), 113, 0.05))
    rg = torch.from_numpy(np.where(valid, np.abs(_rand((cap,), 114)), 0).astype(np.float32)).to(DEV)
    xq, xsf = quantize_gpu(x.to(DEV), api.MX_ROWS)
    w1q, w1sf = quantize_gpu(w1.to(DEV), api.MX_ROWS_GATE_UP, batch=E)
    ws = _ws(cfg)
    u8 = lambda n: torch.full((n,), 0xAB, dtype=torch.uint8, device=DEV)
    outs = []
    for mode in ("plain", "copies", "copies_only"):
        h = torch.zeros((cap, F), dtype=torch.bfloat16, device=DEV) if mode != "copies_only" else None
        z = torch.zeros((cap, 2 * F), dtype=torch.bfloat16, device=DEV)
        q = dict(q_codes=u8(cap * F), q_scales=u8(cap * F // 32), qt_codes=u8(cap * F),
                 qt_scales=u8(cap * F // 32)) if mode != "plain" else {}
        api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, xq, w1q, h, ws, c2=z, row_gate=rg, poffsets=po, a_scales=xsf,
                             b_scales=w1sf, **q)
        torch.cuda.synchronize()
        assert api.moe_read_device_status(ws) == 0
        outs.append((h, z, q))
    (h0, z0, _), (h1, z1, q1), (_, z2, q2) = outs
    for a, b in ((h0, h1), (z0, z1), (z0, z2)):
        assert torch.equal(a[:used].view(torch.int16), b[:used].view(torch.int16))
    rc, rs = quantize_gpu(h1[:used].contiguous(), api.MX_ROWS)
    assert torch.equal(q1["q_codes"][: used * F], rc)
    np.testing.assert_array_equal(untile(q1["q_scales"], cap, F)[:used], untile(rs, used, F))
    tc, ts = quantize_gpu(h1[:used].contiguous(), api.MX_COLS_T)          # [F, used]
    assert torch.equal(q1["qt_codes"].view(F, cap)[:, :used].contiguous().view(-1), tc)
    np.testing.assert_array_equal(untile(q1["qt_scales"], F, cap)[:, : used // 32], untile(ts, F, used))
    for k_ in ("q_codes", "q_scales"):
        assert torch.equal(q2[k_][: used * F // (32 if "scales" in k_ else 1)],
                           q1[k_][: used * F // (32 if "scales" in k_ else 1)])
    assert torch.equal(q2["qt_codes"].view(F, cap)[:, :used], q1["qt_codes"].view(F, cap)[:, :used])


@pytest.mark.parametrize("T,H,E,k,F,skew", MX_CASES)
def test_mx_gemm_wgrad(lib, T, H, E, k, F, skew):
    cfg, m, cap, used, valid = _routed(T, H, E, k, F, skew, 23)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    dz = _rows(cap, 2 * F, valid, 24)
    xp = _rows(cap, H, valid, 25)
    dzT, dzTs = quantize_gpu(dz.to(DEV), api.MX_COLS_T)      # [2F, cap]
    xT, xTs = quantize_gpu(xp.to(DEV), api.MX_COLS_T)        # [H, cap]
    dw1 = torch.full((E, 2 * F, H), 7.0, dtype=torch.float32, device=DEV)
    ws = _ws(cfg)
    api.moe_grouped_gemm(cfg, api.GG_WGRAD_FC1, dzT, xT, dw1, ws, poffsets=po, a_scales=dzTs, b_scales=xTs)
    torch.cuda.synchronize()
    assert api.moe_read_device_status(ws) == 0
    a = O.mxfp8_roundtrip(f64(dz), axis=0)[:used]            # blocks along tokens
    b = O.mxfp8_roundtrip(f64(xp), axis=0)[:used]
    ref = O.expert_wgrad(a, b, m["poffsets"])
    scale = np.einsum("rm,rn->mn", np.abs(a), np.abs(b))
    assert np.all(np.abs(f64(dw1) - ref) <= 2.0 ** -14 * scale[None] + 1e-6)
    assert np.all(f64(dw1)[m["counts"] == 0] == 0)


@pytest.mark.parametrize("T,H,E,k,F,skew", [(512, 896, 8, 2, 256, 0.0), (640, 896, 16, 4, 384, 1.5)])
def test_mx_gemm_wgrad_256x224_tiles(lib, T, H, E, k, F, skew):
    """The fc1 weight gradient on 256 x 224 tiles (x^T's scale tiles grouped by
    224 rows): against the oracle, zero for empty experts, and bit for bit
    against the 128 x 256 tiles."""
    cfg, m, cap, used, valid = _routed(T, H, E, k, F, skew, 91)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    dz = _rows(cap, 2 * F, valid, 92)
    xp = _rows(cap, H, valid, 93)
    dzT, dzTs = quantize_gpu(dz.to(DEV), api.MX_COLS_T)          # [2F, cap]
    xT, xTs = quantize_gpu(xp.to(DEV), api.MX_COLS_T)            # [H, cap]
    xTg, xTgs = quantize_gpu(xp.to(DEV), api.MX_COLS_T_G224)
    ws = _ws(cfg)
    out = []
    for b, bs, g in ((xT, xTs, 0), (xTg, xTgs, 224)):
        dw1 = torch.full((E, 2 * F, H), 7.0, dtype=torch.float32, device=DEV)
        api.moe_grouped_gemm(cfg, api.GG_WGRAD_FC1, dzT, b, dw1, ws, poffsets=po, a_scales=dzTs, b_scales=bs,
                             b_scale_group=g)
        torch.cuda.synchronize()
        assert api.moe_read_device_status(ws) == 0
        out.append(dw1)
    a = O.mxfp8_roundtrip(f64(dz), axis=0)[:used]
    bq = O.mxfp8_roundtrip(f64(xp), axis=0)[:used]
    ref = O.expert_wgrad(a, bq, m["poffsets"])
    scale = np.einsum("rm,rn->mn", np.abs(a), np.abs(bq))
    assert np.all(np.abs(f64(out[1]) - ref) <= 2.0 ** -14 * scale[None] + 1e-6)
    assert np.all(f64(out[1])[m["counts"] == 0] == 0)
    assert torch.equal(out[0], out[1])


@pytest.mark.parametrize("T,H,E,k,F,skew", [(512, 896, 8, 2, 256, 0.0), (640, 896, 16, 4, 512, 1.5)])
def test_mx_gemm_wgrad_fc2_transposed_tiles(lib, T, H, E, k, F, skew):
    """The fc2 weight gradient with its operands swapped (dW2^T = h'^T x dy^T
    on 256 x 224 tiles, dy^T's scales grouped by 224 rows, tiles stored
    transposed): dW2 [E, H, F] against the oracle, zero for empty experts, and
    against the unswapped GEMM."""
    cfg, m, cap, used, valid = _routed(T, H, E, k, F, skew, 95)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    dy = _rows(cap, H, valid, 96)
    hp = _rows(cap, F, valid, 97)
    dyT, dyTs = quantize_gpu(dy.to(DEV), api.MX_COLS_T)          # [H, cap]
    dyTg, dyTgs = quantize_gpu(dy.to(DEV), api.MX_COLS_T_G224)
    hT, hTs = quantize_gpu(hp.to(DEV), api.MX_COLS_T)            # [F, cap]
    ws = _ws(cfg)
    out = []
    for a_, as_, b_, bs_, g in ((dyT, dyTs, hT, hTs, 0), (hT, hTs, dyTg, dyTgs, 224)):
        dw2 = torch.full((E, H, F), 7.0, dtype=torch.float32, device=DEV)
        api.moe_grouped_gemm(cfg, api.GG_WGRAD_FC2, a_, b_, dw2, ws, poffsets=po, a_scales=as_, b_scales=bs_,
                             b_scale_group=g)
        torch.cuda.synchronize()
        assert api.moe_read_device_status(ws) == 0
        out.append(dw2)
    a = O.mxfp8_roundtrip(f64(dy), axis=0)[:used]
    bq = O.mxfp8_roundtrip(f64(hp), axis=0)[:used]
    ref = O.expert_wgrad(a, bq, m["poffsets"])
    scale = np.einsum("rm,rn->mn", np.abs(a), np.abs(bq))
    assert np.all(np.abs(f64(out[1]) - ref) <= 2.0 ** -14 * scale[None] + 1e-6)
    assert np.all(f64(out[1])[m["counts"] == 0] == 0)
    assert np.all(np.abs(f64(out[1]) - f64(out[0])) <= 2.0 ** -20 * scale[None] + 1e-7)


# ------------------------------------------------------------------ layer
MX_LAYERS = {
    "dsv3_mx_small": Workload("dsv3_mx_small", T=384, H=256, E=64, k=8, F=128, S=256, score="sigmoid", zipf_s=1.2,
                              dtype="mxfp8", backward=True),
    "mixtral_mx_small": Workload("mixtral_mx_small", T=256, H=512, E=8, k=2, F=768, dtype="mxfp8", backward=True),
    "wide_mx": Workload("wide_mx", T=256, H=256, E=8, k=2, F=2048, dtype="mxfp8", backward=True),   # few tiles, long K
    # H % 224 == 0: fc2 and the fc1 data gradient on 256 x 224 tiles
    "h896_mx": Workload("h896_mx", T=384, H=896, E=16, k=4, F=256, S=256, score="sigmoid", zipf_s=1.2,
                        dtype="mxfp8", backward=True),
}


@pytest.mark.parametrize("name", list(MX_LAYERS))
def test_mx_layer_against_mxfp8_oracle(lib, name):
    """The MXFP8 layer against the oracle of the same recipe (rel-L2 <= 3e-2),
    and against the unquantised layer (the format's own error: < 15 %)."""
    w = MX_LAYERS[name]
    inp = make_inputs(w, seed=2)
    dinp = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    layer = api.MoELayer(api.config_of(w), dinp, with_backward=True)
    layer.act.fill_(0x7F)      # large finite garbage: the layer must not read memory it did not write
    y = layer.forward(dinp["x"])
    dx, dgate, grads = layer.backward(dinp["x"], dinp["dy"])
    torch.cuda.synchronize()
    assert api.moe_read_device_status(layer.ws) == 0
    sh = dict(w1_shared=None if w.S == 0 else f64(inp["w1_shared"]),
              w2_shared=None if w.S == 0 else f64(inp["w2_shared"]))
    bias = None if inp["bias"] is None else f64(inp["bias"])
    args = (f64(inp["x"]), f64(inp["w_router"]), f64(inp["w1"]), f64(inp["w2"]))
    fwd = O.moe_forward_mx(*args, k=w.k, score=w.score, bias=bias, **sh)
    keys = O.selection_keys(fwd["logits"], w.score, bias)
    stable = O.topk_gap(keys, w.k) >= 1e-5
    np.testing.assert_array_equal(layer.fields()["topk_idx"].cpu().numpy()[stable], fwd["topk_idx"][stable])
    r_y = rel_l2(f64(y)[stable], fwd["y"][stable])
    assert r_y <= 3e-2, r_y
    # y (combine fused into fc2 where H % 256 == 0) = moe_unpermute of the layer's own o, bit for bit
    fl = layer.fields()
    os_rows = layer.view("os", torch.bfloat16, (w.T, w.H)) if w.S else None
    y_cmb = torch.empty_like(y)
    api.moe_unpermute(layer.cfg, fl["o"], fl["slot_row"], os_rows, y_cmb)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_cmb.view(torch.int16))
    plain = O.moe_forward(*args, k=w.k, score=w.score, bias=bias, **sh)
    assert rel_l2(f64(y)[stable], plain["y"][stable]) < 0.15
    bwd = O.moe_backward_mx(*args, fwd, f64(inp["dy"]), score=w.score, **sh)
    assert rel_l2(f64(dx)[stable], bwd["dx"][stable]) <= 3e-2
    assert rel_l2(f64(dgate)[stable], bwd["dgate"][stable]) <= 3e-2
    touched = np.zeros(w.E, bool)
    touched[fwd["topk_idx"][~stable].ravel()] = True
    for gname, oname in (("dw1", "dW1"), ("dw2", "dW2"), ("dw_router", "dWr")):
        r = rel_l2(f64(grads[gname])[~touched], bwd[oname][~touched])
        assert r <= 3e-2, (gname, r)
    if w.S and stable.all():
        for gname, oname in (("dw1_shared", "dW1_shared"), ("dw2_shared", "dW2_shared")):
            r = rel_l2(f64(grads[gname]), bwd[oname])
            assert r <= 3e-2, (gname, r)


def test_mx_layer_dz_copies_without_the_fused_epilogue(lib):
    """Where F % 256 != 0 the fc2 data gradient stores bf16 dz and the layer
    quantises it: the transposed codes and scales left in act equal the column
    quantiser applied to that dz, and the fc1 data gradient the layer computed
    from the row copy equals, bit for bit, the same GEMM fed by the row
    quantiser.  (Where F % 256 == 0 the epilogue writes both copies; see
    test_mx_gemm_dgrad_fc2_mxfp8_copies.)"""
    w = MX_LAYERS["dsv3_mx_small"]
    inp = make_inputs(w, seed=4)
    dinp = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    layer = api.MoELayer(api.config_of(w), dinp, with_backward=True)
    layer.act.fill_(0x7F)
    layer.forward(dinp["x"])
    layer.backward(dinp["x"], dinp["dy"])
    torch.cuda.synchronize()
    assert api.moe_read_device_status(layer.ws) == 0
    fl = layer.fields()
    cap, F2, H, E = layer.layout.cap, 2 * w.F, w.H, w.E
    used = int(fl["poffsets"][-1])
    dz = fl["dz"]
    # transposed copy: [2F, cap] codes, blocks along the rows
    ref_t, ref_ts = quantize_gpu(dz[:used].contiguous(), api.MX_COLS_T)          # [2F, used]
    got_t = layer.view("dz_qt", torch.uint8, (F2, cap))[:, :used]
    assert torch.equal(got_t.contiguous().view(-1), ref_t)
    got_ts = untile(layer.view("dz_qt_sf", torch.uint8, (F2 * cap // 32,)), F2, cap)[:, : used // 32]
    np.testing.assert_array_equal(got_ts, untile(ref_ts, F2, used))
    # row copy, through the fc1 data gradient
    g = 224 if H % 224 == 0 else 0
    dzq, dzsf = quantize_gpu(dz, api.MX_ROWS)
    w1tq, w1tsf = quantize_gpu(dinp["w1"], api.MX_COLS_T_G224 if g else api.MX_COLS_T, batch=E)
    dx = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
    ws = _ws(layer.cfg)
    api.moe_grouped_gemm(layer.cfg, api.GG_DGRAD_FC1, dzq, w1tq, dx, ws, poffsets=fl["poffsets"], a_scales=dzsf,
                         b_scales=w1tsf, b_scale_group=g)
    torch.cuda.synchronize()
    assert api.moe_read_device_status(ws) == 0
    assert torch.equal(dx[:used].view(torch.int16), fl["dx_perm"][:used].view(torch.int16))


def _stable_expert_tokens(w, x64, wr64, bias64, idx_gpu, counts):
    """A mid-sized expert all of whose tokens are routed away from near ties
    (fp64 top-k key gaps >= 1e-5), with its tokens and their oracle routing."""
    order = np.argsort(counts, kind="stable")
    nz = order[counts[order] > 0]
    for j in range(len(nz) // 2, len(nz)):
        e = int(nz[j])
        toks = np.nonzero((idx_gpu == e).any(1))[0]
        logits = O.router_logits(x64[toks], wr64)
        keys = O.selection_keys(logits, w.score, bias64)
        if np.all(O.topk_gap(keys, w.k) >= 1e-5):
            idx, gate = O.route(logits, w.k, w.score, bias64)
            return e, toks, idx, gate
    raise AssertionError("no expert with only stable tokens")


def test_mx_full_size_training_sampled(lib):
    """The DeepSeek-like MXFP8 training layer at full size (T=16384, E=256,
    shared expert), forward and backward as the benchmark runs them:
    * the permutation at full T bit for bit against the oracle's counting sort
      on the GPU's routing;
    * two sampled tokens end to end against the oracle alone (fp64 router,
      every expert they reach and the shared expert quantised by the oracle):
      y, dx, dgate and dlogits within rel-L2 3e-2;
    * a mid-sized expert e, over all of its tokens, against the oracle
      restricted to that expert (its gates given, as router replay does):
      dW1[e] and dW2[e] in full, the gate gradients of its slots, and sampled
      rows of z, o and dx_perm from the oracle's own step functions (h' and
      dz only in MXFP8: through o, dx_perm, dW1[e] and dW2[e]);
    * dWr[e] as the router weight-gradient step on the layer's own dlogits."""
    from gpu_helpers import StreamExperts, check_full_permutation, i64, mx_weight_cache
    from moe_expert_layer_05_gb300.inputs import WORKLOADS, make_inputs_on_device
    w = WORKLOADS["dsv3_mxfp8"]
    dinp = make_inputs_on_device(w, DEV, seed=0)
    layer = api.MoELayer(api.config_of(w), dinp, with_backward=True)
    layer.act.fill_(0x7F)
    y = layer.forward(dinp["x"])
    dx, dgate, grads = layer.backward(dinp["x"], dinp["dy"])
    torch.cuda.synchronize()
    assert api.moe_read_device_status(layer.ws) == 0
    fl = layer.fields()
    check_full_permutation(w, fl, dinp["x"], rows=False)
    counts, po, src = i64(fl["counts"]), i64(fl["poffsets"]), i64(fl["row_src"])
    idx_gpu = i64(fl["topk_idx"])
    x64, dy64 = f64(dinp["x"]), f64(dinp["dy"])
    wr64, bias64 = f64(dinp["w_router"]), f64(dinp["bias"])
    e, toks, idx_o, gate_o = _stable_expert_tokens(w, x64, wr64, bias64, idx_gpu, counts)
    np.testing.assert_array_equal(idx_o, idx_gpu[toks])
    rng = np.random.default_rng(13)
    sample = np.sort(rng.choice(len(toks), size=2, replace=False))
    ts = toks[sample]
    cache = mx_weight_cache(dinp["w1"], dinp["w2"], np.unique(idx_o[sample]), dinp["w1_shared"], dinp["w2_shared"])

    # two tokens end to end, the oracle alone
    W1, W2 = StreamExperts(dinp["w1"]), StreamExperts(dinp["w2"])
    sh = dict(w1_shared=f64(dinp["w1_shared"]), w2_shared=f64(dinp["w2_shared"]), weight_cache=cache)
    fwd = O.moe_forward_mx(x64[ts], wr64, W1, W2, k=w.k, score=w.score, bias=bias64, **sh)
    np.testing.assert_array_equal(fwd["topk_idx"], idx_gpu[ts])
    bwd = O.moe_backward_mx(x64[ts], wr64, W1, W2, fwd, dy64[ts], score=w.score, weight_grads=False, **sh)
    ts_t = torch.from_numpy(ts).to(DEV)
    for what, got, ref in (("y", y[ts_t], fwd["y"]), ("dx", dx[ts_t], bwd["dx"]), ("dgate", dgate[ts_t], bwd["dgate"]),
                           ("dlogits", fl["dlogits"][ts_t], bwd["dlogits"])):
        r = rel_l2(f64(got), ref)
        assert r <= 3e-2, (what, r)

    # expert e over all of its tokens, the oracle restricted to it
    n = len(toks)
    slot_o = np.argmax(idx_o == e, axis=1)
    g_e = gate_o[np.arange(n), slot_o]
    ce = {("w1", 0, a): cache[("w1", e, a)] for a in (-1, 0) if ("w1", e, a) in cache}
    ce.update({("w2", 0, a): cache[("w2", e, a)] for a in (-1, 0) if ("w2", e, a) in cache})
    w1e, w2e = f64(dinp["w1"][e])[None], f64(dinp["w2"][e])[None]
    fwd_e = O.moe_forward_mx(x64[toks], wr64[e:e + 1], w1e, w2e, k=1, score=w.score,
                             routing=(np.zeros((n, 1), np.int64), g_e[:, None]), weight_cache=ce)
    bwd_e = O.moe_backward_mx(x64[toks], wr64[e:e + 1], w1e, w2e, fwd_e, dy64[toks], score=w.score, weight_cache=ce)
    for what, got, ref in (("dW1[e]", grads["dw1"][e], bwd_e["dW1"][0]), ("dW2[e]", grads["dw2"][e], bwd_e["dW2"][0])):
        r = rel_l2(f64(got), ref)
        assert r <= 3e-2, (what, r)
    slot_g = np.argmax(idx_gpu[toks] == e, axis=1)
    r = rel_l2(f64(dgate)[toks, slot_g], bwd_e["dgate"][:, 0])
    assert r <= 3e-2, ("dgate of expert e", r)
    # sampled rows of expert e: z, h', o, dz, dx_perm by the oracle's step functions
    rows = np.sort(po[e] + rng.choice(counts[e], size=8, replace=False))
    rt = src[rows]
    assert np.all(np.isin(rt, toks))
    g_rows = g_e[np.searchsorted(toks, rt)]
    seg = np.array([0, len(rows)])
    z, hp = O.expert_fc1(O.mxfp8_roundtrip(x64[rt], -1), ce[("w1", 0, -1)][None], seg, g_rows)
    o = O.expert_fc2(O.mxfp8_roundtrip(hp, -1), ce[("w2", 0, -1)][None], seg)
    dz, _ = O.expert_dgrad_fc2(O.mxfp8_roundtrip(dy64[rt], -1), ce[("w2", 0, 0)][None], z, seg, g_rows)
    dxp = O.expert_dgrad_fc1(O.mxfp8_roundtrip(dz, -1), ce[("w1", 0, 0)][None], seg)
    rows_t = torch.from_numpy(rows).to(DEV)
    # (h' and dz stay in MXFP8: h''s row copy feeds o and its transposed copy dW2[e], dz's feed
    # dx_perm and dW1[e], all checked)
    for what, name, ref in (("z", "z", z), ("o", "o", o), ("dx_perm", "dx_perm", dxp)):
        r = rel_l2(f64(fl[name][rows_t]), ref)
        assert r <= 3e-2, (what, r)
    # dWr[e] = sum over the tokens of e of dlogits[t, e] x[t] (the step, on the layer's dlogits)
    ref = f64(fl["dlogits"])[:, e] @ x64
    assert rel_l2(f64(grads["dw_router"][e]), ref) <= 1e-4
