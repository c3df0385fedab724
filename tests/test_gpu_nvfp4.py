"""GPU parity of the NVFP4 path through the C ABI.

* the quantiser is bit-exact against the oracle's: E2M1 codes, E4M3 scales
  (tiled) and the tensor amax, over every finite bf16 value, across scales,
  and with the gate/up row interleave;
* each NVFP4 grouped GEMM (fc1 with the gated SwiGLU epilogue, fc2) matches
  the oracle's fp64 GEMM on the same quantised operands (both quantisers are
  bit-exact, so the operands are identical), within bf16 output rounding;
* the NVFP4 layer forward is within rel-L2 3e-2 of the fp64 oracle of the
  same recipe, and within the format's own error of the unquantised layer.
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


def untile16(sf: torch.Tensor, R: int, C: int) -> np.ndarray:
    """NVFP4 scale tiles (512 B per 128 rows x 4 blocks of 16) -> plain [R, C/16]."""
    t = sf.cpu().numpy().reshape(R // 128, C // 64, 512)
    r = np.arange(128)[:, None]
    b = np.arange(4)[None, :]
    idx = (r % 32) * 16 + (r // 32) * 4 + b
    return t[:, :, idx].transpose(0, 2, 1, 3).reshape(R, C // 16)


def unpack(codes: torch.Tensor, R: int, C: int) -> np.ndarray:
    """Two E2M1 codes per byte, the lower-indexed element in the low nibble -> [R, C]."""
    b = codes.cpu().numpy().reshape(R, C // 2)
    out = np.empty((R, C), np.uint8)
    out[:, 0::2] = b & 0xF
    out[:, 1::2] = b >> 4
    return out


def quantize_gpu(x: torch.Tensor, mode: int, batch=1):
    n = x.numel()
    codes = torch.empty(n // 2, dtype=torch.uint8, device=DEV)
    sf = torch.empty(n // 16, dtype=torch.uint8, device=DEV)
    amax = torch.full((1,), -1.0, dtype=torch.float32, device=DEV)
    if mode == api.MX_ROWS:
        api.moe_quantize_nvfp4(x, 1, n // x.shape[-1], x.shape[-1], mode, codes, sf, amax)
    else:
        api.moe_quantize_nvfp4(x, batch, x.shape[-2], x.shape[-1], mode, codes, sf, amax)
    return codes, sf, amax


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape, dtype=np.float32) * np.float32(std)


def _check_quant(x: torch.Tensor, codes, sf, amax):
    R, C = x.shape
    v = f64(x)
    oc, os_, S = O.nvfp4_quantize(v, axis=-1)
    assert float(amax.item()) == float(np.abs(v).max())
    np.testing.assert_array_equal(unpack(codes, R, C), oc)
    np.testing.assert_array_equal(untile16(sf, R, C), os_)


def test_quantize_every_finite_bf16_value(lib):
    """All finite bf16 values, sorted by magnitude into 64-wide rows: blocks
    span every binade, so every scale byte and every rounding case occurs
    (the tensor amax is the largest bf16, so small blocks get subnormal or zero
    scales)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    vals = vals[np.isfinite(vals)]
    vals = vals[np.argsort(np.abs(vals), kind="stable")]
    n = int(np.ceil(len(vals) / (128 * 64))) * 128 * 64
    full = np.zeros(n, np.float32)
    full[:len(vals)] = vals
    x = to_bf16(full.reshape(-1, 64)).to(DEV)
    c, s, a = quantize_gpu(x, api.MX_ROWS)
    torch.cuda.synchronize()
    _check_quant(x, c, s, a)


@pytest.mark.parametrize("R,C,scale", [(256, 512, 1.0), (128, 64, 1e-30), (384, 256, 1e30), (128, 7168, 3.0),
                                       (256, 4096, 0.02)])
def test_quantize_rows(lib, R, C, scale):
    v = _rand((R, C), R + C) * np.float32(scale)
    v[5, 64:80] = 0.0                                        # an all-zero block
    v[7, :16] *= np.float32(1e-3)                            # a block far below the tensor amax
    v[9, 32:48] = np.float32(scale) * np.float32(2.5)        # exact ties of the E2M1 grid after scaling
    x = to_bf16(v).to(DEV)
    c, s, a = quantize_gpu(x, api.MX_ROWS)
    torch.cuda.synchronize()
    _check_quant(x, c, s, a)


def test_quantize_zero_tensor(lib):
    x = torch.zeros((128, 256), dtype=torch.bfloat16, device=DEV)
    c, s, a = quantize_gpu(x, api.MX_ROWS)
    torch.cuda.synchronize()
    assert a.item() == 0.0 and not c.any() and not s.any()


def test_quantize_gate_up_interleave(lib):
    E, F, H = 2, 256, 128
    x = to_bf16(_rand((E, 2 * F, H), 9))
    c, s, a = quantize_gpu(x.to(DEV), api.MX_ROWS_GATE_UP, batch=E)
    torch.cuda.synchronize()
    got = unpack(c, E * 2 * F, H).reshape(E, 2 * F, H)
    gsf = untile16(s, E * 2 * F, H).reshape(E, 2 * F, H // 16)
    oc, os_, _ = O.nvfp4_quantize(f64(x), axis=-1)
    assert float(a.item()) == float(np.abs(f64(x)).max())
    for e in range(E):
        for j in range(2 * F):
            up, jj = divmod(j, F)
            r = (jj // 128) * 256 + up * 128 + jj % 128
            np.testing.assert_array_equal(got[e, r], oc[e, j])
            np.testing.assert_array_equal(gsf[e, r], os_[e, j])


# ------------------------------------------------------------------ grouped GEMMs
def _routed(T, H, E, k, F, skew, seed):
    idx = random_topk_indices(T, E, k, seed=seed, skew=skew)
    m = O.permutation_maps(idx, E, 128)
    cfg = api.make_config(T, H, E, k, F, dtype="nvfp4")
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


NV_CASES = [
    # T, H, E, k, F, skew
    (256, 256, 8, 2, 256, 0.0),
    (640, 512, 16, 4, 512, 1.5),      # ragged experts, some empty
    (384, 768, 64, 8, 256, 1.0),      # H / 256 = 3 k-blocks
    (256, 4096, 4, 2, 768, 0.0),      # long K
]


@pytest.mark.parametrize("T,H,E,k,F,skew", NV_CASES)
def test_nv4_gemm_forward(lib, T, H, E, k, F, skew):
    cfg, m, cap, used, valid = _routed(T, H, E, k, F, skew, 3)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    x = _rows(cap, H, valid, 4)
    w1 = to_bf16(_rand((E, 2 * F, H), 5, 0.05))
    w2 = to_bf16(_rand((E, H, F), 6, 0.05))
    rg = np.where(valid, np.abs(_rand((cap,), 7)), 0).astype(np.float32)
    xq, xsf, xa = quantize_gpu(x.to(DEV), api.MX_ROWS)
    w1q, w1sf, w1a = quantize_gpu(w1.to(DEV), api.MX_ROWS_GATE_UP, batch=E)
    h_in = _rows(cap, F, valid, 8)
    hq, hsf, ha = quantize_gpu(h_in.to(DEV), api.MX_ROWS)
    w2q, w2sf, w2a = quantize_gpu(w2.to(DEV).reshape(E * H, F), api.MX_ROWS)
    h = torch.zeros((cap, F), dtype=torch.bfloat16, device=DEV)
    z = torch.zeros((cap, 2 * F), dtype=torch.bfloat16, device=DEV)
    h2 = torch.zeros((cap, F), dtype=torch.bfloat16, device=DEV)
    o = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg)
    rgd = torch.from_numpy(rg).to(DEV)
    api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, xq, w1q, h, ws, row_gate=rgd, poffsets=po, a_scales=xsf,
                         b_scales=w1sf, a_amax=xa, b_amax=w1a)
    api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, xq, w1q, h2, ws, c2=z, row_gate=rgd, poffsets=po, a_scales=xsf,
                         b_scales=w1sf, a_amax=xa, b_amax=w1a)
    api.moe_grouped_gemm(cfg, api.GG_FC2, hq, w2q, o, ws, poffsets=po, a_scales=hsf, b_scales=w2sf, a_amax=ha,
                         b_amax=w2a)
    torch.cuda.synchronize()
    assert api.moe_read_device_status(ws) == 0
    xd = O.nvfp4_roundtrip(f64(x), axis=-1)
    w1d = O.nvfp4_roundtrip(f64(w1), axis=-1)
    zr, hr = O.expert_fc1(xd[:used], w1d, m["poffsets"], rg[:used])
    assert_bf16_close(f64(h)[:used], hr, "h (nvfp4)")
    assert_bf16_close(f64(h2)[:used], hr, "h with z saved (nvfp4)")
    assert_bf16_close(f64(z)[:used], zr, "z (nvfp4)")
    ref_o = O.expert_fc2(O.nvfp4_roundtrip(f64(h_in), axis=-1)[:used], O.nvfp4_roundtrip(f64(w2), axis=-1),
                         m["poffsets"])
    assert_bf16_close(f64(o)[:used], ref_o, "o (nvfp4)")


def test_nv4_gemm_dense_and_backward_ops_refused(lib):
    """Dense (shared-expert) NVFP4 GEMMs; the backward ops are not offered."""
    T, H, S = 256, 512, 256
    cfg = api.make_config(T, H, 8, 2, 256, S, dtype="nvfp4")
    x = to_bf16(_rand((T, H), 31))
    w1 = to_bf16(_rand((2 * S, H), 32, 0.05))
    xq, xsf, xa = quantize_gpu(x.to(DEV), api.MX_ROWS)
    w1q, w1sf, w1a = quantize_gpu(w1.to(DEV), api.MX_ROWS_GATE_UP)
    h = torch.zeros((T, S), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg)
    api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, xq, w1q, h, ws, dense_rows=T, a_scales=xsf, b_scales=w1sf,
                         a_amax=xa, b_amax=w1a)
    torch.cuda.synchronize()
    assert api.moe_read_device_status(ws) == 0
    _, hr = O.expert_fc1(O.nvfp4_roundtrip(f64(x), axis=-1), O.nvfp4_roundtrip(f64(w1), axis=-1)[None],
                         np.array([0, T]))
    assert_bf16_close(f64(h), hr, "shared h (nvfp4)")
    with pytest.raises(api.MoeError):
        api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC1, xq, w1q, h, ws, dense_rows=T, a_scales=xsf, b_scales=w1sf,
                             a_amax=xa, b_amax=w1a)


# ------------------------------------------------------------------ layer
NV_LAYERS = {
    "tiny_nvfp4": Workload("tiny_nvfp4", T=256, H=256, E=8, k=2, F=512, dtype="nvfp4"),
    "dsv3_nv_small": Workload("dsv3_nv_small", T=384, H=512, E=64, k=8, F=256, S=256, score="sigmoid",
                              zipf_s=1.2, dtype="nvfp4"),
    "wide_nv": Workload("wide_nv", T=256, H=256, E=8, k=2, F=2048, dtype="nvfp4"),
}


@pytest.mark.parametrize("name", list(NV_LAYERS))
def test_nv4_layer_against_nvfp4_oracle(lib, name):
    """The NVFP4 layer forward against the oracle of the same recipe (rel-L2
    <= 3e-2: the two sides round h to bf16 from slightly different fp32 / fp64
    values, and a flipped bf16 ulp can move an E2M1 code), and against the
    unquantised layer (the format's own error: < 30 %)."""
    w = NV_LAYERS[name]
    inp = make_inputs(w, seed=2)
    dinp = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    layer = api.MoELayer(api.config_of(w), dinp, with_backward=False)
    # the activation buffer starts as large finite garbage (bf16 0x7F7F): nothing
    # the forward reads may come from memory it did not write
    layer.act.fill_(0x7F)
    y = layer.forward(dinp["x"])
    torch.cuda.synchronize()
    assert api.moe_read_device_status(layer.ws) == 0
    sh = dict(w1_shared=None if w.S == 0 else f64(inp["w1_shared"]),
              w2_shared=None if w.S == 0 else f64(inp["w2_shared"]))
    bias = None if inp["bias"] is None else f64(inp["bias"])
    args = (f64(inp["x"]), f64(inp["w_router"]), f64(inp["w1"]), f64(inp["w2"]))
    fwd = O.moe_forward_nvfp4(*args, k=w.k, score=w.score, bias=bias, **sh)
    keys = O.selection_keys(fwd["logits"], w.score, bias)
    stable = O.topk_gap(keys, w.k) >= 1e-5
    np.testing.assert_array_equal(layer.fields()["topk_idx"].cpu().numpy()[stable], fwd["topk_idx"][stable])
    r_y = rel_l2(f64(y)[stable], fwd["y"][stable])
    assert r_y <= 3e-2, r_y
    plain = O.moe_forward(*args, k=w.k, score=w.score, bias=bias, **sh)
    assert rel_l2(f64(y)[stable], plain["y"][stable]) < 0.3
    with pytest.raises(api.MoeError):
        api.MoELayer(api.config_of(w), dinp, with_backward=True).forward(dinp["x"])


def test_nv4_full_size_sampled(lib):
    """The Mixtral-like NVFP4 forward at full size, as the benchmark runs it.
    Tensor amaxes are read from the device tensors with torch (exact maxima
    of bf16 values); for the expert with the most rows, seeded sample rows of
    h' and o are recomputed by the oracle from those amaxes (fc1 from x and
    W1, fc2 from the stored h' rows and W2); the combine is checked on the
    sampled tokens; the routing properties hold at any size; and the layer
    stays within the format's error of the bf16 layer."""
    from gpu_helpers import i64
    from moe_expert_layer_05_gb300.inputs import WORKLOADS, make_inputs_on_device
    w = WORKLOADS["mixtral_nvfp4"]
    dinp = make_inputs_on_device(w, DEV, seed=0)
    layer = api.MoELayer(api.config_of(w), dinp, with_backward=False)
    layer.act.fill_(0x7F)
    y = layer.forward(dinp["x"])
    torch.cuda.synchronize()
    assert api.moe_read_device_status(layer.ws) == 0
    fl = layer.fields()
    cap = layer.layout.cap
    counts, po = i64(fl["counts"]), i64(fl["poffsets"])
    assert counts.sum() == w.T * w.k
    slot = i64(fl["slot_row"])
    src = i64(fl["row_src"])
    assert np.all(src[slot] == np.arange(w.T)[:, None])
    valid = torch.from_numpy((np.arange(cap) < po[-1]) & (src >= 0)).to(DEV)
    x_amax = float(dinp["x"].abs().max())
    h_amax = float(fl["h"][valid].abs().max())
    w1_amax, w2_amax = float(dinp["w1"].abs().max()), float(dinp["w2"].abs().max())
    e = int(np.argmax(counts))
    rng = np.random.default_rng(11)
    rows = np.sort(po[e] + rng.choice(counts[e], size=6, replace=False))
    toks = src[rows]
    rows_t = torch.from_numpy(rows).to(DEV)
    F = w.F
    xq = O.nvfp4_roundtrip(f64(dinp["x"][torch.from_numpy(toks).to(DEV)]), x_amax)
    z = xq @ O.nvfp4_roundtrip(f64(dinp["w1"][e]), w1_amax).T
    g = f64(fl["row_gate"][rows_t])
    assert_bf16_close(f64(fl["h"][rows_t]), g[:, None] * O.silu(z[:, :F]) * z[:, F:], "h (nvfp4, full size)")
    hq = O.nvfp4_roundtrip(f64(fl["h"][rows_t]), h_amax)
    o_ref = hq @ O.nvfp4_roundtrip(f64(dinp["w2"][e]), w2_amax).T
    assert_bf16_close(f64(fl["o"][rows_t]), o_ref, "o (nvfp4, full size)")
    # combine on the sampled tokens: y[t] = bf16(sum over the token's k rows of o)
    o_rows = f64(fl["o"][torch.from_numpy(slot[toks].ravel()).to(DEV)]).reshape(len(toks), w.k, w.H)
    assert_bf16_close(f64(y[torch.from_numpy(toks).to(DEV)]), o_rows.sum(1), "y (nvfp4 combine, full size)")
    # the whole layer against the bf16 layer: the format's own error, not a gross one
    ref = api.MoELayer(api.config_of(WORKLOADS["mixtral"]), dinp, with_backward=False).forward(dinp["x"])
    torch.cuda.synchronize()
    r = rel_l2(f64(y), f64(ref))
    assert 0.02 < r < 0.3, r


def test_nv4_layer_graph_replay_is_bit_identical(lib):
    """The NVFP4 forward (amax reductions, quantisers, code gather, GEMMs with
    the fused h' amax) issues no host sync: it captures into one CUDA graph,
    and replays are bit-identical to the eager run (the amaxes are maxima, so
    the atomics' order does not matter)."""
    w = NV_LAYERS["dsv3_nv_small"]
    inp = make_inputs(w, seed=4)
    dinp = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    layer = api.MoELayer(api.config_of(w), dinp, with_backward=False)
    x = dinp["x"]
    y0 = layer.forward(x).clone()
    torch.cuda.synchronize()
    y = torch.empty_like(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x, y)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, y)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))
    assert api.moe_read_device_status(layer.ws) == 0
