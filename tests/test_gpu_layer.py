"""GPU parity of the whole layer (forward, dgrad, wgrad) through the C ABI
against the fp64 oracle, plus the sync-free properties: CUDA-graph capture
and replay, bit-identical reruns.

End-to-end tolerance for bf16 outputs: max-abs <= 2e-2 + 2^-8 |y_ref| and
rel-L2 <= 1e-2.  The 2^-8 |y_ref| term is the output format itself: y is
returned in bf16, whose rounding alone moves a value of magnitude 8 by up to
0.03.  Tokens whose top-k choice is within 1e-5 of a tie (in the oracle's fp64
keys) may be routed differently by a fp32 router; they are counted and left out
of the element comparison.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import LazyExperts, check_full_permutation, f64, i64, rel_l2
from moe_expert_layer_05_gb300 import api
from moe_expert_layer_05_gb300.inputs import WORKLOADS, Workload, make_inputs, make_inputs_on_device
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"
NEAR_TIE = 1e-5

SMALL = {
    "tiny": WORKLOADS["tiny"],
    "tiny_bwd": Workload("tiny_bwd", T=256, H=128, E=8, k=2, F=256, backward=True),
    "mixtral_small": Workload("mixtral_small", T=333, H=512, E=8, k=2, F=768, backward=True),
    "qwen3_small": Workload("qwen3_small", T=512, H=256, E=128, k=8, F=256, backward=True),
    "dsv3_small": Workload("dsv3_small", T=384, H=256, E=256, k=8, F=128, S=256, score="sigmoid",
                           zipf_s=1.2, backward=True),
    "one_token": Workload("one_token", T=1, H=128, E=8, k=2, F=128, S=128, backward=True),
    "odd_k": Workload("odd_k", T=200, H=128, E=16, k=3, F=128, backward=True),
    "wide_ffn": Workload("wide_ffn", T=256, H=256, E=8, k=2, F=2048, backward=True),   # few tiles, long K
}


def _to_dev(inp):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _layer(w: Workload, dev_inp, with_backward):
    cfg = api.config_of(w, tokens=dev_inp["x"].shape[0])
    layer = api.MoELayer(cfg, dev_inp, with_backward=with_backward)
    layer.act.fill_(0x7F)      # large finite garbage: the layer must not read memory it did not write
    return layer


def _oracle_fwd(w, inp_cpu, tokens=None):
    x = f64(inp_cpu["x"])
    if tokens is not None:
        x = x[tokens]
    return O.moe_forward(x, f64(inp_cpu["w_router"]), inp_cpu["w1_np"], inp_cpu["w2_np"], k=w.k, score=w.score,
                         bias=None if inp_cpu["bias"] is None else f64(inp_cpu["bias"]),
                         w1_shared=None if w.S == 0 else f64(inp_cpu["w1_shared"]),
                         w2_shared=None if w.S == 0 else f64(inp_cpu["w2_shared"]))


def _stable_tokens(w, logits, bias):
    keys = O.selection_keys(logits, w.score, None if bias is None else f64(bias))
    return O.topk_gap(keys, w.k) >= NEAR_TIE


def check_e2e(got, ref, what):
    err = np.abs(got - ref)
    bound = 2e-2 + 2.0 ** -8 * np.abs(ref)
    assert np.all(err <= bound), f"{what}: max err {err.max():.4f} (bound at that element {bound.flat[err.argmax()]:.4f})"
    r = rel_l2(got, ref)
    assert r <= 1e-2, f"{what}: rel-L2 {r:.3e}"
    return r


def check_combine_bits(layer, w, y):
    """y of the layer (the combine fused into fc2 where H % 256 == 0, the
    combine kernel otherwise) is bit-identical to moe_unpermute of the layer's
    own o and shared-expert rows."""
    fl = layer.fields()
    sh = layer.view("os", torch.bfloat16, (w.T, w.H)) if w.S else None
    ref = torch.empty_like(y)
    api.moe_unpermute(layer.cfg, fl["o"], fl["slot_row"], sh, ref)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


def check_dlogits(w, fl, dgate, bwd_dlogits, stable, tol):
    """dlogits of the layer: against the oracle's router backward (end to end,
    on the stable tokens), and as a step against the router-backward formula
    applied to the GPU's own fp32 logits, gates and gate gradients."""
    got = f64(fl["dlogits"])
    r = rel_l2(got[stable], bwd_dlogits[stable])
    assert r <= tol, f"dlogits rel-L2 {r:.3e}"
    dg = f64(dgate)
    step = O.router_backward(f64(fl["logits"]), i64(fl["topk_idx"]), f64(fl["topk_gate"]), dg, w.score)
    # fp32 evaluation of the same formula: a few ulps of the row's gate gradients
    row_scale = np.abs(dg).max(axis=1, keepdims=True) + np.abs(step).max(axis=1, keepdims=True)
    assert np.all(np.abs(got - step) <= 1e-5 * np.abs(step) + 1e-6 * row_scale)
    assert rel_l2(got, step) <= 1e-5
    assert np.all(got[step == 0] == 0)           # only the chosen experts' logits get gradient


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_small(lib, name):
    w = SMALL[name]
    inp = make_inputs(w, seed=3)
    inp["w1_np"] = f64(inp["w1"])
    inp["w2_np"] = f64(inp["w2"])
    dinp = _to_dev(inp)
    layer = _layer(w, dinp, w.backward)
    y = layer.forward(dinp["x"])
    torch.cuda.synchronize()
    assert api.moe_read_device_status(layer.ws) == 0
    fwd = _oracle_fwd(w, inp)
    stable = _stable_tokens(w, fwd["logits"], inp["bias"])
    fl = layer.fields()
    # routing: identical on every token that is not a near tie
    np.testing.assert_array_equal(i64(fl["topk_idx"])[stable], fwd["topk_idx"][stable])
    check_e2e(f64(y)[stable], fwd["y"][stable], f"{name} y")
    assert (~stable).sum() <= max(1, w.T // 100)
    check_full_permutation(w, fl, dinp["x"])
    check_combine_bits(layer, w, y)
    if not w.backward:
        return
    dy = dinp["dy"]
    dx, dgate, grads = layer.backward(dinp["x"], dy)
    torch.cuda.synchronize()
    assert api.moe_read_device_status(layer.ws) == 0
    bwd = O.moe_backward(f64(inp["x"]), f64(inp["w_router"]), inp["w1_np"], inp["w2_np"], fwd, f64(inp["dy"]),
                         score=w.score, w1_shared=None if w.S == 0 else f64(inp["w1_shared"]),
                         w2_shared=None if w.S == 0 else f64(inp["w2_shared"]))
    dxr = bwd["dx"][stable]
    r = rel_l2(f64(dx)[stable], dxr)
    assert r <= 1e-2, f"dx rel-L2 {r:.3e}"
    assert np.all(np.abs(f64(dx)[stable] - dxr) <= 2e-2 * max(1.0, np.abs(dxr).max()) + 2.0 ** -7 * np.abs(dxr))
    assert rel_l2(f64(dgate)[stable], bwd["dgate"][stable]) <= 1e-2
    check_dlogits(w, layer.fields(), dgate, bwd["dlogits"], stable, 1e-2)
    touched = np.zeros(w.E, bool)
    touched[fwd["topk_idx"][~stable].ravel()] = True
    for gname, oname in (("dw1", "dW1"), ("dw2", "dW2"), ("dw_router", "dWr")):
        got = f64(grads[gname])[~touched]
        ref = bwd[oname][~touched]
        assert rel_l2(got, ref) <= 1e-2, f"{gname} rel-L2 {rel_l2(got, ref):.3e}"
    if w.S:
        for gname, oname in (("dw1_shared", "dW1_shared"), ("dw2_shared", "dW2_shared")):
            if (~stable).any():
                continue
            assert rel_l2(f64(grads[gname]), bwd[oname]) <= 1e-2, gname


def test_layer_graph_capture_and_determinism(lib):
    """The layer issues no host sync and a fixed launch sequence, so the whole
    forward + backward captures into one CUDA graph; replays give results
    bit-identical to eager runs (the permutation is a stable counting sort; the
    GEMMs' tile counter decides which SM runs a tile, never how it is
    computed).  The counter is back at zero after every launch."""
    w = SMALL["qwen3_small"]
    dinp = _to_dev(make_inputs(w, seed=5))
    layer = _layer(w, dinp, True)
    x, dy = dinp["x"], dinp["dy"]
    y0 = layer.forward(x).clone()
    dx0, dg0, g0 = layer.backward(x, dy)
    dx0, dg0, dw10 = dx0.clone(), dg0.clone(), g0["dw1"].clone()
    torch.cuda.synchronize()
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    dgate = torch.empty_like(dg0)
    grads = {k: torch.empty_like(v) for k, v in g0.items()}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x, y)
        layer.backward(x, dy, grads, dx, dgate)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, y)
        layer.backward(x, dy, grads, dx, dgate)
    for _ in range(3):
        y.zero_()
        dx.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))
        assert torch.equal(dx.view(torch.int16), dx0.view(torch.int16))
        assert torch.equal(dgate, dg0)
        assert torch.equal(grads["dw1"], dw10)
    assert api.moe_read_device_status(layer.ws) == 0
    words = layer.ws[:256].view(torch.int32).cpu()
    assert int(words[32]) == 0 and int(words[33]) == 0


def _full_case(name, n_sample, seed=0):
    w = WORKLOADS[name]
    dinp = make_inputs_on_device(w, DEV, seed=seed)
    inp = {"x": dinp["x"].cpu(), "w_router": dinp["w_router"].cpu(),
           "bias": None if dinp["bias"] is None else dinp["bias"].cpu(),
           "w1_shared": None if w.S == 0 else dinp["w1_shared"].cpu(),
           "w2_shared": None if w.S == 0 else dinp["w2_shared"].cpu(),
           "w1_np": LazyExperts(dinp["w1"]), "w2_np": LazyExperts(dinp["w2"])}
    rng = np.random.default_rng(seed + 17)
    tokens = np.sort(rng.choice(w.T, size=n_sample, replace=False))
    return w, dinp, inp, tokens


@pytest.mark.parametrize("name,n_sample", [("mixtral", 16), ("dsv3", 8)])
def test_layer_full_size_forward_sampled(lib, name, n_sample):
    """Full workload shape, in the launch configuration the benchmark times;
    the oracle evaluates a seeded sample of tokens one by one."""
    w, dinp, inp, tokens = _full_case(name, n_sample)
    layer = _layer(w, dinp, False)
    y = layer.forward(dinp["x"])
    torch.cuda.synchronize()
    assert api.moe_read_device_status(layer.ws) == 0
    fl = layer.fields()
    # the permutation at full T, bit for bit against the oracle's counting sort
    check_full_permutation(w, fl, dinp["x"])
    check_combine_bits(layer, w, y)
    fwd = _oracle_fwd(w, inp, tokens)
    stable = _stable_tokens(w, fwd["logits"], inp["bias"])
    np.testing.assert_array_equal(i64(fl["topk_idx"])[tokens][stable], fwd["topk_idx"][stable])
    check_e2e(f64(y[torch.from_numpy(tokens).to(DEV)])[stable], fwd["y"][stable], f"{name} y")


def test_layer_full_size_qwen3_fwd_bwd_sampled(lib):
    w, dinp, inp, tokens = _full_case("qwen3", 8)
    inp["dy"] = dinp["dy"].cpu()
    layer = _layer(w, dinp, True)
    y = layer.forward(dinp["x"])
    dx, dgate, grads = layer.backward(dinp["x"], dinp["dy"])
    torch.cuda.synchronize()
    assert api.moe_read_device_status(layer.ws) == 0
    fwd = _oracle_fwd(w, inp, tokens)
    stable = _stable_tokens(w, fwd["logits"], None)
    check_e2e(f64(y[torch.from_numpy(tokens).to(DEV)])[stable], fwd["y"][stable], "qwen3 y")
    fl = layer.fields()
    check_full_permutation(w, fl, dinp["x"])
    bwd = O.moe_backward(f64(inp["x"])[tokens], f64(inp["w_router"]), inp["w1_np"], inp["w2_np"], fwd,
                         f64(inp["dy"])[tokens], score=w.score, weight_grads=False)
    tok_t = torch.from_numpy(tokens).to(DEV)
    got_dx = f64(dx[tok_t])[stable]
    assert rel_l2(got_dx, bwd["dx"][stable]) <= 1e-2
    assert rel_l2(f64(dgate[tok_t])[stable], bwd["dgate"][stable]) <= 1e-2
    assert rel_l2(f64(fl["dlogits"][tok_t])[stable], bwd["dlogits"][stable]) <= 1e-2
    # one expert's weight gradients in full: all tokens routed to it
    idx_gpu = i64(fl["topk_idx"])
    order = np.argsort(np.bincount(idx_gpu.ravel(), minlength=w.E))
    for e_star in [int(order[w.E // 2 + j]) for j in range(8)]:
        toks = np.nonzero((idx_gpu == e_star).any(1))[0]
        fwd_e = _oracle_fwd(w, inp, toks)
        if np.all(O.topk_gap(O.selection_keys(fwd_e["logits"], w.score), w.k) >= NEAR_TIE):
            break
    np.testing.assert_array_equal(fwd_e["topk_idx"], idx_gpu[toks])
    bwd_e = O.moe_backward(f64(inp["x"])[toks], f64(inp["w_router"]), inp["w1_np"], inp["w2_np"], fwd_e,
                           f64(inp["dy"])[toks], score=w.score)
    assert rel_l2(f64(grads["dw1"][e_star]), bwd_e["dW1"][e_star]) <= 1e-2
    assert rel_l2(f64(grads["dw2"][e_star]), bwd_e["dW2"][e_star]) <= 1e-2
    assert rel_l2(f64(grads["dw_router"][e_star]), bwd_e["dWr"][e_star]) <= 1e-2


def test_few_tiles_long_k_is_deterministic(lib):
    """Few tiles with long K (fewer tiles than SMs): reruns are bit-identical."""
    w = SMALL["wide_ffn"]
    dinp = _to_dev(make_inputs(w, seed=7))
    layer = _layer(w, dinp, True)
    outs = []
    for _ in range(3):
        y = layer.forward(dinp["x"]).clone()
        dx, dg, g = layer.backward(dinp["x"], dinp["dy"])
        torch.cuda.synchronize()
        outs.append((y.view(torch.int16).clone(), dx.view(torch.int16).clone(), g["dw1"].clone()))
    for o in outs[1:]:
        assert all(torch.equal(a, b) for a, b in zip(o, outs[0]))
    assert api.moe_read_device_status(layer.ws) == 0


def test_router_replay_reproduces_the_layer_permutation(lib):
    """Router replay: the routing a layer forward recorded (topk_idx, gates) is
    fed back to moe_permute, which must rebuild the same expert-ordered batch
    bit for bit (maps, gates per row, x_perm), with no router call."""
    w = SMALL["dsv3_small"]
    dinp = _to_dev(make_inputs(w, seed=21))
    layer = _layer(w, dinp, True)
    layer.forward(dinp["x"])
    torch.cuda.synchronize()
    fl = layer.fields()
    cfg = layer.cfg
    cap = api.moe_capacity_rows(cfg)
    E = w.E
    got = {"counts": torch.empty(E, dtype=torch.int32, device=DEV),
           "offsets": torch.empty(E + 1, dtype=torch.int32, device=DEV),
           "poffsets": torch.empty(E + 1, dtype=torch.int32, device=DEV),
           "slot_row": torch.empty_like(fl["slot_row"]),
           "row_src": torch.full((cap,), -7, dtype=torch.int32, device=DEV),
           "row_gate": torch.empty(cap, dtype=torch.float32, device=DEV),
           "x_perm": torch.empty((cap, w.H), dtype=torch.bfloat16, device=DEV)}
    ws = torch.zeros(max(api.moe_workspace_bytes(cfg), 256), dtype=torch.uint8, device=DEV)
    api.moe_workspace_init(ws)
    api.moe_permute(cfg, dinp["x"], fl["topk_idx"].clone(), fl["topk_gate"].clone(), got["counts"], got["offsets"],
                    got["poffsets"], got["slot_row"], got["row_src"], got["row_gate"], got["x_perm"], 1, ws)
    torch.cuda.synchronize()
    assert api.moe_read_device_status(ws) == 0
    used = int(fl["poffsets"][-1])
    for name in ("counts", "offsets", "poffsets", "slot_row"):
        assert torch.equal(got[name], fl[name]), name
    assert torch.equal(got["row_src"][:used], fl["row_src"][:used])
    assert torch.equal(got["row_gate"][:used], fl["row_gate"][:used])
    assert torch.equal(got["x_perm"][:used].view(torch.int16), fl["x_perm"][:used].view(torch.int16))


@pytest.mark.parametrize("nan", [False, True])
@pytest.mark.parametrize("E,k,score", [(8, 2, "softmax"), (16, 3, "sigmoid"), (16, 16, "softmax"), (32, 4, "softmax"),
                                       (64, 8, "sigmoid")])
def test_fused_topk_matches_the_standalone_gating(lib, E, k, score, nan):
    """The layer's top-k (fused with the counting-sort histogram: one thread
    per token for E <= 16, one warp per token above) gives indices and gates
    bit-identical to the standalone gating kernel on the same logits.  With
    nan: one expert's router row and two tokens are NaN, so NaN logits reach
    both paths (a NaN key ranks last in both)."""
    w = Workload("topk", T=640, H=128, E=E, k=k, F=128, score=score, zipf_s=1.2 if score == "sigmoid" else 0.0)
    dinp = _to_dev(make_inputs(w, seed=9))
    if nan:
        dinp["w_router"][min(3, E - 1)] = float("nan")
        dinp["x"][5] = float("nan")
        dinp["x"][300] = float("nan")
    layer = _layer(w, dinp, False)
    layer.forward(dinp["x"])
    fl = layer.fields()
    idx = torch.empty_like(fl["topk_idx"])
    gate = torch.empty_like(fl["topk_gate"])
    api.moe_topk_gating(layer.cfg, fl["logits"], dinp["bias"], idx, gate)
    torch.cuda.synchronize()
    assert torch.equal(idx, fl["topk_idx"])
    assert torch.equal(gate.view(torch.int32), fl["topk_gate"].view(torch.int32))
    if nan:
        lg = fl["logits"].cpu().numpy()
        bias = None if dinp["bias"] is None else dinp["bias"].cpu().numpy()
        want = O.topk_select(O.selection_keys_f32(lg, score, bias), k)
        got = i64(idx)
        assert all(len(set(r)) == k for r in got)
        np.testing.assert_array_equal(got[5], np.arange(k))
        rows = np.ones(len(got), bool)
        rows[[5, 300]] = False                     # every logit NaN: experts 0..k-1
        if k < E:
            assert not (got[rows] == min(3, E - 1)).any()     # the NaN expert is never chosen
        if score == "softmax":
            np.testing.assert_array_equal(got, want)
