"""The permutation entry point for callers that cannot allocate device memory
(moe_permute_noalloc: no workspace argument, scratch in a fixed device array
owned by the library).  Checked through the C ABI against moe_permute, which
uses a caller-provided workspace, on two calls in a row: the second call has a
different shape and routing, so anything it wrongly kept from the first call's
scratch would show.  Also against the oracle's permutation maps, on the
documented handling of out-of-range expert ids (the pair is dropped, its
slot_row is -1, nothing outside the buffers is written), and that a call
changes the device's free memory by nothing.  Collected last on purpose."""
import numpy as np
import pytest
import torch

from moe_expert_layer_05_gb300 import api
from moe_expert_layer_05_gb300.inputs import random_topk_indices, to_bf16
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _buffers(cfg):
    cap = api.moe_capacity_rows(cfg)
    T, E, k, H = cfg.T, cfg.E, cfg.k, cfg.H
    return {
        "counts": torch.full((E,), -7, dtype=torch.int32, device=DEV),
        "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
        "poffsets": torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
        "slot_row": torch.full((max(T, 1), k), -7, dtype=torch.int32, device=DEV),
        "row_src": torch.full((cap,), -7, dtype=torch.int32, device=DEV),
        "row_gate": torch.full((cap,), -7.0, dtype=torch.float32, device=DEV),
        "x_perm": torch.full((cap, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16),
    }


def _run(fn, cfg, x, idx, gate, extra):
    b = _buffers(cfg)
    fn(cfg, x, idx, gate, b["counts"], b["offsets"], b["poffsets"], b["slot_row"], b["row_src"], b["row_gate"],
       b["x_perm"], 1, *extra)
    return b


@pytest.mark.parametrize("first,second", [((4096, 256, 8, 1.2, 256, 3), (1000, 16, 4, 0.0, 128, 4))])
def test_noalloc_permute_matches_workspace_permute(first, second):
    api.load()
    for T, E, k, skew, H, seed in (first, second):
        cfg = api.make_config(T, H, E, k, 128)
        idx = torch.from_numpy(random_topk_indices(T, E, k, seed=seed, skew=skew)).to(DEV)
        gate = torch.rand((T, k), generator=torch.Generator().manual_seed(seed)).to(DEV)
        x = to_bf16(np.random.default_rng(seed).standard_normal((T, H), dtype=np.float32)).to(DEV)
        ws = torch.zeros(api.moe_workspace_bytes(cfg), dtype=torch.uint8, device=DEV)
        api.moe_workspace_init(ws)
        ref = _run(api.moe_permute, cfg, x, idx, gate, (ws,))
        got = _run(api.moe_permute_noalloc, cfg, x, idx, gate, ())
        torch.cuda.synchronize()
        used = int(ref["poffsets"][-1])
        for name in ("counts", "offsets", "poffsets", "slot_row"):
            assert torch.equal(got[name], ref[name]), name
        assert torch.equal(got["row_src"][:used], ref["row_src"][:used])
        assert torch.equal(got["row_gate"][:used], ref["row_gate"][:used])
        assert torch.equal(got["x_perm"][:used].view(torch.int16), ref["x_perm"][:used].view(torch.int16))


def test_noalloc_permute_rejects_shapes_beyond_its_scratch():
    # ceil(T / (256/k)) * E = 1025 * 256 > 262144: refused before any launch
    cfg = api.make_config(1025 * 32, 128, 256, 8, 128)
    with pytest.raises(api.MoeError) as ei:
        api.moe_permute_noalloc(cfg, 16, 16, None, 16, 16, 16, 16, 16, None, 16, 0)
    assert ei.value.code == -4


def test_noalloc_permute_matches_the_oracle_maps():
    """Bit for bit against the oracle's stable counting sort (128-row padding)."""
    api.load()
    T, E, k, H = 3000, 64, 6, 256
    idx_np = random_topk_indices(T, E, k, seed=31, skew=1.1)
    cfg = api.make_config(T, H, E, k, 128)
    x_np = np.random.default_rng(31).standard_normal((T, H), dtype=np.float32)
    x = to_bf16(x_np).to(DEV)
    gate = torch.rand((T, k), generator=torch.Generator().manual_seed(31)).to(DEV)
    got = _run(api.moe_permute_noalloc, cfg, x, torch.from_numpy(idx_np).to(DEV), gate, ())
    torch.cuda.synchronize()
    m = O.permutation_maps(idx_np, E, 128)
    for name in ("counts", "offsets", "poffsets", "slot_row"):
        np.testing.assert_array_equal(got[name].cpu().numpy(), m[name], err_msg=name)
    used = int(m["poffsets"][-1])
    np.testing.assert_array_equal(got["row_src"][:used].cpu().numpy(), m["row_src"])
    valid = m["row_src"] >= 0
    xp = got["x_perm"][:used].view(torch.int16).cpu().numpy()
    xb = x.view(torch.int16).cpu().numpy()
    np.testing.assert_array_equal(xp[valid], xb[m["row_src"][valid]])
    assert np.all(xp[~valid] == 0)                 # padding rows zeroed (zero_pad = 1)
    g = gate.cpu().numpy()
    np.testing.assert_array_equal(got["row_gate"][:used].cpu().numpy()[valid],
                                  g[m["row_src"][valid], m["row_slot"][valid]])


def test_noalloc_permute_drops_out_of_range_pairs():
    """A pair whose expert id is outside [0, E) is dropped: its slot_row entry
    is -1, the counts leave it out, the other pairs keep the rows the oracle
    gives them without it, and nothing past the output buffers is written."""
    api.load()
    T, E, k, H = 500, 16, 4, 128
    idx_np = random_topk_indices(T, E, k, seed=41, skew=0.5)
    bad = [(3, 1, -1), (17, 0, E), (250, 3, E + 1000), (499, 2, -77)]
    for t, i, v in bad:
        idx_np[t, i] = v
    keep = np.ones((T, k), bool)
    for t, i, _ in bad:
        keep[t, i] = False
    cfg = api.make_config(T, H, E, k, 128)
    cap = api.moe_capacity_rows(cfg)
    x = to_bf16(np.random.default_rng(41).standard_normal((T, H), dtype=np.float32)).to(DEV)
    guard = 64                                     # sentinel rows / entries after every output
    counts = torch.full((E + guard,), -7, dtype=torch.int32, device=DEV)
    offsets = torch.full((E + 1 + guard,), -7, dtype=torch.int32, device=DEV)
    poffsets = torch.full((E + 1 + guard,), -7, dtype=torch.int32, device=DEV)
    slot_row = torch.full((T * k + guard,), -7, dtype=torch.int32, device=DEV)
    row_src = torch.full((cap + guard,), -7, dtype=torch.int32, device=DEV)
    row_gate = torch.full((cap + guard,), -7.0, dtype=torch.float32, device=DEV)
    x_perm = torch.full(((cap + guard) * H,), -1, dtype=torch.int16, device=DEV)
    gate = torch.rand((T, k), generator=torch.Generator().manual_seed(41)).to(DEV)
    api.moe_permute_noalloc(cfg, x, torch.from_numpy(idx_np).to(DEV), gate, counts, offsets, poffsets, slot_row,
                            row_src, row_gate, x_perm, 1)
    torch.cuda.synchronize()
    sr = slot_row[:T * k].cpu().numpy().reshape(T, k)
    assert np.all(sr[~keep] == -1)
    cnt = counts[:E].cpu().numpy()
    assert cnt.sum() == T * k - len(bad)
    # the oracle's layout of the remaining pairs: per expert, ascending token
    valid_idx = np.where(keep, idx_np, -1)
    np.testing.assert_array_equal(cnt, np.bincount(valid_idx[keep], minlength=E))
    po = poffsets[:E + 1].cpu().numpy()
    seen = np.zeros(E, np.int64)
    for t in range(T):
        for i in range(k):
            e = valid_idx[t, i]
            if e < 0:
                continue
            assert sr[t, i] == po[e] + seen[e]
            seen[e] += 1
    rs = row_src[:cap].cpu().numpy()
    assert np.all(rs[sr[keep]] == np.nonzero(keep)[0])
    # nothing written past any output
    assert torch.all(counts[E:] == -7) and torch.all(offsets[E + 1:] == -7)
    assert torch.all(poffsets[E + 1:] == -7) and torch.all(slot_row[T * k:] == -7)
    assert torch.all(row_src[cap:] == -7) and torch.all(row_gate[cap:] == -7.0)
    assert torch.all(x_perm[cap * H:] == -1)


def test_noalloc_permute_allocates_nothing():
    """After the first calls (which load the kernels and look up the scratch
    array's address), a call leaves the device's free memory unchanged."""
    api.load()
    T, E, k, H = 2048, 32, 4, 512
    cfg = api.make_config(T, H, E, k, 128)
    idx = torch.from_numpy(random_topk_indices(T, E, k, seed=51, skew=0.8)).to(DEV)
    x = to_bf16(np.random.default_rng(51).standard_normal((T, H), dtype=np.float32)).to(DEV)
    b = _buffers(cfg)
    args = (cfg, x, idx, None, b["counts"], b["offsets"], b["poffsets"], b["slot_row"], b["row_src"], None,
            b["x_perm"], 1)
    for _ in range(2):
        api.moe_permute_noalloc(*args)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    api.moe_permute_noalloc(*args)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
