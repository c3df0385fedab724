"""The permutation entry point for callers that cannot allocate device memory
(moe_permute_noalloc: no workspace argument, scratch in a fixed device array
owned by the library).  Checked through the C ABI against moe_permute, which
uses a caller-provided workspace, on two calls in a row: the second call has a
different shape and routing, so anything it wrongly kept from the first call's
scratch would show.  Collected last on purpose."""
import numpy as np
import pytest
import torch

from moe_expert_layer_05_gb300 import api
from moe_expert_layer_05_gb300.inputs import random_topk_indices, to_bf16

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
