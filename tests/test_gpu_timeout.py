"""The bounded-wait failure path of the grouped GEMMs, made to run on the GPU
without a hang: every pipeline wait is limited (moe_debug_set_wait_limit_ns),
so a launch whose waits cannot be met in time gives up, lets its in-flight
copies and MMAs finish, frees its TMEM and records MOE_ERR_TIMEOUT in the
status word; the next launch with the default limit computes correctly in the
same context.  Nothing waits on a flag that nothing sets: the waits are the
kernel's own, only their limit is 1 ns."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_bf16_close, f64
from moe_expert_layer_05_gb300 import api
from moe_expert_layer_05_gb300.inputs import random_topk_indices, to_bf16
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_grouped_gemm_wait_limit_gives_timeout_status_and_the_context_recovers(lib):
    # fc2 on one-CTA 256-row tiles with a long contraction (K = 16384: hundreds
    # of k-blocks per tile), so the epilogue's wait for a finished accumulator
    # and the producer's wait for a free stage both outlast any short limit
    T, H, E, k, F = 1024, 512, 4, 2, 16384
    idx = random_topk_indices(T, E, k, seed=61)
    m = O.permutation_maps(idx, E, 128)
    cfg = api.make_config(T, H, E, k, F)
    cap = api.moe_capacity_rows(cfg)
    used = int(m["poffsets"][-1])
    rng = np.random.default_rng(62)
    h = rng.standard_normal((cap, F), dtype=np.float32)
    h[used:] = 0.0
    h[:used][m["row_src"] < 0] = 0.0
    h = to_bf16(h).to(DEV)
    w2 = to_bf16(rng.standard_normal((E, H, F), dtype=np.float32) * np.float32(0.02)).to(DEV)
    po = torch.from_numpy(m["poffsets"].astype(np.int32)).to(DEV)
    ws = torch.zeros(api.moe_workspace_bytes(cfg), dtype=torch.uint8, device=DEV)
    api.moe_workspace_init(ws)
    o = torch.zeros((cap, H), dtype=torch.bfloat16, device=DEV)
    api.moe_debug_set_wait_limit_ns(1)
    try:
        api.moe_grouped_gemm(cfg, api.GG_FC2, h, w2, o, ws, poffsets=po)
        torch.cuda.synchronize()
    finally:
        api.moe_debug_set_wait_limit_ns(0)
    assert api.moe_read_device_status(ws) == -6            # MOE_ERR_TIMEOUT
    words = ws[:256].view(torch.int32).cpu()
    assert int(words[32]) == 0 and int(words[33]) == 0      # the tile counter is back at zero
    # the same context, the default limit: a complete and correct result
    api.moe_workspace_init(ws)
    o.zero_()
    api.moe_grouped_gemm(cfg, api.GG_FC2, h, w2, o, ws, poffsets=po)
    torch.cuda.synchronize()
    assert api.moe_read_device_status(ws) == 0
    w2_64 = f64(w2)
    ref = O.expert_fc2(f64(h)[:used], w2_64, m["poffsets"])
    assert_bf16_close(f64(o)[:used], ref, "o after recovery")
