"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function the public header declares, sizes and layouts are consistent,
and bad arguments are rejected before any launch."""
import ctypes
import os
import re

import pytest
import torch

from moe_expert_layer_05_gb300 import api

# Calls whose arguments pass every check reach the device check; on a machine
# without a GPU that is where they stop.  Those asserts use fake device
# pointers, so they run only where no GPU could launch anything with them.
NO_GPU = not torch.cuda.is_available()

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_gb300.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_function_is_exported():
    lib = api.load()
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    # and the binding wraps each under the same name
    for n in names:
        assert hasattr(api, n), f"binding lacks {n}"


def test_status_strings_and_version():
    lib = api.load()
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.moe_status_string(code)
    assert lib.moe_version() > 0


@pytest.mark.parametrize("T,H,E,k,F,S", [(4096, 4096, 8, 2, 14336, 0), (8192, 7168, 256, 8, 2048, 2048),
                                         (0, 128, 8, 2, 128, 0), (1, 128, 8, 8, 128, 128)])
def test_layout_is_consistent(T, H, E, k, F, S):
    cfg = api.make_config(T, H, E, k, F, S)
    cap = api.moe_capacity_rows(cfg)
    assert cap % 128 == 0 and cap >= T * k + 127 * E
    for bwd in (False, True):
        L = api.moe_activation_layout(cfg, bwd)
        assert L.cap == cap
        fields = [(n, getattr(L, n)) for n, _ in api.MoeActLayout._fields_[:-3]]
        used = sorted(v for n, v in fields if v != (1 << 64) - 1)
        assert used == sorted(set(used)), "fields overlap"
        assert all(v % 256 == 0 for v in used)
        assert L.total >= used[-1]
        assert (L.dz != (1 << 64) - 1) == bwd
    assert api.moe_workspace_bytes(cfg) >= 256


@pytest.mark.parametrize("bad", [dict(k=0), dict(k=9, E=8), dict(E=300, k=2), dict(H=100), dict(F=200),
                                 dict(S=64), dict(T=-1), dict(k=33, E=64)])
def test_bad_configs_rejected(bad):
    base = dict(T=16, H=128, E=8, k=2, F=128, S=0)
    base.update(bad)
    cfg = api.make_config(**base)
    assert api.moe_capacity_rows(cfg) == -1
    assert api.moe_workspace_bytes(cfg) == 0
    L = api.MoeActLayout()
    assert api.load().moe_activation_layout(ctypes.byref(cfg), 0, ctypes.byref(L)) == -1


def test_null_and_misaligned_pointers_rejected_before_launch():
    lib = api.load()
    cfg = api.make_config(16, 128, 8, 2, 128)
    w = api.MoeWeights(None, None, None, None, None, None)
    assert lib.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(w), 16, 16, 16, 1 << 30, 0, 16, 1 << 20,
                                 None) == -1
    w = api.MoeWeights(16, None, 16, 16, None, None)
    # misaligned x
    assert lib.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(w), 17, 16, 16, 1 << 30, 0, 16, 1 << 20,
                                 None) == -1
    # activation buffer too small
    assert lib.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(w), 16, 16, 16, 64, 0, 16, 1 << 20, None) == -4
    args = api.MoeGemmArgs(0, 0, 16, 16, 16, None, None, None, None, None)  # routed without offsets
    assert lib.moe_grouped_gemm(ctypes.byref(cfg), ctypes.byref(args), 16, None) == -1
    args = api.MoeGemmArgs(9, 16, 16, 16, 16, None, None, None, None, None)
    assert lib.moe_grouped_gemm(ctypes.byref(cfg), ctypes.byref(args), 16, None) == -1   # unknown op


def test_nvfp4_config_rules_and_sizes():
    """NVFP4 layers: T % 128, H/F/S % 256; their workspace holds the E2M1 codes
    (half a byte per element) and E4M3 scales (one byte per 16); the weight
    buffer likewise; backward calls and NVFP4 backward GEMM ops are refused
    before any launch."""
    lib = api.load()
    ok = api.make_config(256, 256, 8, 2, 512, 0, dtype="nvfp4")
    assert api.moe_capacity_rows(ok) > 0
    for bad in (dict(H=128), dict(F=384), dict(S=128), dict(T=100)):
        kw = dict(T=256, H=256, E=8, k=2, F=512, S=0)
        kw.update(bad)
        assert api.moe_capacity_rows(api.make_config(dtype="nvfp4", **kw)) == -1, bad
    bf = api.make_config(256, 256, 8, 2, 512, 0)
    cap = api.moe_capacity_rows(ok)
    extra = api.moe_workspace_bytes(ok) - api.moe_workspace_bytes(bf)
    assert extra >= (cap * 256 + cap * 512 + 256 * 256) * (1 / 2 + 1 / 16)
    wb = api.moe_nvfp4_weights_bytes(ok)
    assert wb >= 8 * (2 * 512 * 256 + 256 * 512) * (1 / 2 + 1 / 16)
    assert api.moe_nvfp4_weights_bytes(bf) == 0
    w = api.MoeWeights(16, None, 16, 16, None, None, 16)
    assert lib.moe_layer_forward(ctypes.byref(ok), ctypes.byref(w), 16, 16, 16, 1 << 40, 1, 16, 1 << 40,
                                 None) == -2
    assert lib.moe_layer_backward_dgrad(ctypes.byref(ok), ctypes.byref(w), 16, 16, 16, None, 16, 1 << 40, 16,
                                        1 << 40, None) == -2
    # quantiser argument checks: cols % 64, rows % 128, known mode, amax pointer
    assert lib.moe_quantize_nvfp4(16, 1, 128, 96, 0, 16, 16, 16, None) == -1
    assert lib.moe_quantize_nvfp4(16, 1, 100, 64, 0, 16, 16, 16, None) == -1
    assert lib.moe_quantize_nvfp4(16, 1, 128, 64, 1, 16, 16, 16, None) == -1
    assert lib.moe_quantize_nvfp4(16, 1, 128, 64, 0, 16, 16, None, None) == -1


def test_gathered_fc1_arguments_checked_before_launch():
    """MOE_GG_FC1_SWIGLU_GATHERED needs the row map (a_rows) and a routed call;
    MXFP8 / NVFP4 layers do not offer it."""
    lib = api.load()
    cfg = api.make_config(256, 128, 8, 2, 256)
    no_rows = api.MoeGemmArgs(api.GG_FC1_SWIGLU_GATHERED, 0, 16, 16, 16, None, None, None, None, 16)
    assert lib.moe_grouped_gemm(ctypes.byref(cfg), ctypes.byref(no_rows), 16, None) == -1
    dense = api.MoeGemmArgs(api.GG_FC1_SWIGLU_GATHERED, 128, 16, 16, 16, None, None, None, None, 16)
    dense.a_rows = 16
    assert lib.moe_grouped_gemm(ctypes.byref(cfg), ctypes.byref(dense), 16, None) == -1
    for dt in ("mxfp8", "nvfp4"):
        c = api.make_config(256, 256, 8, 2, 256, dtype=dt)
        a = api.MoeGemmArgs(api.GG_FC1_SWIGLU_GATHERED, 0, 16, 16, 16, None, None, None, None, 16, 16, 16, 16, 16, 16)
        assert lib.moe_grouped_gemm(ctypes.byref(c), ctypes.byref(a), 16, None) == -1


def test_low_precision_gemm_arguments_checked_before_launch():
    """MXFP8 / NVFP4 grouped GEMMs need their scale tiles (and NVFP4 the tensor
    amaxes); NVFP4 offers the forward ops only (MOE_ERR_UNSUPPORTED for the
    rest); dense calls need whole 128-row scale tiles."""
    lib = api.load()
    nv = api.make_config(256, 256, 8, 2, 256, dtype="nvfp4")
    mx = api.make_config(256, 256, 8, 2, 256, dtype="mxfp8")

    def call(cfg, op, dense_rows=0, scales=16, amax=16):
        a = api.MoeGemmArgs(op, dense_rows, 16, 16, 16, None, 16, None, None, 16, scales, scales, amax, amax)
        return lib.moe_grouped_gemm(ctypes.byref(cfg), ctypes.byref(a), 16, None)

    assert call(nv, api.GG_FC1_SWIGLU, scales=None) == -1
    assert call(nv, api.GG_FC2, amax=None) == -1
    assert call(nv, api.GG_FC2, amax=18) == -1                 # misaligned fp32
    for op in (api.GG_DGRAD_FC2, api.GG_DGRAD_FC1, api.GG_WGRAD_FC1, api.GG_WGRAD_FC2):
        assert call(nv, op) == -2
    assert call(mx, api.GG_FC2, scales=None) == -1
    assert call(mx, api.GG_FC1_SWIGLU, dense_rows=100) == -1
    # B scale tiles grouped by 224 rows: MXFP8 FC2 / DGRAD_FC1 / WGRAD_FC1 / WGRAD_FC2 (F % 256 == 0),
    # routed, H % 224 == 0 only
    mx224 = api.make_config(256, 896, 8, 2, 256, dtype="mxfp8")
    bf224 = api.make_config(256, 896, 8, 2, 256)

    def call_g(cfg, op, group, dense_rows=0):
        a = api.MoeGemmArgs(op, dense_rows, 16, 16, 16, None, 16, None, None, 16, 16, 16, 16, 16)
        a.b_scale_group = group
        return lib.moe_grouped_gemm(ctypes.byref(cfg), ctypes.byref(a), 16, None)

    assert call_g(mx, api.GG_FC2, 224) == -1                   # H = 256
    assert call_g(mx224, api.GG_FC2, 100) == -1
    assert call_g(mx224, api.GG_FC1_SWIGLU, 224) == -1
    assert call_g(api.make_config(256, 896, 8, 2, 384, dtype="mxfp8"), api.GG_WGRAD_FC2, 224) == -1   # F % 256
    assert call_g(mx224, api.GG_FC2, 224, dense_rows=128) == -1
    assert call_g(bf224, api.GG_FC2, 224) == -1
    if NO_GPU:
        for op in (api.GG_FC2, api.GG_DGRAD_FC1, api.GG_WGRAD_FC1, api.GG_WGRAD_FC2):   # accepted: device check left
            assert call_g(mx224, op, 224) != -1
    # dz's MXFP8 copies: MXFP8 DGRAD_FC2 only, routed, F % 256 == 0, both pointers of a pair
    def call_q(cfg, op, dense_rows=0, **kw):
        a = api.MoeGemmArgs(op, dense_rows, 16, 16, 16, None, 16, None, None, 16, 16, 16, 16, 16)
        for k_, v in kw.items():
            setattr(a, k_, v)
        return lib.moe_grouped_gemm(ctypes.byref(cfg), ctypes.byref(a), 16, None)

    both = dict(q_codes=16, q_scales=16, qt_codes=16, qt_scales=16)
    if NO_GPU:
        assert call_q(mx, api.GG_DGRAD_FC2, **both) != -1             # F = 256: accepted
        assert call_q(mx, api.GG_DGRAD_FC2, c=None, **both) != -1     # no bf16 dz: both copies asked
    assert call_q(mx, api.GG_DGRAD_FC2, q_codes=16) == -1             # half a pair
    assert call_q(mx, api.GG_DGRAD_FC2, c=None, q_codes=16, q_scales=16) == -1
    assert call_q(mx, api.GG_FC2, **both) == -1
    assert call_q(mx, api.GG_FC1_SWIGLU, dense_rows=128, **both) == -1     # routed only
    assert call_q(api.make_config(256, 256, 8, 2, 256), api.GG_FC1_SWIGLU, **both) == -1
    if NO_GPU:
        assert call_q(mx, api.GG_FC1_SWIGLU, **both) != -1                  # h''s copies: accepted
        assert call_q(mx, api.GG_FC1_SWIGLU, c=None, q_codes=16, q_scales=16) != -1
    assert call_q(mx, api.GG_DGRAD_FC2, dense_rows=128, **both) == -1
    assert call_q(api.make_config(256, 256, 8, 2, 256), api.GG_DGRAD_FC2, **both) == -1
    assert call_q(api.make_config(256, 256, 8, 2, 384, dtype="mxfp8"), api.GG_DGRAD_FC2, **both) == -1
    assert lib.moe_quantize_mxfp8(16, 1, 200, 128, api.MX_ROWS_G224, 16, 16, None) == -1
    assert lib.moe_quantize_mxfp8(16, 1, 128, 256, api.MX_COLS_T_G224, 16, 16, None) == -1
