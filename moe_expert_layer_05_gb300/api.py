"""Python binding of libmoe_gb300.so (ctypes): the C-ABI calls under the same
names, plus a small buffer holder that uses PyTorch only to allocate device
memory and to pick the stream.  Every step of the layer runs in the library's
CUDA kernels; there is no fallback path — if the library is missing or the GPU
is not a GB300 the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MOE_OK = 0
STATUS_NAMES = {0: "ok", -1: "invalid argument", -2: "unsupported", -3: "CUDA error", -4: "workspace too small",
                -5: "bad expert index", -6: "device wait timed out"}
SCORE = {"softmax": 0, "sigmoid": 1}
GEMM_DTYPE = {"bf16": 0, "mxfp8": 1, "nvfp4": 2}

(GG_FC1_SWIGLU, GG_FC2, GG_DGRAD_FC2, GG_DGRAD_FC1, GG_WGRAD_FC1, GG_WGRAD_FC2, GG_FC1_SWIGLU_GATHERED,
 GG_FC2_COMBINE) = range(8)
MX_ROWS, MX_COLS_T, MX_ROWS_GATE_UP, MX_ROWS_G224, MX_COLS_T_G224 = range(5)

c_i32 = ctypes.c_int32
c_vp = ctypes.c_void_p
c_sz = ctypes.c_size_t


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", c_i32), ("H", c_i32), ("E", c_i32), ("k", c_i32), ("F", c_i32), ("S", c_i32),
                ("score", c_i32), ("dtype", c_i32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("w_router", c_vp), ("router_bias", c_vp), ("w1", c_vp), ("w2", c_vp),
                ("w1_shared", c_vp), ("w2_shared", c_vp), ("mx", c_vp)]


class MoeGrads(ctypes.Structure):
    _fields_ = [("dw_router", c_vp), ("dw1", c_vp), ("dw2", c_vp), ("dw1_shared", c_vp), ("dw2_shared", c_vp)]


_LAYOUT_FIELDS = ["logits", "topk_idx", "topk_gate", "counts", "offsets", "poffsets", "slot_row", "row_src",
                  "row_gate", "x_perm", "z", "h", "o", "zs", "hs", "os", "dy_perm", "dz", "dx_perm",
                  "dgate_part", "dlogits", "row_dlogit", "dzs", "dxs", "dz_qt", "dz_qt_sf", "h_qt",
                  "h_qt_sf"]


class MoeActLayout(ctypes.Structure):
    _fields_ = [(n, c_sz) for n in _LAYOUT_FIELDS] + [("total", c_sz), ("cap", c_i32), ("backward", c_i32)]


class MoeGemmArgs(ctypes.Structure):
    _fields_ = [("op", c_i32), ("dense_rows", c_i32), ("a", c_vp), ("b", c_vp), ("c", c_vp), ("c2", c_vp),
                ("aux", c_vp), ("row_gate", c_vp), ("dgate_part", c_vp), ("poffsets", c_vp),
                ("a_scales", c_vp), ("b_scales", c_vp), ("a_amax", c_vp), ("b_amax", c_vp), ("a_rows", c_vp),
                ("slot_row", c_vp), ("b_scale_group", c_i32), ("q_codes", c_vp), ("q_scales", c_vp),
                ("qt_codes", c_vp), ("qt_scales", c_vp)]


_P = ctypes.POINTER
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [c_i32]),
    "moe_version": (c_i32, []),
    "moe_kernel_launches": (ctypes.c_uint64, []),
    "moe_debug_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "moe_capacity_rows": (c_i32, [_P(MoeConfig)]),
    "moe_activation_layout": (c_i32, [_P(MoeConfig), c_i32, _P(MoeActLayout)]),
    "moe_workspace_bytes": (c_sz, [_P(MoeConfig)]),
    "moe_workspace_init": (c_i32, [c_vp, c_sz, c_vp]),
    "moe_read_device_status": (c_i32, [c_vp, _P(c_i32), c_vp]),
    "moe_router_topk": (c_i32, [_P(MoeConfig), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "moe_topk_gating": (c_i32, [_P(MoeConfig), c_vp, c_vp, c_vp, c_vp, c_vp]),
    "moe_permute": (c_i32, [_P(MoeConfig), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32,
                            c_vp, c_vp]),
    "moe_permute_noalloc": (c_i32, [_P(MoeConfig), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                    c_i32, c_vp]),
    "moe_grouped_gemm": (c_i32, [_P(MoeConfig), _P(MoeGemmArgs), c_vp, c_vp]),
    "moe_unpermute": (c_i32, [_P(MoeConfig), c_vp, c_vp, c_vp, c_vp, c_vp]),
    "moe_quantize_mxfp8": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "moe_mxfp8_weights_bytes": (c_sz, [_P(MoeConfig)]),
    "moe_prepare_mxfp8_weights": (c_i32, [_P(MoeConfig), _P(MoeWeights), c_vp, c_sz, c_vp]),
    "moe_quantize_nvfp4": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp]),
    "moe_nvfp4_weights_bytes": (c_sz, [_P(MoeConfig)]),
    "moe_prepare_nvfp4_weights": (c_i32, [_P(MoeConfig), _P(MoeWeights), c_vp, c_sz, c_vp]),
    "moe_layer_forward": (c_i32, [_P(MoeConfig), _P(MoeWeights), c_vp, c_vp, c_vp, c_sz, c_i32, c_vp, c_sz,
                                  c_vp]),
    "moe_layer_backward_dgrad": (c_i32, [_P(MoeConfig), _P(MoeWeights), c_vp, c_vp, c_vp, c_vp, c_vp, c_sz,
                                         c_vp, c_sz, c_vp]),
    "moe_layer_backward_wgrad": (c_i32, [_P(MoeConfig), _P(MoeWeights), c_vp, c_vp, _P(MoeGrads), c_vp, c_sz,
                                         c_vp, c_sz, c_vp]),
}

_lib = None


def library_path() -> str:
    """libmoe_gb300.so built in-tree, or the file MOE_GB300_LIBRARY names."""
    return os.environ.get("MOE_GB300_LIBRARY") or _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libmoe_gb300.so (building it first if absent).  Raises if it cannot."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libmoe_gb300.so not built ({path}); run __graft_entry__.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)} ({code})")
        self.code = code


def check(code: int, what: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, what)


def ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def stream_ptr(stream=None) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def make_config(T, H, E, k, F, S=0, score="softmax", dtype="bf16") -> MoeConfig:
    return MoeConfig(T, H, E, k, F, S, SCORE[score] if isinstance(score, str) else int(score),
                     GEMM_DTYPE[dtype] if isinstance(dtype, str) else int(dtype))


def config_of(workload, tokens: int | None = None) -> MoeConfig:
    w = workload
    return make_config(w.T if tokens is None else tokens, w.H, w.E, w.k, w.F, w.S, w.score, w.dtype)


# ---------------------------------------------------------------- C calls, same names
def moe_capacity_rows(cfg: MoeConfig) -> int:
    return load().moe_capacity_rows(ctypes.byref(cfg))


def moe_activation_layout(cfg: MoeConfig, with_backward: bool) -> MoeActLayout:
    L = MoeActLayout()
    check(load().moe_activation_layout(ctypes.byref(cfg), int(with_backward), ctypes.byref(L)),
          "moe_activation_layout")
    return L


def moe_workspace_bytes(cfg: MoeConfig) -> int:
    return load().moe_workspace_bytes(ctypes.byref(cfg))


def moe_workspace_init(ws: torch.Tensor, stream=None) -> None:
    check(load().moe_workspace_init(ptr(ws), ws.numel() * ws.element_size(), stream_ptr(stream)),
          "moe_workspace_init")


def moe_read_device_status(ws: torch.Tensor, stream=None) -> int:
    code = c_i32(0)
    check(load().moe_read_device_status(ptr(ws), ctypes.byref(code), stream_ptr(stream)), "moe_read_device_status")
    return code.value


def moe_router_topk(cfg, x, w_router, bias, logits, topk_idx, topk_gate, ws, stream=None) -> None:
    check(load().moe_router_topk(ctypes.byref(cfg), ptr(x), ptr(w_router), ptr(bias), ptr(logits), ptr(topk_idx),
                                 ptr(topk_gate), ptr(ws), stream_ptr(stream)), "moe_router_topk")


def moe_topk_gating(cfg, logits, bias, topk_idx, topk_gate, stream=None) -> None:
    check(load().moe_topk_gating(ctypes.byref(cfg), ptr(logits), ptr(bias), ptr(topk_idx), ptr(topk_gate),
                                 stream_ptr(stream)), "moe_topk_gating")


def moe_permute(cfg, x, topk_idx, topk_gate, counts, offsets, poffsets, slot_row, row_src, row_gate, x_perm,
                zero_pad, ws, stream=None) -> None:
    check(load().moe_permute(ctypes.byref(cfg), ptr(x), ptr(topk_idx), ptr(topk_gate), ptr(counts), ptr(offsets),
                             ptr(poffsets), ptr(slot_row), ptr(row_src), ptr(row_gate), ptr(x_perm), int(zero_pad),
                             ptr(ws), stream_ptr(stream)), "moe_permute")


def moe_permute_noalloc(cfg, x, topk_idx, topk_gate, counts, offsets, poffsets, slot_row, row_src, row_gate,
                        x_perm, zero_pad, stream=None) -> None:
    """moe_permute for callers that cannot allocate: no workspace argument;
    the scratch is a fixed 1 MiB device array inside the library."""
    check(load().moe_permute_noalloc(ctypes.byref(cfg), ptr(x), ptr(topk_idx), ptr(topk_gate), ptr(counts),
                                     ptr(offsets), ptr(poffsets), ptr(slot_row), ptr(row_src), ptr(row_gate),
                                     ptr(x_perm), int(zero_pad), stream_ptr(stream)), "moe_permute_noalloc")


def moe_grouped_gemm(cfg, op, a, b, c, ws, c2=None, aux=None, row_gate=None, dgate_part=None, poffsets=None,
                     dense_rows=0, a_scales=None, b_scales=None, a_amax=None, b_amax=None, a_rows=None,
                     slot_row=None, b_scale_group=0, q_codes=None, q_scales=None, qt_codes=None, qt_scales=None,
                     stream=None) -> None:
    args = MoeGemmArgs(op, dense_rows, ptr(a), ptr(b), ptr(c), ptr(c2), ptr(aux), ptr(row_gate), ptr(dgate_part),
                       ptr(poffsets), ptr(a_scales), ptr(b_scales), ptr(a_amax), ptr(b_amax), ptr(a_rows),
                       ptr(slot_row), int(b_scale_group), ptr(q_codes), ptr(q_scales), ptr(qt_codes), ptr(qt_scales))
    check(load().moe_grouped_gemm(ctypes.byref(cfg), ctypes.byref(args), ptr(ws), stream_ptr(stream)),
          "moe_grouped_gemm")


def moe_quantize_mxfp8(src, batch, rows, cols, mode, codes, scales, stream=None) -> None:
    check(load().moe_quantize_mxfp8(ptr(src), batch, rows, cols, mode, ptr(codes), ptr(scales),
                                    stream_ptr(stream)), "moe_quantize_mxfp8")


def moe_mxfp8_weights_bytes(cfg) -> int:
    return int(load().moe_mxfp8_weights_bytes(ctypes.byref(cfg)))


def moe_prepare_mxfp8_weights(cfg, weights: MoeWeights, mx, stream=None) -> None:
    check(load().moe_prepare_mxfp8_weights(ctypes.byref(cfg), ctypes.byref(weights), ptr(mx),
                                           mx.numel() * mx.element_size(), stream_ptr(stream)),
          "moe_prepare_mxfp8_weights")


def moe_quantize_nvfp4(src, batch, rows, cols, mode, codes, scales, amax, stream=None) -> None:
    check(load().moe_quantize_nvfp4(ptr(src), batch, rows, cols, mode, ptr(codes), ptr(scales), ptr(amax),
                                    stream_ptr(stream)), "moe_quantize_nvfp4")


def moe_nvfp4_weights_bytes(cfg) -> int:
    return int(load().moe_nvfp4_weights_bytes(ctypes.byref(cfg)))


def moe_prepare_nvfp4_weights(cfg, weights: MoeWeights, buf, stream=None) -> None:
    check(load().moe_prepare_nvfp4_weights(ctypes.byref(cfg), ctypes.byref(weights), ptr(buf),
                                           buf.numel() * buf.element_size(), stream_ptr(stream)),
          "moe_prepare_nvfp4_weights")


def moe_unpermute(cfg, o_perm, slot_row, shared_out, y, stream=None) -> None:
    check(load().moe_unpermute(ctypes.byref(cfg), ptr(o_perm), ptr(slot_row), ptr(shared_out), ptr(y),
                               stream_ptr(stream)), "moe_unpermute")


def moe_layer_forward(cfg, weights: MoeWeights, x, y, act, with_backward, ws, stream=None) -> None:
    check(load().moe_layer_forward(ctypes.byref(cfg), ctypes.byref(weights), ptr(x), ptr(y), ptr(act),
                                   act.numel() * act.element_size(), int(with_backward), ptr(ws),
                                   ws.numel() * ws.element_size(), stream_ptr(stream)), "moe_layer_forward")


def moe_layer_backward_dgrad(cfg, weights: MoeWeights, x, dy, dx, dgate, act, ws, stream=None) -> None:
    check(load().moe_layer_backward_dgrad(ctypes.byref(cfg), ctypes.byref(weights), ptr(x), ptr(dy), ptr(dx),
                                          ptr(dgate), ptr(act), act.numel() * act.element_size(), ptr(ws),
                                          ws.numel() * ws.element_size(), stream_ptr(stream)),
          "moe_layer_backward_dgrad")


def moe_layer_backward_wgrad(cfg, weights: MoeWeights, x, dy, grads: MoeGrads, act, ws, stream=None) -> None:
    check(load().moe_layer_backward_wgrad(ctypes.byref(cfg), ctypes.byref(weights), ptr(x), ptr(dy),
                                          ctypes.byref(grads), ptr(act), act.numel() * act.element_size(),
                                          ptr(ws), ws.numel() * ws.element_size(), stream_ptr(stream)),
          "moe_layer_backward_wgrad")


# ---------------------------------------------------------------- buffers
class MoELayer:
    """Device buffers for one layer shape (weights are the caller's tensors).

    Owns the activation buffer and the workspace (torch.uint8 device tensors)
    and exposes views of the activation fields for inspection.
    """

    def __init__(self, cfg: MoeConfig, weights: dict, with_backward: bool = False, device="cuda"):
        self.cfg = cfg
        self.with_backward = with_backward
        self.w = weights
        self.layout = moe_activation_layout(cfg, with_backward)
        self.act = torch.empty(self.layout.total, dtype=torch.uint8, device=device)
        self.ws = torch.zeros(max(moe_workspace_bytes(cfg), 256), dtype=torch.uint8, device=device)
        moe_workspace_init(self.ws)
        self.cw = MoeWeights(ptr(weights["w_router"]), ptr(weights.get("bias")), ptr(weights["w1"]),
                             ptr(weights["w2"]), ptr(weights.get("w1_shared")), ptr(weights.get("w2_shared")),
                             None)
        self.mx = None
        if cfg.dtype == GEMM_DTYPE["mxfp8"]:
            self.mx = torch.empty(moe_mxfp8_weights_bytes(cfg), dtype=torch.uint8, device=device)
        elif cfg.dtype == GEMM_DTYPE["nvfp4"]:
            self.mx = torch.empty(moe_nvfp4_weights_bytes(cfg), dtype=torch.uint8, device=device)
        if self.mx is not None:
            self.cw.mx = ptr(self.mx)
            self.prepare_weights()

    def prepare_weights(self, stream=None) -> None:
        """(MXFP8 / NVFP4) quantise the weights into the layer's buffer; call after a weight update."""
        if self.cfg.dtype == GEMM_DTYPE["nvfp4"]:
            moe_prepare_nvfp4_weights(self.cfg, self.cw, self.mx, stream)
        else:
            moe_prepare_mxfp8_weights(self.cfg, self.cw, self.mx, stream)

    def view(self, name: str, dtype, shape) -> torch.Tensor:
        off = getattr(self.layout, name)
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.act[off:off + nbytes].view(dtype).view(*shape)

    def fields(self) -> dict:
        c = self.cfg
        cap = self.layout.cap
        d = {
            "logits": self.view("logits", torch.float32, (c.T, c.E)),
            "topk_idx": self.view("topk_idx", torch.int32, (c.T, c.k)),
            "topk_gate": self.view("topk_gate", torch.float32, (c.T, c.k)),
            "counts": self.view("counts", torch.int32, (c.E,)),
            "offsets": self.view("offsets", torch.int32, (c.E + 1,)),
            "poffsets": self.view("poffsets", torch.int32, (c.E + 1,)),
            "slot_row": self.view("slot_row", torch.int32, (c.T, c.k)),
            "row_src": self.view("row_src", torch.int32, (cap,)),
            "row_gate": self.view("row_gate", torch.float32, (cap,)),
            "x_perm": self.view("x_perm", torch.bfloat16, (cap, c.H)),
            "z": self.view("z", torch.bfloat16, (cap, 2 * c.F)),
            "h": self.view("h", torch.bfloat16, (cap, c.F)),
            "o": self.view("o", torch.bfloat16, (cap, c.H)),
        }
        if self.with_backward:
            d.update({
                "dy_perm": self.view("dy_perm", torch.bfloat16, (cap, c.H)),
                "dz": self.view("dz", torch.bfloat16, (cap, 2 * c.F)),
                "dx_perm": self.view("dx_perm", torch.bfloat16, (cap, c.H)),
                "dlogits": self.view("dlogits", torch.float32, (c.T, c.E)),
            })
        return d

    def forward(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty_like(x)
        moe_layer_forward(self.cfg, self.cw, x, y, self.act, self.with_backward, self.ws, stream)
        return y

    def backward(self, x, dy, grads: dict | None = None, dx=None, dgate=None, stream=None):
        c = self.cfg
        dev = x.device
        if dx is None:
            dx = torch.empty_like(x)
        if dgate is None:
            dgate = torch.empty((c.T, c.k), dtype=torch.float32, device=dev)
        if grads is None:
            grads = {"dw_router": torch.empty((c.E, c.H), dtype=torch.float32, device=dev),
                     "dw1": torch.empty((c.E, 2 * c.F, c.H), dtype=torch.float32, device=dev),
                     "dw2": torch.empty((c.E, c.H, c.F), dtype=torch.float32, device=dev)}
            if c.S > 0:
                grads["dw1_shared"] = torch.empty((2 * c.S, c.H), dtype=torch.float32, device=dev)
                grads["dw2_shared"] = torch.empty((c.H, c.S), dtype=torch.float32, device=dev)
        moe_layer_backward_dgrad(c, self.cw, x, dy, dx, dgate, self.act, self.ws, stream)
        g = MoeGrads(ptr(grads["dw_router"]), ptr(grads["dw1"]), ptr(grads["dw2"]), ptr(grads.get("dw1_shared")),
                     ptr(grads.get("dw2_shared")))
        moe_layer_backward_wgrad(c, self.cw, x, dy, g, self.act, self.ws, stream)
        return dx, dgate, grads


def moe_debug_set_wait_limit_ns(ns: int) -> None:
    """Test hook: the grouped GEMMs' pipeline waits give up after ns (0: 2 s)."""
    load().moe_debug_set_wait_limit_ns(int(ns))


def moe_kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load().moe_kernel_launches())


def moe_status_string(code: int) -> str:
    return load().moe_status_string(int(code)).decode()


def moe_version() -> int:
    return int(load().moe_version())
