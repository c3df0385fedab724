"""Seeded synthetic inputs for the MoE expert layer (shared by the tests, the
oracle checks and the benchmark).

This module draws random numbers and casts them to the storage types; it holds
none of the layer's arithmetic.  Each tensor comes from its own numpy PCG64
stream (``64*seed + slot``), so a tensor does not change when another one is
added or resized.  The workloads are the layer shapes that the Megatron Core MoE
summary ("Scalable Training of Mixture-of-Experts Models with Megatron Core",
section 3, results table) trains: Mixtral-, Qwen3-235B- and DeepSeek-V3-like
layers, plus a tiny case that the fp64 oracle finishes in well under a second.
No dataset is used: x ~ N(0,1), weights ~ N(0, 0.02), upstream grad ~ N(0,1).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int           # tokens
    H: int           # hidden size
    E: int           # routed experts
    k: int           # experts per token
    F: int           # routed expert SwiGLU ffn size
    S: int = 0       # shared expert ffn size (0: no shared expert)
    score: str = "softmax"   # "softmax" or "sigmoid"
    zipf_s: float = 0.0      # >0: router bias ~ Zipf(s) over experts (sigmoid only)
    dtype: str = "bf16"      # expert GEMM operand type: "bf16", "mxfp8" or "nvfp4" (forward only)
    backward: bool = False

    def as_dict(self) -> dict:
        return dataclasses.asdict(self)


WORKLOADS = {
    "tiny": Workload("tiny", T=256, H=128, E=8, k=2, F=256),
    "mixtral": Workload("mixtral", T=4096, H=4096, E=8, k=2, F=14336),
    "qwen3": Workload("qwen3", T=8192, H=4096, E=128, k=8, F=1536, backward=True),
    "dsv3": Workload("dsv3", T=8192, H=7168, E=256, k=8, F=2048, S=2048,
                     score="sigmoid", zipf_s=1.2),
    "dsv3_mxfp8": Workload("dsv3_mxfp8", T=16384, H=7168, E=256, k=8, F=2048, S=2048,
                           score="sigmoid", zipf_s=1.2, dtype="mxfp8", backward=True),
    # NVFP4 expert GEMMs (forward): the Mixtral-like layer, and a small case for the oracle
    "mixtral_nvfp4": Workload("mixtral_nvfp4", T=4096, H=4096, E=8, k=2, F=14336, dtype="nvfp4"),
    "tiny_nvfp4": Workload("tiny_nvfp4", T=256, H=256, E=8, k=2, F=512, dtype="nvfp4"),
}

# Weight of the router bias: b_e = ZIPF_C * ln(E * p_e), p_e ∝ rank_e^(-s).
ZIPF_C = 0.05

_SLOTS = {"x": 0, "w_router": 1, "w1": 2, "w2": 3, "w1_shared": 4, "w2_shared": 5, "dy": 6}


def _normal(seed: int, slot: str, shape, std: float) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed * 64 + _SLOTS[slot]))
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """Round a float32 array to bfloat16 (round-to-nearest-even, torch's cast)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def zipf_router_bias(E: int, s: float, c: float = ZIPF_C) -> np.ndarray:
    """Per-expert selection bias that makes a few experts hot.

    rank = a fixed random permutation of 1..E (seed 1); p_e ∝ rank_e^-s;
    b_e = c * ln(E * p_e).  Returned as float32 (the router keeps fp32 state).
    """
    rank = np.random.default_rng(1).permutation(E).astype(np.float64) + 1.0
    p = rank ** (-s)
    p /= p.sum()
    return (c * np.log(E * p)).astype(np.float32)


def make_inputs(w: Workload, seed: int = 0, with_dy: bool | None = None,
                tokens: int | None = None) -> dict:
    """CPU tensors for one layer call: bf16 activations and weights, fp32 bias.

    ``tokens`` overrides T (same weights, fewer rows of x / dy).
    """
    T = w.T if tokens is None else tokens
    H, E, F, S = w.H, w.E, w.F, w.S
    out = {
        "x": to_bf16(_normal(seed, "x", (T, H), 1.0)),
        "w_router": to_bf16(_normal(seed, "w_router", (E, H), 0.02)),
        "w1": to_bf16(_normal(seed, "w1", (E, 2 * F, H), 0.02)),
        "w2": to_bf16(_normal(seed, "w2", (E, H, F), 0.02)),
        "bias": None,
        "w1_shared": None,
        "w2_shared": None,
        "dy": None,
    }
    if w.zipf_s > 0:
        out["bias"] = torch.from_numpy(zipf_router_bias(E, w.zipf_s))
    if S > 0:
        out["w1_shared"] = to_bf16(_normal(seed, "w1_shared", (2 * S, H), 0.02))
        out["w2_shared"] = to_bf16(_normal(seed, "w2_shared", (H, S), 0.02))
    if with_dy if with_dy is not None else w.backward:
        out["dy"] = to_bf16(_normal(seed, "dy", (T, H), 1.0))
    return out


def make_inputs_on_device(w: Workload, device, seed: int = 0, with_dy: bool | None = None) -> dict:
    """Same recipe as make_inputs, drawn directly on ``device`` by torch's
    generator (a different stream from the CPU one).  Used where the CPU copy of
    a multi-GB weight set would be slow to draw; tests copy back what the oracle
    needs, so both sides still see identical values."""
    gen = torch.Generator(device=device)
    T, H, E, F, S = w.T, w.H, w.E, w.F, w.S

    def normal(slot, shape, std):
        gen.manual_seed(seed * 64 + _SLOTS[slot])
        t = torch.empty(shape, dtype=torch.float32, device=device)
        t.normal_(0.0, std, generator=gen)
        return t.to(torch.bfloat16)

    out = {
        "x": normal("x", (T, H), 1.0),
        "w_router": normal("w_router", (E, H), 0.02),
        "w1": normal("w1", (E, 2 * F, H), 0.02),
        "w2": normal("w2", (E, H, F), 0.02),
        "bias": None, "w1_shared": None, "w2_shared": None, "dy": None,
    }
    if w.zipf_s > 0:
        out["bias"] = torch.from_numpy(zipf_router_bias(E, w.zipf_s)).to(device)
    if S > 0:
        out["w1_shared"] = normal("w1_shared", (2 * S, H), 0.02)
        out["w2_shared"] = normal("w2_shared", (H, S), 0.02)
    if with_dy if with_dy is not None else w.backward:
        out["dy"] = normal("dy", (T, H), 1.0)
    return out


def make_router_inputs_on_device(w: Workload, device, seed: int = 0) -> dict:
    """x, the router weight and (sigmoid workloads) the router bias of
    make_inputs_on_device, without the expert weights: for runs that time the
    routing and permutation alone."""
    gen = torch.Generator(device=device)

    def normal(slot, shape, std):
        gen.manual_seed(seed * 64 + _SLOTS[slot])
        t = torch.empty(shape, dtype=torch.float32, device=device)
        t.normal_(0.0, std, generator=gen)
        return t.to(torch.bfloat16)

    return {"x": normal("x", (w.T, w.H), 1.0), "w_router": normal("w_router", (w.E, w.H), 0.02),
            "bias": torch.from_numpy(zipf_router_bias(w.E, w.zipf_s)).to(device) if w.zipf_s > 0 else None}


def random_topk_indices(T: int, E: int, k: int, seed: int = 0, skew: float = 0.0) -> np.ndarray:
    """Routing indices drawn directly (no router): k distinct experts per token.

    skew > 0 biases toward low expert ids (weights ∝ (e+1)^-skew), which makes
    some experts empty and some hot.  Used by the permutation tests and the
    router-replay path."""
    rng = np.random.Generator(np.random.PCG64(seed * 64 + 7))
    p = (np.arange(E, dtype=np.float64) + 1.0) ** (-skew)
    p /= p.sum()
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        out[t] = rng.choice(E, size=k, replace=False, p=p)
    return out
