"""Shared helpers of the GPU parity tests (comparison metrics, host copies)."""
from __future__ import annotations

import numpy as np
import torch


def f64(t) -> np.ndarray:
    """Exact fp64 copy of a CPU/GPU tensor (bf16 and fp32 widen exactly)."""
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def i64(t) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.int64)


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def max_abs(got, ref) -> float:
    return float(np.max(np.abs(got - ref))) if np.size(ref) else 0.0


def assert_bf16_close(got: np.ndarray, ref: np.ndarray, what: str, rel_l2_tol: float = 4e-3,
                      elem_rel: float = 2.0 ** -7, elem_abs_frac: float = 2e-3):
    """Output rounded once to bf16 from an fp32 accumulation, against fp64.

    Element bound: |got - ref| <= 2^-7 |ref| + 2e-3 * rms(ref) (bf16 keeps 8
    significant bits: rounding alone is <= 2^-8 |ref|; the rest covers fp32
    accumulation order and operands that were themselves bf16-rounded).
    Aggregate bound: rel-L2 <= 4e-3."""
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(got - ref)
    bound = elem_rel * np.abs(ref) + elem_abs_frac * rms + 1e-30
    bad = err > bound
    if bad.any():
        j = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of bound; worst violation err "
                             f"{float(err.flat[j]):.3e} > bound {float(bound.flat[j]):.3e} at ref "
                             f"{float(ref.flat[j]):.3e}; max err {float(err.max()):.3e}, rms {rms:.3e}")
    r = rel_l2(got, ref)
    assert r <= rel_l2_tol, f"{what}: rel-L2 {r:.3e} > {rel_l2_tol}"
    return r


class LazyExperts:
    """Per-expert fp64 view of a [E, ...] device tensor, copied on demand."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.shape = tuple(t.shape)
        self._cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self._cache:
            self._cache[e] = f64(self.t[e])
        return self._cache[e]
