"""Shared helpers of the GPU parity tests (comparison metrics, host copies)."""
from __future__ import annotations

import concurrent.futures as cf

import numpy as np
import torch

from oracle import moe_oracle as O


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


class StreamExperts:
    """Per-expert view of a [E, ...] device tensor, copied to the host (fp32,
    exact for bf16) on every access and never kept: for oracle runs over many
    large experts."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        return self.t[int(e)].to("cpu", torch.float32).numpy()


def mx_weight_cache(w1: torch.Tensor, w2: torch.Tensor, experts, w1s=None, w2s=None, threads: int = 8) -> dict:
    """The oracle's MX weight cache ((name, expert, axis) -> quantise-dequantise
    of that weight along axis) for the given experts and the shared expert,
    each entry made by the oracle's own quantiser; the entries are independent,
    so they are made in parallel threads (numpy releases the GIL in its loops)."""
    jobs = []
    for e in sorted({int(e) for e in experts}):
        for axis in (-1, 0):
            jobs += [("w1", e, w1, axis), ("w2", e, w2, axis)]
    if w1s is not None:
        for axis in (-1, 0):
            jobs += [("w1s", 0, w1s, axis), ("w2s", 0, w2s, axis)]

    def run(job):
        name, e, t, axis = job
        src = t if name in ("w1s", "w2s") else t[e]
        return (name, e, axis), O.mxfp8_roundtrip(f64(src), axis)

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        return dict(ex.map(run, jobs))


def check_full_permutation(w, fl, x, n_rows=4096, seed=0, rows=True):
    """The layer's permutation at its full T against the oracle's counting sort
    run on the GPU's own routing: counts, offsets, padded offsets, slot_row,
    row_src and row_gate bit for bit over every pair; x_perm bit for bit on a
    seeded sample of rows (every padding row of the sample must be zero when
    the layer trains)."""
    idx = i64(fl["topk_idx"])
    m = O.permutation_maps(idx, w.E, 128)
    for name in ("counts", "offsets", "poffsets", "slot_row"):
        np.testing.assert_array_equal(i64(fl[name]), m[name], err_msg=name)
    used = int(m["poffsets"][-1])
    np.testing.assert_array_equal(i64(fl["row_src"][:used]), m["row_src"])
    valid = m["row_src"] >= 0
    rg = fl["row_gate"][:used].view(torch.int32).cpu().numpy()
    tg = fl["topk_gate"].view(torch.int32).cpu().numpy()
    np.testing.assert_array_equal(rg[valid], tg[m["row_src"][valid], m["row_slot"][valid]])
    assert np.all(rg[~valid] == 0)
    if not rows:            # (quantised layers permute codes, not bf16 rows)
        return m
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(used, size=min(n_rows, used), replace=False))
    rows_t = torch.from_numpy(rows).to(x.device)
    xp = fl["x_perm"][rows_t].view(torch.int16).cpu().numpy()
    v = valid[rows]
    src = torch.from_numpy(m["row_src"][rows][v]).to(x.device)
    np.testing.assert_array_equal(xp[v], x[src].view(torch.int16).cpu().numpy())
    return m


