#!/usr/bin/env python3
"""Throughput of the MoE expert layer on GB300 (one JSON line on rank 0).

A step is one pass of the layer over one batch: router GEMM, top-k gating,
sync-free permutation, grouped-GEMM SwiGLU experts with the gate applied at the
activation, combine, plus the data and weight gradients for the workloads that
train.  Seeded synthetic inputs of the layer shapes the Megatron Core MoE
summary trains (Mixtral-, Qwen3- and DeepSeek-V3-like layers).

With no --workload the run measures all five configurations one after the
other (tiny, Mixtral-like, Qwen3-like training, DeepSeek-like bf16 forward,
DeepSeek-like MXFP8 training) and prints one line whose headline is the
largest, the DeepSeek-like MXFP8 training layer (T=16384, H=7168, E=256 + one
shared expert, k=8, F=2048); the other four are complete sub-records under
"configs".  Under torchrun (N>1) every rank runs the headline only.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events on
the launching stream, with L2 flushed (a 512 MB write) before every step outside
the events; barrier + synchronize on both sides; the max over ranks.  Every rank
runs its own tokens through replicated experts (no data-path collective): weak
scaling.  The end-to-end figure (e2e) streams K batches from pinned host memory
and reads every result back, on two copy streams with double-buffered device
inputs.  Each grouped GEMM of the step is then timed alone on the same inputs
and set against its roofline: max(flops / tensor peak, algorithmic bytes / HBM
bandwidth), both terms reported.  nvidia-smi samples the clocks from the first
warm-up step to the end of the end-to-end leg.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import dataclasses
import gc
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from moe_expert_layer_05_gb300.inputs import (WORKLOADS, make_inputs, make_inputs_on_device,  # noqa: E402
                                              make_router_inputs_on_device)

METRIC = "MoE layer tokens/s on 1 GB300; grouped-GEMM TFLOPS as % of tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 512 << 20
HEADLINE = "dsv3_mxfp8"
SUITE = ("tiny", "mixtral", "qwen3", "dsv3", HEADLINE)
# DRAM traffic of one launch of a grouped GEMM (dram__bytes_read.sum +
# dram__bytes_write.sum, one ncu pass) over its algorithmic bytes, captured on
# a case with the workload's rows per expert and fewer experts, so the ratio
# carries to the full launch (traffic grows with the experts):
# (workload, op) -> (ratio, capture).
_CAP_MX = "ncu 2026-12-03, T=4096 E=64 (512 rows per expert, as at full size)"
TRAFFIC = {
    ("dsv3_mxfp8", "fc1"): (1.0504, _CAP_MX),
    ("dsv3_mxfp8", "fc2"): (1.0344, _CAP_MX),
    ("dsv3_mxfp8", "dgrad_fc2"): (1.1201, _CAP_MX),
    ("dsv3_mxfp8", "dgrad_fc1"): (1.0314, _CAP_MX),
    ("dsv3_mxfp8", "wgrad_fc1"): (1.0047, _CAP_MX),
    ("dsv3_mxfp8", "wgrad_fc2"): (0.9979, _CAP_MX),
    ("qwen3", "wgrad_fc1"): (0.9831, "ncu 2026-12-03, T=2048 E=32 (512 rows per expert, as at full size)"),
    ("dsv3", "fc1"): (1.0709, "ncu 2026-12-03, T=2048 E=64 (256 rows per expert, as at full size)"),
    ("mixtral", "fc1"): (1.0463, "ncu 2026-12-03, T=2048 E=4 (1024 rows per expert, as at full size)"),
}


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, use_cuda: bool):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend="nccl" if use_cuda else "gloo")


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(v: float, world: int, device) -> float:
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, steps: int, world: int, max_total_ms: float) -> float:
    """Whole-job throughput: tokens all ranks processed / slowest rank's time."""
    return world * tokens_per_rank * steps / (max_total_ms / 1e3)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms.  A sample is 'under load' when the
    board draws at least 1.5x the lowest power seen in the run."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines: list[str] = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]),
                             {n for n, v in zip(self.REASONS, parts[5:9]) if v.lower() == "active"}))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_under_load": 0}
        p_min = min(r[2] for r in rows)
        load = [r for r in rows if r[2] >= 1.5 * p_min] or rows
        reasons = set()
        for r in load:
            reasons |= r[3]
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "reasons": sorted(reasons), "samples": len(rows),
                "samples_under_load": len(load)}


def read_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- oracle timing (CPU)
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class _HostExperts:
    """Expert weights as fp64 numpy (exact bf16 values), filled for the experts
    a sample needs before any timing, so the timed oracle call converts nothing."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.shape = tuple(t.shape)
        self.c = {}

    def fill(self, e: int):
        if e not in self.c:
            self.c[e] = self.t[e].to("cpu", torch.float32).numpy().astype(np.float64)
        return self.c[e]

    def __getitem__(self, e):
        return self.c[int(e)] if int(e) in self.c else self.fill(int(e))


def _oracle_fns(w):
    from oracle import moe_oracle as O
    if w.dtype == "mxfp8":
        return O.moe_forward_mx, O.moe_backward_mx
    if w.dtype == "nvfp4":
        return O.moe_forward_nvfp4, None         # forward-only workloads
    return O.moe_forward, O.moe_backward


def oracle_inputs(w, dinp) -> dict:
    def npf(t):
        return None if t is None else t.to("cpu", torch.float32).numpy().astype(np.float64)
    return {"x_np": npf(dinp["x"]), "wr_np": npf(dinp["w_router"]), "bias_np": npf(dinp["bias"]),
            "w1s_np": npf(dinp["w1_shared"]), "w2s_np": npf(dinp["w2_shared"]), "dy_np": npf(dinp["dy"]),
            "w1": _HostExperts(dinp["w1"]), "w2": _HostExperts(dinp["w2"]), "wcache": {}}


def sample_experts(w, inp, tokens) -> np.ndarray:
    from oracle import moe_oracle as O
    logits = O.router_logits(inp["x_np"][tokens], inp["wr_np"])
    idx, _ = O.route(logits, w.k, w.score, inp["bias_np"])
    return np.unique(idx)


def warm_experts(w, inp, experts, threads: int | None = None):
    """Untimed preparation of what the timed oracle call reads: fp64 host
    copies of the given experts' weights, and for the quantised recipes the
    weights quantised once (as the recipe does), in parallel threads."""
    from oracle import moe_oracle as O
    for e in experts:
        inp["w1"].fill(int(e))
        inp["w2"].fill(int(e))
    jobs = []
    if w.dtype == "mxfp8":
        for e in experts:
            for name in ("w1", "w2"):
                for axis in (-1, 0):
                    if (name, int(e), axis) not in inp["wcache"]:
                        jobs.append((name, int(e), axis, inp[name][int(e)]))
        if inp["w1s_np"] is not None:
            for name, W in (("w1s", inp["w1s_np"]), ("w2s", inp["w2s_np"])):
                for axis in (-1, 0):
                    if (name, 0, axis) not in inp["wcache"]:
                        jobs.append((name, 0, axis, W))

        def run(j):
            return (j[0], j[1], j[2]), O.mxfp8_roundtrip(j[3], j[2])

        with cf.ThreadPoolExecutor(max_workers=threads or min(8, host_cores())) as ex:
            inp["wcache"].update(dict(ex.map(run, jobs)))
    elif w.dtype == "nvfp4":
        for e in experts:
            O.nvfp4_weight(inp["wcache"], "w1", inp["w1"], int(e))
            O.nvfp4_weight(inp["wcache"], "w2", inp["w2"], int(e))


def oracle_step_timed(w, inp, tokens: np.ndarray) -> float:
    """One step of the oracle (forward, plus backward for training workloads)
    on the given tokens, with everything it reads already on the host; seconds."""
    fwd_fn, bwd_fn = _oracle_fns(w)
    x = inp["x_np"][tokens]
    sh = dict(w1_shared=inp["w1s_np"], w2_shared=inp["w2s_np"])
    if w.dtype != "bf16":
        sh["weight_cache"] = inp["wcache"]      # weights quantised once, as the recipe does
    t0 = time.perf_counter()
    fwd = fwd_fn(x, inp["wr_np"], inp["w1"], inp["w2"], k=w.k, score=w.score, bias=inp["bias_np"], **sh)
    if w.backward:
        bwd_fn(x, inp["wr_np"], inp["w1"], inp["w2"], fwd, inp["dy_np"][tokens], score=w.score, **sh)
    return time.perf_counter() - t0


def oracle_sample(w, inp, target_s: float, max_experts: int) -> tuple[np.ndarray, float]:
    """The first n tokens, n doubled from 1 while one oracle step stays under
    target_s and the experts the sample reaches stay within max_experts (their
    host copies and quantised weights are prepared untimed).  Returns the
    tokens and the last step's seconds."""
    n = 1
    while True:
        toks = np.arange(n)
        warm_experts(w, inp, sample_experts(w, inp, toks))
        t = oracle_step_timed(w, inp, toks)
        nxt = min(w.T, 2 * n)
        if t >= 0.5 * target_s or n >= w.T or len(sample_experts(w, inp, np.arange(nxt))) > max_experts:
            return toks, t
        n = nxt


def _max_experts(w) -> int:
    # bound the untimed preparation: host copies (and quantised copies) of the experts a sample reaches
    per_expert = 3 * w.F * w.H * 8 * (3 if w.dtype == "mxfp8" else 1)
    return max(w.k, min(w.E, int(24e9 // per_expert)))


def cpu_baseline(w, dinp, target_s: float = 10.0) -> dict:
    """The oracle, as it stands, timed on a bounded sample of the workload's tokens."""
    inp = oracle_inputs(w, dinp)
    toks, _ = oracle_sample(w, inp, target_s, _max_experts(w))
    t = oracle_step_timed(w, inp, toks)
    what = "forward + backward" if w.backward else "forward"
    n = len(toks)
    return {"value": n / t, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"first {n} of {w.T} tokens ({len(sample_experts(w, inp, toks))} experts reached), {what}, "
                      f"fp64 numpy, {t:.2f} s; weights copied to the host and (quantised recipes) quantised "
                      f"before timing"}


# ---------------------------------------------------------------- algorithmic work of each grouped GEMM
GEMM_OPS = ("fc1", "fc2", "fc2_combine", "dgrad_fc2", "dgrad_fc1", "wgrad_fc1", "wgrad_fc2")


def op_work(w, op: str, n_active: int) -> tuple[float, float]:
    """(flops, algorithmic HBM bytes) of one routed grouped-GEMM launch: R = T*k
    rows (padding not counted), n_active experts with rows read their weights
    once, every expert's weight gradient is written (zero where empty)."""
    R, H, F, E = w.T * w.k, w.H, w.F, w.E
    # operand bytes per element: bf16 2; MXFP8 codes + an E8M0 scale per 32; NVFP4 half a byte + an E4M3 per 16
    bw = ba = {"bf16": 2.0, "mxfp8": 1 + 1 / 32, "nvfp4": 0.5 + 1 / 16}[w.dtype]
    z_saved = w.backward
    if op == "fc1":
        if w.dtype == "mxfp8":
            # h' written only as its MXFP8 copies (rows; transposed too when training), as the layer runs it
            return 4.0 * R * H * F, (n_active * 2 * F * H * bw + R * H * ba + R * F * ba * (2 if z_saved else 1)
                                     + (R * 2 * F * 2 if z_saved else 0))
        return 4.0 * R * H * F, n_active * 2 * F * H * bw + R * H * ba + R * F * 2 + (R * 2 * F * 2 if z_saved else 0)
    if op == "fc2":
        return 2.0 * R * H * F, n_active * H * F * bw + R * F * ba + R * H * 2
    if op == "fc2_combine":
        # fc2, then the combine: o's rows read once more, y written (and the shared rows read)
        return 2.0 * R * H * F, (n_active * H * F * bw + R * F * ba + R * H * 2 + R * H * 2 + w.T * H * 2
                                 + (w.T * H * 2 if w.S else 0))
    if op == "dgrad_fc2":
        if w.dtype == "mxfp8" and F % 256 == 0:
            # z read; dz written only as its two MXFP8 copies (rows, and transposed), as the layer runs it
            return 2.0 * R * H * F, n_active * H * F * bw + R * H * ba + R * 2 * F * 2 + 2 * R * 2 * F * ba
        return 2.0 * R * H * F, n_active * H * F * bw + R * H * ba + R * 2 * F * 2 * 2
    if op == "dgrad_fc1":
        return 4.0 * R * H * F, n_active * 2 * F * H * bw + R * 2 * F * ba + R * H * 2
    if op == "wgrad_fc1":
        return 4.0 * R * H * F, E * 2 * F * H * 4 + R * 2 * F * ba + R * H * ba
    if op == "wgrad_fc2":
        return 2.0 * R * H * F, E * H * F * 4 + R * H * ba + R * F * ba
    raise ValueError(op)


def roofline_of(w, op, ms, n_active, peaks, peak_src) -> dict:
    flop, nbytes = op_work(w, op, n_active)
    p_tensor = float(peaks["bf16_tflops"]) * (2.0 if w.dtype == "mxfp8" else 6.0 if w.dtype == "nvfp4" else 1.0)
    bw = float(peaks["hbm_gbs"])
    t_tensor = flop / (p_tensor * 1e12) * 1e3
    t_hbm = nbytes / (bw * 1e9) * 1e3
    tensor = t_tensor >= t_hbm
    tflops = flop / (ms / 1e3) / 1e12
    gbs = nbytes / (ms / 1e3) / 1e9
    note = {"bf16": "bf16_tflops", "mxfp8": "2 x bf16_tflops (fp8:bf16 nominal ratio)",
            "nvfp4": "6 x bf16_tflops (fp4:bf16 nominal ratio on GB300)"}[w.dtype]
    return {"bound": "tensor" if tensor else "hbm",
            "achieved": tflops if tensor else gbs, "peak": p_tensor if tensor else bw,
            "unit": "TFLOP/s" if tensor else "GB/s", "frac": max(t_tensor, t_hbm) / ms,
            "peak_source": (f"{note} of {peak_src} peaks (burst; kernel timed alone)" if tensor
                            else f"hbm_gbs of {peak_src} peaks"),
            "ms_per_launch": ms, "flop_per_launch": flop, "bytes_per_launch": nbytes,
            "tflops": tflops, "gbs": gbs, "t_tensor_ms": t_tensor, "t_hbm_ms": t_hbm,
            "tensor_frac": t_tensor / ms, "hbm_frac": t_hbm / ms,
            "traffic": (TRAFFIC[(w.name, op)][0] * nbytes) if (w.name, op) in TRAFFIC else None,
            "traffic_note": (f"measured DRAM bytes / algorithmic bytes = {TRAFFIC[(w.name, op)][0]:.4f} "
                             f"({TRAFFIC[(w.name, op)][1]}) x this launch's algorithmic bytes"
                             if (w.name, op) in TRAFFIC else None)}


def _timed(fn, n, flush, stream) -> float:
    fn()                                   # one untimed run (a new graph's first replay uploads it)
    s = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    e = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for i in range(n):
        flush.zero_()
        s[i].record(stream)
        fn()
        e[i].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in zip(s, e))


def gemm_op_calls(api, w, layer, dinp, grads, dev) -> dict:
    """One closure per grouped GEMM of the step, on the layer's own saved
    tensors; quantised operands (MXFP8) are made by the library's quantiser
    into buffers owned here."""
    cfg, fl, ws = layer.cfg, layer.fields(), layer.ws
    po, cap, H, F, E = fl["poffsets"], layer.layout.cap, w.H, w.F, w.E
    calls = {}
    if w.dtype == "bf16":
        calls["fc1"] = lambda: api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, fl["x_perm"], dinp["w1"], fl["h"], ws,
                                                    c2=fl["z"] if w.backward else None, row_gate=fl["row_gate"],
                                                    poffsets=po)
        calls["fc2"] = lambda: api.moe_grouped_gemm(cfg, api.GG_FC2, fl["h"], dinp["w2"], fl["o"], ws, poffsets=po)
        if H % 256 == 0:
            y_c = torch.empty((w.T, H), dtype=torch.bfloat16, device=dev)
            sh = layer.view("os", torch.bfloat16, (w.T, H)) if w.S else None
            calls["fc2_combine"] = lambda: api.moe_grouped_gemm(cfg, api.GG_FC2_COMBINE, fl["h"], dinp["w2"], fl["o"],
                                                                ws, c2=y_c, aux=sh, poffsets=po, a_rows=fl["row_src"],
                                                                slot_row=fl["slot_row"])
        if w.backward:
            dpart = layer.view("dgate_part", torch.float32, (cap, F // 128))
            calls["dgrad_fc2"] = lambda: api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC2, fl["dy_perm"], dinp["w2"],
                                                              fl["dz"], ws, aux=fl["z"], row_gate=fl["row_gate"],
                                                              dgate_part=dpart, poffsets=po)
            calls["dgrad_fc1"] = lambda: api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC1, fl["dz"], dinp["w1"],
                                                              fl["dx_perm"], ws, poffsets=po)
            calls["wgrad_fc1"] = lambda: api.moe_grouped_gemm(cfg, api.GG_WGRAD_FC1, fl["dz"], fl["x_perm"],
                                                              grads["dw1"], ws, poffsets=po)
            calls["wgrad_fc2"] = lambda: api.moe_grouped_gemm(cfg, api.GG_WGRAD_FC2, fl["dy_perm"], fl["h"],
                                                              grads["dw2"], ws, poffsets=po)
        return calls
    if w.dtype == "nvfp4":
        # the NVFP4 layer permutes quantised codes and leaves x_perm unwritten:
        # permute x (padding rows zeroed), then quantise it, h and the weights
        # with the library's own quantiser
        api.moe_permute(cfg, dinp["x"], fl["topk_idx"], fl["topk_gate"], fl["counts"], fl["offsets"], po,
                        fl["slot_row"], fl["row_src"], fl["row_gate"], fl["x_perm"], 1, ws)

        def q4(t, batch, rows, cols, mode):
            c = torch.empty(batch * rows * cols // 2, dtype=torch.uint8, device=dev)
            sf = torch.empty(batch * rows * cols // 16, dtype=torch.uint8, device=dev)
            a = torch.empty(1, dtype=torch.float32, device=dev)
            api.moe_quantize_nvfp4(t, batch, rows, cols, mode, c, sf, a)
            return c, sf, a

        (xq, xsf, xa), (w1q, w1sf, w1a) = q4(fl["x_perm"], 1, cap, H, api.MX_ROWS), \
            q4(dinp["w1"], E, 2 * F, H, api.MX_ROWS_GATE_UP)
        calls["fc1"] = lambda: api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, xq, w1q, fl["h"], ws,
                                                    row_gate=fl["row_gate"], poffsets=po, a_scales=xsf,
                                                    b_scales=w1sf, a_amax=xa, b_amax=w1a)
        (hq, hsf, ha), (w2q, w2sf, w2a) = q4(fl["h"], 1, cap, F, api.MX_ROWS), \
            q4(dinp["w2"], 1, E * H, F, api.MX_ROWS)
        calls["fc2"] = lambda: api.moe_grouped_gemm(cfg, api.GG_FC2, hq, w2q, fl["o"], ws, poffsets=po,
                                                    a_scales=hsf, b_scales=w2sf, a_amax=ha, b_amax=w2a)
        return calls
    if w.dtype != "mxfp8":
        return calls

    def q(t, batch, rows, cols, mode):
        c = torch.empty(batch * rows * cols, dtype=torch.uint8, device=dev)
        sf = torch.empty(batch * rows * cols // 28 + 512, dtype=torch.uint8, device=dev)   # room for G224 layouts
        api.moe_quantize_mxfp8(t, batch, rows, cols, mode, c, sf)
        return c, sf

    # the MXFP8 layer keeps x and dy in token order (x_perm, dy_perm unwritten):
    # expert-ordered bf16 copies for the operands here, by the permutation entry point
    perm = lambda src, dst: api.moe_permute(cfg, src, fl["topk_idx"], fl["topk_gate"], fl["counts"], fl["offsets"],
                                            po, fl["slot_row"], fl["row_src"], fl["row_gate"], dst, 1, ws)
    perm(dinp["x"], fl["x_perm"])
    if w.backward:
        perm(dinp["dy"], fl["dy_perm"])

    xq, xsf = q(fl["x_perm"], 1, cap, H, api.MX_ROWS)
    w1q, w1sf = q(dinp["w1"], E, 2 * F, H, api.MX_ROWS_GATE_UP)
    # as the layer runs it: h' only as its MXFP8 copies (the transposed one when training)
    u8 = lambda n: torch.empty(n, dtype=torch.uint8, device=dev)
    hc = dict(q_codes=u8(cap * F), q_scales=u8(cap * F // 32))
    if w.backward:
        hc.update(qt_codes=u8(cap * F), qt_scales=u8(cap * F // 32))
    calls["fc1"] = lambda: api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, xq, w1q, None, ws,
                                                c2=fl["z"] if w.backward else None, row_gate=fl["row_gate"],
                                                poffsets=po, a_scales=xsf, b_scales=w1sf, **hc)
    calls["fc1"]()
    torch.cuda.synchronize()
    hq, hsf = hc["q_codes"], hc["q_scales"]
    w2q, w2sf = q(dinp["w2"], 1, E * H, F, api.MX_ROWS)
    # the layer runs fc2 and the fc1 data gradient on 256 x 224 tiles where H allows (B scales grouped by 224)
    g224 = 224 if H % 224 == 0 else 0
    w2g, w2gsf = q(dinp["w2"], 1, E * H, F, api.MX_ROWS_G224) if g224 else (w2q, w2sf)
    calls["fc2"] = lambda: api.moe_grouped_gemm(cfg, api.GG_FC2, hq, w2g, fl["o"], ws, poffsets=po, a_scales=hsf,
                                                b_scales=w2gsf, b_scale_group=g224)
    if H % 256 == 0:
        y_c = torch.empty((w.T, H), dtype=torch.bfloat16, device=dev)
        sh = layer.view("os", torch.bfloat16, (w.T, H)) if w.S else None
        calls["fc2_combine"] = lambda: api.moe_grouped_gemm(cfg, api.GG_FC2_COMBINE, hq, w2q, fl["o"], ws, c2=y_c,
                                                            aux=sh, poffsets=po, a_scales=hsf, b_scales=w2sf,
                                                            a_rows=fl["row_src"], slot_row=fl["slot_row"])
    if w.backward:
        dpart = layer.view("dgate_part", torch.float32, (cap, F // 128))
        dyq, dysf = q(fl["dy_perm"], 1, cap, H, api.MX_ROWS)
        w2tq, w2tsf = q(dinp["w2"], E, H, F, api.MX_COLS_T)
        # as the layer runs it where F % 256 == 0: dz only as its two MXFP8 copies
        dzc = {}
        if F % 256 == 0:
            u8 = lambda n: torch.empty(n, dtype=torch.uint8, device=dev)
            dzc = dict(q_codes=u8(cap * 2 * F), q_scales=u8(cap * 2 * F // 32), qt_codes=u8(cap * 2 * F),
                       qt_scales=u8(cap * 2 * F // 32))
        calls["dgrad_fc2"] = lambda: api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC2, dyq, w2tq,
                                                          None if dzc else fl["dz"], ws, aux=fl["z"],
                                                          row_gate=fl["row_gate"], dgate_part=dpart, poffsets=po,
                                                          a_scales=dysf, b_scales=w2tsf, **dzc)
        if dzc:                                 # the data gradient's own MXFP8 copies of dz
            calls["dgrad_fc2"]()
            torch.cuda.synchronize()
            dzq, dzsf = dzc["q_codes"], dzc["q_scales"]
        else:
            dzq, dzsf = q(fl["dz"], 1, cap, 2 * F, api.MX_ROWS)
        w1tq, w1tsf = q(dinp["w1"], E, 2 * F, H, api.MX_COLS_T_G224 if g224 else api.MX_COLS_T)
        calls["dgrad_fc1"] = lambda: api.moe_grouped_gemm(cfg, api.GG_DGRAD_FC1, dzq, w1tq, fl["dx_perm"], ws,
                                                          poffsets=po, a_scales=dzsf, b_scales=w1tsf,
                                                          b_scale_group=g224)
        dzt, dztsf = (dzc["qt_codes"], dzc["qt_scales"]) if dzc else q(fl["dz"], 1, cap, 2 * F, api.MX_COLS_T)
        xt, xtsf = q(fl["x_perm"], 1, cap, H, api.MX_COLS_T_G224 if g224 else api.MX_COLS_T)
        calls["wgrad_fc1"] = lambda: api.moe_grouped_gemm(cfg, api.GG_WGRAD_FC1, dzt, xt, grads["dw1"], ws,
                                                          poffsets=po, a_scales=dztsf, b_scales=xtsf,
                                                          b_scale_group=g224)
        ht, htsf = hc["qt_codes"], hc["qt_scales"]
        if g224 and F % 256 == 0:               # dW2^T on 256 x 224 tiles, stored transposed (operands swapped)
            dyt, dytsf = q(fl["dy_perm"], 1, cap, H, api.MX_COLS_T_G224)
            calls["wgrad_fc2"] = lambda: api.moe_grouped_gemm(cfg, api.GG_WGRAD_FC2, ht, dyt, grads["dw2"], ws,
                                                              poffsets=po, a_scales=htsf, b_scales=dytsf,
                                                              b_scale_group=224)
        else:
            dyt, dytsf = q(fl["dy_perm"], 1, cap, H, api.MX_COLS_T)
            calls["wgrad_fc2"] = lambda: api.moe_grouped_gemm(cfg, api.GG_WGRAD_FC2, dyt, ht, grads["dw2"], ws,
                                                              poffsets=po, a_scales=dytsf, b_scales=htsf)
    return calls


def _as_graph(fn, stream, dev):
    """fn's launches captured once into a CUDA graph (as the layer's step runs
    them), returned as its replay: the stage is then timed without the host's
    per-launch overhead between its kernels."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g.replay, g


def stage_breakdown(api, w, layer, dinp, x, y, flush, stream, n, dev=None) -> dict:
    """The HBM-bound steps alone (CUDA events, L2 flushed; each stage replayed
    as a CUDA graph, as in the layer's step), with their algorithmic bytes:
    permute (1+k)*T*H*2, combine (k+1)*T*H*2 (+T*H*2 shared).  A graph of one
    trivial kernel, timed the same way, gives the fixed cost of a graph launch
    between two events (`graph_launch`, about 7 us), which the layer's step
    pays once, not per stage; the `*_gbs` rates are taken over each stage's
    time less that cost, the `*_gbs_raw` ones over the whole time."""
    cfg, fl = layer.cfg, layer.fields()
    T, H, k = w.T, w.H, w.k
    dev = x.device if dev is None else dev
    shared = layer.view("os", torch.bfloat16, (T, H)) if w.S > 0 else None
    graphs = []

    def timed(fn):
        run, g = _as_graph(fn, stream, dev)
        graphs.append(g)
        return _timed(run, n, flush, stream)

    out = {}
    out["router_topk"] = timed(lambda: api.moe_router_topk(cfg, x, dinp["w_router"], dinp["bias"], fl["logits"],
                                                            fl["topk_idx"], fl["topk_gate"], layer.ws))
    out["permute"] = timed(lambda: api.moe_permute(cfg, x, fl["topk_idx"], fl["topk_gate"], fl["counts"],
                                                   fl["offsets"], fl["poffsets"], fl["slot_row"], fl["row_src"],
                                                   fl["row_gate"], fl["x_perm"], int(w.backward), layer.ws))
    out["combine"] = timed(lambda: api.moe_unpermute(cfg, fl["o"], fl["slot_row"], shared, y))
    pbytes = (1 + k) * T * H * 2
    cbytes = (k + 1) * T * H * 2 + (T * H * 2 if w.S > 0 else 0)
    tiny = torch.zeros(16, device=dev)
    out["graph_launch"] = timed(lambda: tiny.add_(1.0))
    net = lambda ms: max(ms - out["graph_launch"], 1e-6)
    out["permute_gbs"] = pbytes / (net(out["permute"]) / 1e3) / 1e9
    out["combine_gbs"] = cbytes / (net(out["combine"]) / 1e3) / 1e9
    out["permute_gbs_raw"] = pbytes / (out["permute"] / 1e3) / 1e9
    out["combine_gbs_raw"] = cbytes / (out["combine"] / 1e3) / 1e9
    return out


def e2e_pipelined(api, w, layer, x, y, dy, grads, stream, K, no_graph, dev):
    """K steps through the public API with host buffers: returns (ms for all K
    steps, host->device bytes per step, device->host bytes per step)."""
    xs = [x, torch.empty_like(x)]
    ys = [y, torch.empty_like(y)]
    dys = [dy, torch.empty_like(dy)] if w.backward else [None, None]
    x_h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    x_h.copy_(x)
    dy_h = None
    if w.backward:
        dy_h = torch.empty(dy.shape, dtype=dy.dtype, pin_memory=True)
        dy_h.copy_(dy)
    y_h = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for _ in range(2)]

    def step_on(b):
        layer.forward(xs[b], ys[b])
        if w.backward:
            layer.backward(xs[b], dys[b], grads)

    runs = [lambda b=b: step_on(b) for b in range(2)]
    if not no_graph:
        runs = []
        for b in range(2):
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                step_on(b)
            stream.wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step_on(b)
            runs.append(g.replay)
    for b in range(2):
        runs[b]()
    torch.cuda.synchronize()

    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    comp_done = [ev() for _ in range(K)]
    out_done = [ev() for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(cin)
    for i in range(K):
        b = i % 2
        with torch.cuda.stream(cin):
            if i >= 2:
                cin.wait_event(comp_done[i - 2])        # inputs of buffer b no longer read
            xs[b].copy_(x_h, non_blocking=True)
            if w.backward:
                dys[b].copy_(dy_h, non_blocking=True)
        in_ready = ev()
        in_ready.record(cin)
        stream.wait_event(in_ready)
        if i >= 2:
            stream.wait_event(out_done[i - 2])          # output of buffer b read back
        with torch.cuda.stream(stream):
            runs[b]()
        comp_done[i].record(stream)
        cout.wait_event(comp_done[i])
        with torch.cuda.stream(cout):
            y_h[b].copy_(ys[b], non_blocking=True)
        out_done[i].record(cout)
    for i in range(max(0, K - 2), K):
        cout.wait_event(out_done[i])
    end.record(cout)
    torch.cuda.synchronize()
    h2d = x.numel() * x.element_size() + (dy.numel() * dy.element_size() if w.backward else 0)
    return start.elapsed_time(end), h2d, y.numel() * y.element_size()


# ---------------------------------------------------------------- our arm
def bench_workload(args, w, world, rank, local, dev, cpu_target_s: float | None) -> dict | None:
    from moe_expert_layer_05_gb300 import api

    dinp = make_inputs_on_device(w, dev, seed=rank)
    cfg = api.config_of(w)
    layer = api.MoELayer(cfg, dinp, with_backward=w.backward, device=dev)
    x = dinp["x"]
    y = torch.empty_like(x)
    dy = dinp["dy"]
    grads = None
    clocks = ClockSampler(local)
    clocks.start()
    if w.backward:
        layer.forward(x, y)
        _, _, grads = layer.backward(x, dy)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        layer.forward(x, y)
        if w.backward:
            layer.backward(x, dy, grads)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # One step as a CUDA graph (the layer issues a fixed launch sequence and no
    # host sync, so it captures whole); --no-graph launches it eagerly.
    run = step
    launches_per_step = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()                      # warm the capture stream's first use
        stream.wait_stream(side)
        torch.cuda.synchronize()
        l0 = api.moe_kernel_launches()
        with torch.cuda.graph(graph):
            step()
        launches_per_step = api.moe_kernel_launches() - l0
        run = graph.replay
        for _ in range(args.warmup):
            run()
        torch.cuda.synchronize()

    # ---- timed region
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    l0 = api.moe_kernel_launches()
    for i in range(K):
        flush.zero_()
        starts[i].record(stream)
        run()
        ends[i].record(stream)
    torch.cuda.synchronize()
    launches = api.moe_kernel_launches() - l0
    if launches_per_step is not None:
        launches = launches_per_step * K      # graph replays: the library's kernels, counted at capture
    barrier(world)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = aggregate(w.T, K, world, total_ms)
    assert api.moe_read_device_status(layer.ws) == 0, "device status not ok"

    # ---- each grouped GEMM alone, same inputs, same stream
    Kk = max(10, min(K, 200))
    n_active = int((layer.fields()["counts"] > 0).sum())
    calls = gemm_op_calls(api, w, layer, dinp, grads, dev)
    op_ms = {op: _timed(fn, Kk, flush, stream) for op, fn in calls.items()}
    del calls
    stages = stage_breakdown(api, w, layer, dinp, x, y, flush, stream, Kk) if w.dtype != "nvfp4" else {}
    assert api.moe_read_device_status(layer.ws) == 0, "device status not ok"

    # ---- end to end through the public API, host buffers, copies inside the timed region
    e2e_total, e2e_in, e2e_out = e2e_pipelined(api, w, layer, x, y, dy, grads, stream, K, args.no_graph, dev)
    barrier(world)
    e2e_total = max_over_ranks(e2e_total, world, dev)
    clk = clocks.stop()

    if rank != 0:
        return None
    peaks, peak_src = read_peaks()
    R = w.T * w.k
    fwd_flop = 6.0 * R * w.H * w.F + 6.0 * w.T * w.H * w.S
    step_flop = fwd_flop * (3 if w.backward else 1)
    ops = {op: roofline_of(w, op, ms, n_active, peaks, peak_src) for op, ms in op_ms.items()}
    for r in ops.values():
        if clk.get("sm_mhz"):
            r["ms_x_sm_mhz"] = r["ms_per_launch"] * clk["sm_mhz"]
    # the layer runs the plain fc2 and the combine kernel; the fused fc2 + combine
    # is an op of its own, timed beside it but not launched by the step
    step_ops = [o for o in ops if o != "fc2_combine"]
    dominant = max(step_ops, key=lambda o: ops[o]["ms_per_launch"])
    roof = dict(ops[dominant])
    roof["kernel"] = f"{dominant} grouped GEMM (tcgen05" + \
        (", mxf8f6f4 block-scaled" if w.dtype == "mxfp8" else "") + ")"
    roof["why_this_kernel"] = "the longest grouped GEMM of the step, timed alone"
    out = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": total_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "F": w.F, "S": w.S,
                   "score": w.score, "pass": "fwd+bwd" if w.backward else "fwd",
                   "l2": "flushed (512 MB write) before every timed step, outside the events",
                   "parallelism": f"replicas x{world}",
                   "cuda_graph": not args.no_graph},
        "expert_gemm_tflops_per_gpu": step_flop / (total_ms / K / 1e3) / 1e12,
        "expert_gemm_frac_of_bf16_peak": step_flop / (total_ms / K / 1e3) / 1e12 / float(peaks["bf16_tflops"]),
        "roofline": roof,
        "gemm_ops": ops,
        "experts_with_rows": n_active,
        "stages_ms": stages,
        "e2e": {"value": aggregate(w.T, K, world, e2e_total), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e_in, "d2h_bytes_per_step": e2e_out,
                "how": "pinned host x (and dy) -> device and y -> pinned host every step on two copy "
                       "streams, double-buffered so copies overlap the neighbouring steps' compute; "
                       "no L2 flush (the expert weights exceed L2); first copy to last read back"},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if cpu_target_s is not None and world == 1:
        out["cpu_baseline"] = cpu_baseline(w, dinp, cpu_target_s)
    del layer, grads, dinp, flush
    gc.collect()
    torch.cuda.empty_cache()
    return out


def run_ours(args) -> dict | None:
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (GB300); there is no CPU path")
    torch.cuda.set_device(local)
    dist_init(world, True)
    dev = torch.device("cuda", local)
    cpu = None if args.no_cpu_baseline else 10.0
    if args.workload is not None:
        w = WORKLOADS[args.workload]
        if args.tokens is not None:
            w = dataclasses.replace(w, T=args.tokens, name=f"{w.name}_T{args.tokens}")
        if args.experts is not None:
            w = dataclasses.replace(w, E=args.experts, name=f"{w.name}_E{args.experts}")
        return bench_workload(args, w, world, rank, local, dev, cpu)
    if world > 1:
        return bench_workload(args, WORKLOADS[HEADLINE], world, rank, local, dev, cpu)
    sub = {}
    for name in SUITE[:-1]:
        sub[name] = bench_workload(args, WORKLOADS[name], world, rank, local, dev, None if cpu is None else 5.0)
    out = bench_workload(args, WORKLOADS[HEADLINE], world, rank, local, dev, cpu)
    out["configs"] = sub
    out["headline"] = ("the largest configuration: DeepSeek-V3-like layer, fwd+bwd, MXFP8 expert GEMMs, "
                       "T=16384; the other four configurations are under 'configs'")
    return out


# ---------------------------------------------------------------- profiler captures
PROFILE_OPS = GEMM_OPS + ("router", "permute", "combine", "step")


def profile_op(args) -> dict:
    """For `ncu --profile-from-start off` captures: set up once, then exactly one
    launch of the chosen op between cudaProfilerStart and cudaProfilerStop.
    permute / combine allocate only x, the routing and the expert-ordered rows
    (and y); the grouped GEMMs run one untimed layer step first."""
    from moe_expert_layer_05_gb300 import api
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload or HEADLINE]
    if args.tokens is not None:
        w = dataclasses.replace(w, T=args.tokens)
    if args.experts is not None:
        w = dataclasses.replace(w, E=args.experts)
    cfg = api.config_of(w)
    if args.profile_op == "step":
        # one whole step of the layer (forward, and backward where the workload
        # trains) after three warm-up steps, launched eagerly
        d = make_inputs_on_device(w, dev, seed=0, with_dy=w.backward)
        layer = api.MoELayer(api.config_of(w), d, with_backward=w.backward, device=dev)
        x, dy = d["x"], d["dy"]
        y = torch.empty_like(x)
        layer.forward(x, y)
        grads = layer.backward(x, dy)[2] if w.backward else None

        def one():
            layer.forward(x, y)
            if w.backward:
                layer.backward(x, dy, grads)

        for _ in range(3):
            one()
        torch.cuda.synchronize()
        l0 = api.moe_kernel_launches()
        torch.cuda.profiler.start()
        one()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        return {"profile_op": "step", "workload": w.name, "T": w.T, "E": w.E,
                "launches": api.moe_kernel_launches() - l0, "status": api.moe_read_device_status(layer.ws)}
    if args.profile_op in ("router", "permute", "combine"):
        cfg = api.make_config(w.T, w.H, w.E, w.k, w.F, 0, w.score, "bf16")   # the routing and row copies only
        d = make_router_inputs_on_device(w, dev, seed=0)
        T, E, k, H = w.T, w.E, w.k, w.H
        cap = api.moe_capacity_rows(cfg)
        ws = torch.zeros(max(api.moe_workspace_bytes(cfg), 256), dtype=torch.uint8, device=dev)
        api.moe_workspace_init(ws)
        i32 = lambda *s: torch.empty(s, dtype=torch.int32, device=dev)
        logits = torch.empty((T, E), dtype=torch.float32, device=dev)
        idx, gate = i32(T, k), torch.empty((T, k), dtype=torch.float32, device=dev)
        counts, offs, poffs, slot_row, row_src = i32(E), i32(E + 1), i32(E + 1), i32(T, k), i32(cap)
        row_gate = torch.empty(cap, dtype=torch.float32, device=dev)
        rows = torch.empty((cap, H), dtype=torch.bfloat16, device=dev)
        bias = d["bias"] if w.score == "sigmoid" else None
        api.moe_router_topk(cfg, d["x"], d["w_router"], bias, logits, idx, gate, ws)
        perm = lambda: api.moe_permute(cfg, d["x"], idx, gate, counts, offs, poffs, slot_row, row_src, row_gate, rows,
                                       0, ws)
        perm()
        y = torch.empty_like(d["x"])
        call = {"permute": perm,
                "combine": lambda: api.moe_unpermute(cfg, rows, slot_row, None, y),
                "router": lambda: api.moe_router_topk(cfg, d["x"], d["w_router"], bias, logits, idx, gate, ws),
                }[args.profile_op]
        call()
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        call()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        return {"profile_op": args.profile_op, "workload": w.name, "T": T, "E": E,
                "algorithmic_bytes": (1 + k) * T * H * 2 if args.profile_op != "router" else None, "status": api.moe_read_device_status(ws),
                "max_memory_gb": torch.cuda.max_memory_allocated(dev) / 1e9}
    if w.dtype == "nvfp4":
        return profile_op_nvfp4(args, w, dev)
    bwd = args.profile_op not in ("fc1", "fc2") or w.backward
    w = dataclasses.replace(w, backward=bwd)
    d = make_inputs_on_device(w, dev, seed=0, with_dy=bwd)
    layer = api.MoELayer(api.config_of(w), d, with_backward=bwd)
    layer.forward(d["x"])
    grads = layer.backward(d["x"], d["dy"])[2] if bwd else None
    torch.cuda.synchronize()
    call = gemm_op_calls(api, w, layer, d, grads, dev)[args.profile_op]
    n_active = int((layer.fields()["counts"] > 0).sum())
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    call()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    flop, nbytes = op_work(w, args.profile_op, n_active)
    return {"profile_op": args.profile_op, "workload": w.name, "T": w.T, "E": w.E, "experts_with_rows": n_active,
            "flop": flop, "algorithmic_bytes": nbytes, "status": api.moe_read_device_status(layer.ws),
            "max_memory_gb": torch.cuda.max_memory_allocated(dev) / 1e9}


def profile_op_nvfp4(args, w, dev) -> dict:
    """--profile-op for an NVFP4 workload: the NVFP4 forward once, then x_perm
    (permuted, padding zeroed), h and the weights quantised by the library into
    bench-owned buffers, and the chosen NVFP4 GEMM once inside the profiler range."""
    from moe_expert_layer_05_gb300 import api
    if args.profile_op not in ("fc1", "fc2"):
        raise SystemExit("--profile-op: NVFP4 workloads have fc1 and fc2 only")
    d = make_inputs_on_device(w, dev, seed=0, with_dy=False)
    cfg = api.config_of(w)
    layer = api.MoELayer(cfg, d, with_backward=False)
    x = d["x"]
    layer.forward(x)
    fl, ws, cap = layer.fields(), layer.ws, layer.layout.cap
    api.moe_permute(cfg, x, fl["topk_idx"], fl["topk_gate"], fl["counts"], fl["offsets"], fl["poffsets"],
                    fl["slot_row"], fl["row_src"], fl["row_gate"], fl["x_perm"], 1, ws)

    def q(t, batch, rows, cols, mode):
        c = torch.empty(t.numel() // 2, dtype=torch.uint8, device=dev)
        sf = torch.empty(t.numel() // 16, dtype=torch.uint8, device=dev)
        a = torch.empty(1, dtype=torch.float32, device=dev)
        api.moe_quantize_nvfp4(t, batch, rows, cols, mode, c, sf, a)
        return c, sf, a

    po = fl["poffsets"]
    if args.profile_op == "fc1":
        (aq, asf, aa), (bq, bsf, ba) = q(fl["x_perm"], 1, cap, w.H, api.MX_ROWS), \
            q(d["w1"], w.E, 2 * w.F, w.H, api.MX_ROWS_GATE_UP)
        call = lambda: api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, aq, bq, fl["h"], ws, row_gate=fl["row_gate"],
                                            poffsets=po, a_scales=asf, b_scales=bsf, a_amax=aa, b_amax=ba)
    else:
        (aq, asf, aa), (bq, bsf, ba) = q(fl["h"], 1, cap, w.F, api.MX_ROWS), q(d["w2"], 1, w.E * w.H, w.F, api.MX_ROWS)
        call = lambda: api.moe_grouped_gemm(cfg, api.GG_FC2, aq, bq, fl["o"], ws, poffsets=po, a_scales=asf,
                                            b_scales=bsf, a_amax=aa, b_amax=ba)
    call()
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    call()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    return {"profile_op": args.profile_op, "workload": args.workload, "T": w.T, "E": w.E,
            "status": api.moe_read_device_status(ws),
            "max_memory_gb": torch.cuda.max_memory_allocated(dev) / 1e9}


# ---------------------------------------------------------------- reference arm
def run_reference(args) -> dict | None:
    """The fp64 oracle on the host cores, on our arm's workload, metric and
    unit: every step runs the same bounded sample of the workload's tokens,
    with the weights it reads copied (and, for the quantised recipes,
    quantised) once before the first step."""
    world, rank, local = dist_env()
    if rank != 0:
        return None
    w = WORKLOADS[args.workload or HEADLINE]
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
        dinp = make_inputs_on_device(w, torch.device("cuda", local), seed=0)
    else:
        dinp = make_inputs(w, seed=0)
    inp = oracle_inputs(w, dinp)
    per_step = min(10.0, 100.0 / max(1, args.steps + args.warmup))
    toks, _ = oracle_sample(w, inp, per_step, _max_experts(w))
    for _ in range(args.warmup):
        oracle_step_timed(w, inp, toks)
    total = 0.0
    for _ in range(args.steps):
        total += oracle_step_timed(w, inp, toks)
    n = len(toks)
    value = n * args.steps / total
    sample = (f"first {n} of {w.T} tokens every step ({len(sample_experts(w, inp, toks))} experts reached), "
              f"{'forward + backward' if w.backward else 'forward'}, fp64 numpy; weights copied to the host and "
              f"(quantised recipes) quantised before the first step")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "F": w.F, "S": w.S,
                   "score": w.score, "pass": "fwd+bwd" if w.backward else "fwd",
                   "l2": "flushed (512 MB write) before every timed step, outside the events",
                   "parallelism": f"replicas x{world}", "cuda_graph": True},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=None,
                    help="one workload only (default: all five configurations, headline the largest)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch each timed step eagerly, not as a CUDA graph")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (smaller cases for profiler captures; not a bench line)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (smaller cases for profiler captures; not a bench line)")
    ap.add_argument("--profile-op", choices=sorted(PROFILE_OPS), default=None,
                    help="for profiler captures: set up, then this op once inside cudaProfilerStart/Stop "
                         "(ncu --profile-from-start off); prints one JSON line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile_op is not None:
        out = profile_op(args)
    else:
        out = run_reference(args) if args.impl == "reference" else run_ours(args)
    if out is not None:
        print(json.dumps(out), flush=True)
    world, _, _ = dist_env()
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
