#!/usr/bin/env python3
"""Throughput of the MoE expert layer on GB300 (one JSON line on rank 0).

A step is one pass of the layer over one batch: router GEMM, top-k gating,
sync-free permutation, grouped-GEMM SwiGLU experts with the gate applied at the
activation, combine (plus dgrad + wgrad for workloads that train).  The default
workload is the Mixtral-like forward layer (T=4096, H=4096, E=8, k=2,
F=14336, bf16), seeded synthetic inputs.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events on
the launching stream, with L2 flushed (a 512 MB write) before every step outside
the events; barrier + synchronize on both sides; the max over ranks.  With
--gpus N under torchrun every rank runs its own tokens through replicated
experts (no data-path collective): weak scaling.  The end-to-end figure (e2e)
streams K batches from pinned host memory and reads every result back, on two
copy streams with double-buffered device inputs, so the copies of one step
overlap the compute of its neighbours.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores
"""
from __future__ import annotations

import argparse
import dataclasses
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

from moe_expert_layer_05_gb300.inputs import WORKLOADS, make_inputs, make_inputs_on_device  # noqa: E402

METRIC = "MoE layer tokens/s on 1 GB300; grouped-GEMM TFLOPS as % of tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 512 << 20
# dram__bytes_read.sum + dram__bytes_write.sum of one fc1 launch, from the ncu
# capture summarised in profiles/ (None until captured for the current kernel).
FC1_TRAFFIC_BYTES = 2.295e9   # profiles/fc1_grouped_gemm_mixtral_full.md (bf16 Mixtral-like fc1, DRAM read + write)
# NVFP4 Mixtral-like fc1: captured at T=2048, E=4 (the same 1024 rows per
# expert), 374.1 MB; the traffic grows with the experts, so x2 for E=8
# (profiles/fc1_grouped_gemm_mixtral_nvfp4.md)
FC1_NV4_TRAFFIC_BYTES = 2 * 374.1e6


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
    """nvidia-smi sampled every 100 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

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
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.01)
        self.lines.clear()

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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def read_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- oracle timing (CPU)
class _F32Experts:
    """Expert weights as fp32 numpy (exact bf16 values), per expert on demand."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.shape = tuple(t.shape)
        self.c = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.c:
            self.c[e] = self.t[e].to("cpu", torch.float32).numpy()
        return self.c[e]

    def warm(self):
        for e in range(self.shape[0]):
            self[e]
        return self


def _oracle_fns(w):
    from oracle import moe_oracle as O
    if w.dtype == "mxfp8":
        return O.moe_forward_mx, O.moe_backward_mx
    if w.dtype == "nvfp4":
        return O.moe_forward_nvfp4, None         # forward-only workloads
    return O.moe_forward, O.moe_backward


def oracle_step_timed(w, inp_cpu, tokens: np.ndarray) -> float:
    """One step of the oracle (forward, plus backward for training workloads)
    on the given tokens; returns seconds."""
    fwd_fn, bwd_fn = _oracle_fns(w)
    x = inp_cpu["x_np"][tokens]
    sh = dict(w1_shared=inp_cpu["w1s_np"], w2_shared=inp_cpu["w2s_np"])
    if w.dtype != "bf16":
        sh["weight_cache"] = inp_cpu["wcache"]      # weights quantised once, as the recipe does
    t0 = time.perf_counter()
    fwd = fwd_fn(x, inp_cpu["wr_np"], inp_cpu["w1"], inp_cpu["w2"], k=w.k, score=w.score, bias=inp_cpu["bias_np"],
                 **sh)
    if w.backward:
        bwd_fn(x, inp_cpu["wr_np"], inp_cpu["w1"], inp_cpu["w2"], fwd, inp_cpu["dy_np"][tokens], score=w.score, **sh)
    return time.perf_counter() - t0


def oracle_inputs(w, dinp) -> dict:
    def npf(t):
        return None if t is None else t.to("cpu", torch.float32).numpy().astype(np.float64)
    return {"x_np": npf(dinp["x"]), "wr_np": npf(dinp["w_router"]), "bias_np": npf(dinp["bias"]),
            "w1s_np": npf(dinp["w1_shared"]), "w2s_np": npf(dinp["w2_shared"]), "dy_np": npf(dinp["dy"]),
            "w1": _F32Experts(dinp["w1"]), "w2": _F32Experts(dinp["w2"]), "wcache": {}}


def warm_experts(w, inp, tokens):
    """Copy to host (untimed) the experts the given tokens route to."""
    from oracle import moe_oracle as O
    logits = O.router_logits(inp["x_np"][tokens], inp["wr_np"])
    idx, _ = O.route(logits, w.k, w.score, inp["bias_np"])
    quantised = w.dtype == "mxfp8"
    for e in np.unique(idx):
        inp["w1"][e]
        inp["w2"][e]
        if w.dtype == "nvfp4":
            O.nvfp4_weight(inp["wcache"], "w1", inp["w1"], int(e))
            O.nvfp4_weight(inp["wcache"], "w2", inp["w2"], int(e))
        if quantised:
            # the recipe quantises weights once; do it here, outside the timed oracle call
            for name, W in (("w1", inp["w1"][e]), ("w2", inp["w2"][e])):
                for axis in (-1, 0):
                    key = (name, int(e), axis)
                    if key not in inp["wcache"]:
                        inp["wcache"][key] = O.mxfp8_roundtrip(W, axis)
    if quantised and inp["w1s_np"] is not None:
        for name, W in (("w1s", inp["w1s_np"]), ("w2s", inp["w2s_np"])):
            for axis in (-1, 0):
                inp["wcache"].setdefault((name, 0, axis), O.mxfp8_roundtrip(W, axis))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, dinp, target_s: float = 10.0) -> dict:
    """The oracle, as it stands, on the first n tokens; n grows until one run
    takes about target_s seconds (or covers all tokens)."""
    inp = oracle_inputs(w, dinp)
    n = 8
    while True:
        warm_experts(w, inp, np.arange(n))
        t = oracle_step_timed(w, inp, np.arange(n))
        if t >= 0.7 * target_s or n >= w.T:
            break
        n = min(w.T, max(n * 2, int(n * target_s / max(t, 1e-3))))
    what = "forward + backward" if w.backward else "forward"
    return {"value": n / t, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"first {n} of {w.T} tokens, {what} (fp64 numpy), {t:.1f} s"}


# ---------------------------------------------------------------- our arm
def run_ours(args) -> dict | None:
    from moe_expert_layer_05_gb300 import api

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (GB300); there is no CPU path")
    torch.cuda.set_device(local)
    dist_init(world, True)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    if args.tokens is not None:
        w = dataclasses.replace(w, T=args.tokens, name=f"{w.name}_T{args.tokens}")
    if args.experts is not None:
        w = dataclasses.replace(w, E=args.experts, name=f"{w.name}_E{args.experts}")
    dinp = make_inputs_on_device(w, dev, seed=rank)
    cfg = api.config_of(w)
    layer = api.MoELayer(cfg, dinp, with_backward=w.backward, device=dev)
    x = dinp["x"]
    y = torch.empty_like(x)
    dy = dinp["dy"]
    grads = None
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
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
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
    clk = clocks.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = aggregate(w.T, K, world, total_ms)
    assert api.moe_read_device_status(layer.ws) == 0, "device status not ok"

    # ---- the dominant kernel (fc1 grouped GEMM) alone, same inputs, same stream
    fl = layer.fields()
    Kk = max(10, min(K, 200))
    s_ev = [torch.cuda.Event(enable_timing=True) for _ in range(Kk)]
    e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(Kk)]
    z = fl["z"] if w.backward else None
    mx = w.dtype == "mxfp8"
    nv = w.dtype == "nvfp4"
    if nv:
        # the NVFP4 layer permutes quantised codes and leaves x_perm unwritten:
        # permute x (padding rows zeroed), then quantise it and W1 with the
        # library's own quantiser into bench-owned buffers
        cap = layer.layout.cap
        api.moe_permute(cfg, x, fl["topk_idx"], fl["topk_gate"], fl["counts"], fl["offsets"], fl["poffsets"],
                        fl["slot_row"], fl["row_src"], fl["row_gate"], fl["x_perm"], 1, layer.ws)
        xq = torch.empty(cap * w.H // 2, dtype=torch.uint8, device=dev)
        xsf = torch.empty(cap * w.H // 16, dtype=torch.uint8, device=dev)
        w1q = torch.empty(dinp["w1"].numel() // 2, dtype=torch.uint8, device=dev)
        w1sf = torch.empty(dinp["w1"].numel() // 16, dtype=torch.uint8, device=dev)
        amax = torch.empty(2, dtype=torch.float32, device=dev)
        api.moe_quantize_nvfp4(fl["x_perm"], 1, cap, w.H, api.MX_ROWS, xq, xsf, amax[0:1])
        api.moe_quantize_nvfp4(dinp["w1"], w.E, 2 * w.F, w.H, api.MX_ROWS_GATE_UP, w1q, w1sf, amax[1:2])
        fc1_args = (xq, w1q, fl["h"], layer.ws)
        fc1_kw = dict(c2=None, row_gate=fl["row_gate"], poffsets=fl["poffsets"], a_scales=xsf, b_scales=w1sf,
                      a_amax=amax[0:1], b_amax=amax[1:2])
    elif mx:
        # operands quantised by the library's own quantiser into bench-owned buffers
        cap = layer.layout.cap
        xq = torch.empty(cap * w.H, dtype=torch.uint8, device=dev)
        xsf = torch.empty(cap * w.H // 32, dtype=torch.uint8, device=dev)
        w1q = torch.empty(dinp["w1"].numel(), dtype=torch.uint8, device=dev)
        w1sf = torch.empty(dinp["w1"].numel() // 32, dtype=torch.uint8, device=dev)
        api.moe_quantize_mxfp8(fl["x_perm"], 1, cap, w.H, api.MX_ROWS, xq, xsf)
        api.moe_quantize_mxfp8(dinp["w1"], w.E, 2 * w.F, w.H, api.MX_ROWS_GATE_UP, w1q, w1sf)
        fc1_args = (xq, w1q, fl["h"], layer.ws)
        fc1_kw = dict(c2=z, row_gate=fl["row_gate"], poffsets=fl["poffsets"], a_scales=xsf, b_scales=w1sf)
    else:
        fc1_args = (fl["x_perm"], dinp["w1"], fl["h"], layer.ws)
        fc1_kw = dict(c2=z, row_gate=fl["row_gate"], poffsets=fl["poffsets"])
    for i in range(Kk):
        flush.zero_()
        s_ev[i].record(stream)
        api.moe_grouped_gemm(cfg, api.GG_FC1_SWIGLU, *fc1_args, **fc1_kw)
        e_ev[i].record(stream)
    torch.cuda.synchronize()
    fc1_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(s_ev, e_ev))
    # the rest of the forward chain, one stage at a time (context for the line)
    stages = {} if (mx or nv) else stage_breakdown(api, cfg, layer, dinp, x, y, flush, stream, Kk)
    stages["fc1_grouped_gemm"] = fc1_ms

    # ---- end to end: host buffers, copies inside the timed region.  Two sets
    # of device inputs/outputs: step i's host->device copy (copy stream) and
    # step i-1's device->host read (a second copy stream) overlap step i-1's /
    # step i's compute, the way a user streams batches through the layer.
    e2e_total, e2e_in, e2e_out = e2e_pipelined(api, w, layer, x, y, dy, grads, stream, K, args.no_graph, dev)
    barrier(world)
    e2e_total = max_over_ranks(e2e_total, world, dev)

    if rank != 0:
        return None
    peaks, peak_src = read_peaks()
    R = w.T * w.k
    fc1_flop = 4.0 * R * w.H * w.F
    achieved = fc1_flop / (fc1_ms / 1e3) / 1e12
    peak = float(peaks["bf16_tflops"])
    peak_note = f"bf16_tflops of {peak_src} peaks (burst; kernel timed alone)"
    if mx:
        peak *= 2.0   # dense fp8 / bf16 nominal ratio (4.5 / 2.25 PFLOP/s)
        peak_note = f"2 x bf16_tflops of {peak_src} peaks (fp8:bf16 nominal ratio; burst)"
    if nv:
        peak *= 6.0   # dense fp4 / bf16 nominal ratio on GB300 (13.5 / 2.25 PFLOP/s)
        peak_note = f"6 x bf16_tflops of {peak_src} peaks (fp4:bf16 nominal ratio on GB300; burst)"
    fwd_flop = 6.0 * R * w.H * w.F + 6.0 * w.T * w.H * w.S
    step_flop = fwd_flop * (3 if w.backward else 1)
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
        "roofline": {"bound": "tensor",
                     "kernel": "fc1 grouped GEMM (tcgen05" + (" mxf8f6f4 block-scaled" if mx else "") +
                               (" mxf4nvf4 block-scaled" if nv else "") +
                               ", fused gated SwiGLU)",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": peak_note,
                     "traffic": (FC1_TRAFFIC_BYTES if w.name == "mixtral" else
                                 FC1_NV4_TRAFFIC_BYTES if w.name == "mixtral_nvfp4" else None),
                     "flop_per_launch": fc1_flop, "ms_per_launch": fc1_ms},
        "stages_ms": stages,
        "e2e": {"value": aggregate(w.T, K, world, e2e_total), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e_in, "d2h_bytes_per_step": e2e_out,
                "how": "pinned host x (and dy) -> device and y -> pinned host every step on two copy "
                       "streams, double-buffered so copies overlap the neighbouring steps' compute; "
                       "no L2 flush (the expert weights exceed L2); first copy to last read back"},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(w, dinp)
    return out


PROFILE_OPS = ("fc1", "fc2", "dgrad_fc2", "dgrad_fc1", "wgrad_fc1", "wgrad_fc2")


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


def profile_op(args) -> dict:
    """One untimed step of the workload, then one grouped GEMM of it between
    cudaProfilerStart and cudaProfilerStop, for `ncu --profile-from-start off`
    captures.  bf16 workloads (every op) and NVFP4 workloads (fc1, fc2)."""
    from moe_expert_layer_05_gb300 import api
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    if args.tokens is not None:
        w = dataclasses.replace(w, T=args.tokens)
    if args.experts is not None:
        w = dataclasses.replace(w, E=args.experts)
    if w.dtype == "nvfp4":
        return profile_op_nvfp4(args, w, dev)
    if w.dtype != "bf16":
        raise SystemExit("--profile-op: bf16 and NVFP4 workloads only")
    bwd = args.profile_op not in ("fc1", "fc2")
    d = make_inputs_on_device(w, dev, seed=0, with_dy=bwd)
    layer = api.MoELayer(api.config_of(w), d, with_backward=True)
    layer.forward(d["x"])
    grads = layer.backward(d["x"], d["dy"])[2] if bwd else None
    torch.cuda.synchronize()
    fl, c, ws = layer.fields(), layer.cfg, layer.ws
    po = fl["poffsets"]
    calls = {
        "fc1": lambda: api.moe_grouped_gemm(c, api.GG_FC1_SWIGLU, fl["x_perm"], d["w1"], fl["h"], ws, c2=fl["z"],
                                            row_gate=fl["row_gate"], poffsets=po),
        "fc2": lambda: api.moe_grouped_gemm(c, api.GG_FC2, fl["h"], d["w2"], fl["o"], ws, poffsets=po),
        "dgrad_fc2": lambda: api.moe_grouped_gemm(c, api.GG_DGRAD_FC2, fl["dy_perm"], d["w2"], fl["dz"], ws,
                                                  aux=fl["z"], row_gate=fl["row_gate"], poffsets=po),
        "dgrad_fc1": lambda: api.moe_grouped_gemm(c, api.GG_DGRAD_FC1, fl["dz"], d["w1"], fl["dx_perm"], ws,
                                                  poffsets=po),
        "wgrad_fc1": lambda: api.moe_grouped_gemm(c, api.GG_WGRAD_FC1, fl["dz"], fl["x_perm"], grads["dw1"], ws,
                                                  poffsets=po),
        "wgrad_fc2": lambda: api.moe_grouped_gemm(c, api.GG_WGRAD_FC2, fl["dy_perm"], fl["h"], grads["dw2"], ws,
                                                  poffsets=po),
    }
    torch.cuda.profiler.start()
    calls[args.profile_op]()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    return {"profile_op": args.profile_op, "workload": args.workload, "T": w.T, "E": w.E,
            "status": api.moe_read_device_status(ws),
            "max_memory_gb": torch.cuda.max_memory_allocated(dev) / 1e9}


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


def stage_breakdown(api, cfg, layer, dinp, x, y, flush, stream, n) -> dict:
    fl = layer.fields()
    lay = layer.layout
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k

    def timed(fn):
        s = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        e = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            flush.zero_()
            s[i].record(stream)
            fn()
            e[i].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in zip(s, e))

    out = {}
    out["router_topk"] = timed(lambda: api.moe_router_topk(cfg, x, dinp["w_router"], dinp["bias"], fl["logits"],
                                                            fl["topk_idx"], fl["topk_gate"], layer.ws))
    row_src = fl["row_src"]
    out["permute"] = timed(lambda: api.moe_permute(cfg, x, fl["topk_idx"], fl["topk_gate"], fl["counts"],
                                                   fl["offsets"], fl["poffsets"], fl["slot_row"], row_src,
                                                   fl["row_gate"], fl["x_perm"], 0, layer.ws))
    out["fc2_grouped_gemm"] = timed(lambda: api.moe_grouped_gemm(cfg, api.GG_FC2, fl["h"], dinp["w2"], fl["o"],
                                                                 layer.ws, poffsets=fl["poffsets"]))
    out["combine"] = timed(lambda: api.moe_unpermute(cfg, fl["o"], fl["slot_row"], None, y))
    # algorithmic bytes of the two HBM-bound copies: (1+k)*T*H*2 each
    nbytes = (1 + k) * T * H * 2
    out["permute_gbs"] = nbytes / (out["permute"] / 1e3) / 1e9
    out["combine_gbs"] = nbytes / (out["combine"] / 1e3) / 1e9
    return out


# ---------------------------------------------------------------- reference arm
def run_reference(args) -> dict | None:
    world, rank, local = dist_env()
    if rank != 0:
        return None
    w = WORKLOADS[args.workload]
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
        dinp = make_inputs_on_device(w, torch.device("cuda", local), seed=0)
    else:
        dinp = make_inputs(w, seed=0)
    inp = oracle_inputs(w, dinp)
    warm_experts(w, inp, np.arange(4))
    # size the per-step sample so that W + K steps end within ~2 minutes
    t1 = oracle_step_timed(w, inp, np.arange(4)) / 4
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(w.T, per_step_budget / max(t1, 1e-6))))
    rng = np.random.default_rng(0)
    samples = [np.sort(rng.choice(w.T, n, replace=False)) for _ in range(args.warmup + args.steps)]
    warm_experts(w, inp, np.unique(np.concatenate(samples)))   # host copies of the weights, untimed
    for smp in samples[:args.warmup]:
        oracle_step_timed(w, inp, smp)
    total = 0.0
    for smp in samples[args.warmup:]:
        total += oracle_step_timed(w, inp, smp)
    value = n * args.steps / total
    sample = (f"{n} random tokens of {w.T} per step (fp64 numpy oracle, "
              f"{'forward + backward' if w.backward else 'forward'})")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "F": w.F, "S": w.S,
                   "score": w.score, "pass": "fwd+bwd" if w.backward else "fwd"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="mixtral")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch each timed step eagerly, not as a CUDA graph")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (smaller cases for profiler captures; not a bench line)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (smaller cases for profiler captures; not a bench line)")
    ap.add_argument("--profile-op", choices=sorted(PROFILE_OPS), default=None,
                    help="for profiler captures: one untimed step, then this grouped GEMM once inside "
                         "cudaProfilerStart/Stop (ncu --profile-from-start off); prints one JSON line")
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
