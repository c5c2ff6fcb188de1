"""Benchmark of the GB300 4-bit MoE layer.

One step = one whole layer (routing, expert GEMMs or GEMVs, combine) through
the C ABI over one batch of synthetic input. The headline workload is the
prefill layer at T=4096 tokens (D=2048, E=256, top-8 + 1 shared expert,
I=512, 4-bit g64 weights, Zipf(1.1) router bias); decode (T=1) µs/token is
measured in the same run and reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the workload
(the layer needs no exchange between replicas), timing is max over ranks and
the value counts every rank's tokens. --impl reference times the CPU oracle
(the slow plain definition) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s at T=4096 & decode µs/token; % of HBM/tensor roofline"
HEADLINE = "prefill4096_zipf"
L2_FLUSH_BYTES = 512 << 20  # > 126 MB L2
HOST_LEAD_CYCLES = 400_000  # GPU spin before each timed step so the host enqueues the step ahead of the GPU


# --- peaks -----------------------------------------------------------------------------------

def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def profiled_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or None
    when there is no record or the kernel source has changed since it was taken."""
    import glob
    import hashlib
    for path in glob.glob(os.path.join(ROOT, "profiles", "*_dram.txt")):
        rec = {}
        with open(path) as f:
            for line in f:
                if line.startswith("#") or ":" not in line:
                    continue
                key, val = line.split(":", 1)
                rec[key.strip()] = val.strip()
        if kernel not in rec or "source" not in rec:
            continue
        src = os.path.join(ROOT, rec["source"])
        if not os.path.exists(src):
            continue
        with open(src, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec.get("source_sha256"):
                return None
        return int(rec[kernel])
    return None


# --- distributed plumbing (replicas only) ----------------------------------------------------

def dist_env() -> tuple[int, int, int]:
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def init_dist(world: int, backend: str | None = None):
    if world <= 1:
        return None
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index] if device is not None else None)
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    dev = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    dev = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --- clocks ----------------------------------------------------------------------------------

class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons every 20 ms while running.

    The sampler is running before the caller starts timing (its first line has
    arrived), and summary() keeps only the samples stamped inside the window
    the caller marks with window_start() / window_end() (wall clock)."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self._t = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            deadline = time.time() + 5.0
            while not self.lines and time.time() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def window_start(self):
        self.t0 = time.time()

    def window_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=2)

    @staticmethod
    def _stamp(text: str):
        """Wall-clock seconds of an nvidia-smi timestamp such as 2026/12/02 13:45:01.123."""
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self) -> dict:
        rows = []
        for t_read, ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            t = self._stamp(parts[0])
            try:
                rows.append(dict(t=t if t is not None else t_read, sm=float(parts[2]), smax=float(parts[3]),
                                 active=parts[5], hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except ValueError:
                continue
        if self.t0 is not None and self.t1 is not None:
            inside = [r for r in rows if self.t0 <= r["t"] <= self.t1]
        else:
            inside = rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": rows[0]["smax"] if rows else None, "reasons": ["unsampled"],
                    "samples": 0}
        reasons = set()
        for r in inside:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        sms = sorted(r["sm"] for r in inside)
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": inside[0]["smax"], "reasons": sorted(reasons),
                "samples": len(inside), "sm_mhz_min": sms[0]}


# --- algorithmic work ------------------------------------------------------------------------

def expert_bytes(D: int, I: int) -> int:
    """Packed bytes of one expert's three matrices: 0.5 B per code + 4 B per 64-weight group."""
    per_matrix = D * I // 2 + (D * I // 64) * 4
    return 3 * per_matrix


def layer_work(layer, idx_np) -> dict:
    import numpy as np
    T, k = idx_np.shape
    D, I, E = layer.D, layer.I, layer.E
    used = int((np.bincount(idx_np.reshape(-1), minlength=E) > 0).sum())
    rows = T * k + T
    return dict(
        rows=rows, experts_touched=used + 1,
        gateup_flops=2.0 * rows * D * 2 * I, down_flops=2.0 * rows * I * D,
        weight_bytes=(used + 1) * expert_bytes(D, I),
        gateup_weight_bytes=(used + 1) * expert_bytes(D, I) * 2 // 3,
        down_weight_bytes=(used + 1) * expert_bytes(D, I) // 3,
        router_flops=2.0 * T * E * D)


def touched_weight_bytes(layer, idx_np) -> int:
    """Packed bytes of the distinct experts a batch's top-k selects, plus the shared expert."""
    import numpy as np
    return (len(np.unique(idx_np)) + 1) * expert_bytes(layer.D, layer.I)


def capture_graph(torch, device, stream, fn):
    """A CUDA graph of fn() (which launches on torch's current stream); one
    eager run on a side stream first, outside the capture."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
    stream.wait_stream(side)
    torch.cuda.synchronize(device)
    with torch.cuda.graph(g, stream=side):
        fn()
    torch.cuda.synchronize(device)
    return g


def sample_us(torch, stream, flush, fn) -> float:
    """Device µs of one fn() on `stream` between CUDA events, with L2 flushed
    before it and a GPU-side lead so the host has enqueued fn() in time."""
    flush.zero_()
    torch.cuda._sleep(HOST_LEAD_CYCLES)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    fn()
    b.record(stream)
    b.synchronize()
    return 1e3 * a.elapsed_time(b)


def med(v):
    v = sorted(v)
    return v[len(v) // 2]


def p95(v):
    v = sorted(v)
    return v[int(0.95 * (len(v) - 1))]


def run_workloads(args, moe, synth, torch, device, stream, peaks, headline: dict, decode: dict | None) -> dict:
    """The five seeded workloads side by side: µs, tokens/s and roofline
    fraction of each (C1, the tiny case, is a correctness case only), and the
    small-row sweep run on both the GEMV and the grouped-GEMM path to fix the
    row count where the GEMM takes over."""
    import ctypes

    import numpy as np
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    out = {"prefill4096_zipf": headline}
    if decode is not None:
        out["decode"] = dict(T=1, us=decode["us_per_token"], tokens_per_s=decode["tokens_per_s"],
                             bound="hbm", weight_bytes=decode["roofline"]["bytes_per_launch"],
                             frac_hbm=decode["layer_GBps_on_expert_bytes"] / peaks["hbm_gbs"],
                             timing="graph replay, median")

    def layer_forward(dl, x, y, ws, T):
        def fwd():
            sp = ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
            st = moe.moe_layer_forward(dl.w, x.data_ptr(), T, y.data_ptr(), ws.data_ptr(), ws.numel(), sp)
            if st != moe.MOE_OK:
                raise moe.MoEError(st, "moe_layer_forward")
        return fwd

    def status_ok(ws):
        st = moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
        if st != moe.MOE_OK:
            raise moe.MoEError(st, "device status")

    # C3: T=512, near-uniform routing (HBM-bound: ~all experts touched)
    layer, x_np = synth.make_config("prefill512")
    dl = moe.DeviceLayer(layer, device=device)
    T = x_np.shape[0]
    x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).to(device)
    y = torch.empty_like(x)
    ws = dl.workspace(T)
    fwd = layer_forward(dl, x, y, ws, T)
    for _ in range(3):
        fwd()
    g = capture_graph(torch, device, stream, fwd)
    n = max(args.steps, 50)
    us = [sample_us(torch, stream, flush, g.replay) for _ in range(n)]
    status_ok(ws)
    # per-kernel device times of the same layer, stream-launched
    moe.moe_kernel_times()
    moe.moe_set_option(moe.MOE_OPT_KERNEL_TIMING, 1)
    for _ in range(10):
        sample_us(torch, stream, flush, fwd)
    moe.moe_set_option(moe.MOE_OPT_KERNEL_TIMING, 0)
    kt3 = {nm: 1e3 * tms / cnt for nm, (tms, cnt) in moe.moe_kernel_times().items()}
    v = dl.view(T, ws)
    idx = moe.ws_tensor(ws, v.topk_idx, (T, layer.k), torch.int32).cpu().numpy()
    work = layer_work(layer, idx)
    t = med(us)
    out["prefill512"] = dict(
        T=T, us=t, us_p95=p95(us), tokens_per_s=T / (t / 1e6), bound="hbm", weight_bytes=work["weight_bytes"],
        experts_touched=work["experts_touched"], frac_hbm=work["weight_bytes"] / (t / 1e6) / 1e9 / peaks["hbm_gbs"],
        flops=work["gateup_flops"] + work["down_flops"],
        frac_tensor=(work["gateup_flops"] + work["down_flops"]) / (t / 1e6) / 1e12 / peaks["bf16_tflops"],
        samples=n, timing="graph replay, median; L2 flushed before each sample",
        kernel_us=kt3, block_rows=v.block_m)
    del dl, x, y, ws, g

    # C5: T in {2,3,4,5,8} on both paths, forced; graph-replayed, L2 flushed,
    # blocks of samples alternating between the paths
    layer, x_all = synth.make_config("sweep")
    dl = moe.DeviceLayer(layer, device=device)
    block = 20
    n_blocks = 2 * max(5, (args.sweep_samples + block - 1) // block)  # half of the blocks per path
    sweep = {}
    old_force = moe.moe_get_option(moe.MOE_OPT_FORCE_PATH)
    try:
        for T in synth.SWEEP_T:
            x = torch.from_numpy(np.ascontiguousarray(x_all[:T]).view(np.int16)).view(torch.bfloat16).to(device)
            graphs, wss, ys = {}, {}, {}
            for name, path in (("gemv", moe.PATH_GEMV), ("gemm", moe.PATH_GEMM)):
                moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, path)
                ys[name], wss[name] = torch.empty_like(x), dl.workspace(T)
                f = layer_forward(dl, x, ys[name], wss[name], T)
                for _ in range(3):
                    f()
                graphs[name] = capture_graph(torch, device, stream, f)
            moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, old_force)
            times = {"gemv": [], "gemm": []}
            for b in range(n_blocks):
                for name in (("gemv", "gemm") if b % 2 == 0 else ("gemm", "gemv")):
                    for _ in range(block):
                        times[name].append(sample_us(torch, stream, flush, graphs[name].replay))
            for name in wss:
                status_ok(wss[name])
            v = dl.view(T, wss["gemv"])
            idx = moe.ws_tensor(wss["gemv"], v.topk_idx, (T, layer.k), torch.int32).cpu().numpy()
            wb = touched_weight_bytes(layer, idx)
            row = dict(weight_bytes=wb, experts_touched=len(np.unique(idx)) + 1, samples=len(times["gemv"]))
            for name in ("gemv", "gemm"):
                t = med(times[name])
                row[f"{name}_us"] = t
                row[f"{name}_p95_us"] = p95(times[name])
                row[f"{name}_frac_hbm"] = wb / (t / 1e6) / 1e9 / peaks["hbm_gbs"]
            row["faster"] = "gemv" if row["gemv_us"] <= row["gemm_us"] else "gemm"  # a tie keeps the GEMV path
            sweep[str(T)] = row
            del graphs, wss, ys, x
    finally:
        moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, old_force)
    out["sweep"] = sweep
    # the switch point: the largest swept row count up to which the GEMV path
    # is at least as fast at every swept count (1 if the GEMM wins at 2 rows)
    thr = 1
    for T in synth.SWEEP_T:
        if sweep[str(T)]["faster"] != "gemv":
            break
        thr = T
    out["crossover"] = dict(measured_gemv_max_rows=thr,
                            library_default=moe.moe_get_option(moe.MOE_OPT_GEMV_MAX_ROWS),
                            rule="largest swept T with the GEMV path at least as fast at every swept T up to it",
                            timing=f"graph replay, median of {block * n_blocks // 2} samples per point, "
                                   f"L2 flushed, blocks of {block} alternating between the paths")
    return out


# --- our arm ---------------------------------------------------------------------------------

def run_ours(args) -> dict:
    import ctypes

    import numpy as np
    import torch

    import bit_moe_expert_routing_gb300 as moe
    from bit_moe_expert_routing_gb300 import build as moe_build, synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world)
    moe_build.build()
    moe.lib()
    peaks = measured_peaks()

    cfg = synth.CONFIGS[args.workload]
    layer, x_np = synth.make_config(args.workload)
    T = x_np.shape[0]
    dl = moe.DeviceLayer(layer, device=device)
    x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).to(device)
    y = torch.empty_like(x)
    ws = dl.workspace(T, host_staging=True)
    ws_bytes = ws.numel()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    sp = ctypes.c_void_p(stream.cuda_stream)

    def forward():
        st = moe.moe_layer_forward(dl.w, x.data_ptr(), T, y.data_ptr(), ws.data_ptr(), ws_bytes, sp)
        if st != moe.MOE_OK:
            raise moe.MoEError(st, "moe_layer_forward")

    moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, moe.PATH_AUTO)
    for _ in range(args.warmup):
        flush.zero_()
        forward()
    torch.cuda.synchronize(device)
    st = moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), sp)
    if st != moe.MOE_OK:
        raise moe.MoEError(st, "device status after warm-up")

    # timed region: per-step event pairs, L2 flushed between steps
    moe.moe_kernel_times()
    moe.moe_set_option(moe.MOE_OPT_KERNEL_TIMING, 1)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    launches = 0
    barrier(dist, device)
    torch.cuda.synchronize(device)
    with ClockSampler(device.index) as clk:
        clk.window_start()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            evs[i][0].record(stream)
            forward()
            evs[i][1].record(stream)
            launches += moe.moe_last_launch_count()
        torch.cuda.synchronize(device)
        t_wall = time.perf_counter() - t_wall
        clk.window_end()
    barrier(dist, device)
    moe.moe_set_option(moe.MOE_OPT_KERNEL_TIMING, 0)
    kt = moe.moe_kernel_times()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms_local = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(dist, ms_local, device)
    tokens_all = sum_over_ranks(dist, float(T), device)
    value = tokens_all / (ms / 1e3)

    # routing statistics for the algorithmic work (from the device tables of the last step)
    v = dl.view(T, ws)
    idx = moe.ws_tensor(ws, v.topk_idx, (T, layer.k), torch.int32).cpu().numpy()
    work = layer_work(layer, idx)
    kernels = {n: dict(ms_per_launch=t / c, launches=c, share=0.0) for n, (t, c) in kt.items()}
    tot = sum(t for t, _ in kt.values()) or 1.0
    for n, (t, c) in kt.items():
        kernels[n]["share"] = t / tot
    dominant = max(kernels, key=lambda n: kernels[n]["ms_per_launch"] * kernels[n]["launches"])
    flops_of = {"gateup_tc": work["gateup_flops"], "gateup_simt": work["gateup_flops"],
                "down_tc": work["down_flops"], "down_simt": work["down_flops"]}
    bytes_of = {"gemv_gateup": work["gateup_weight_bytes"], "gemv_down": work["down_weight_bytes"]}
    if dominant in flops_of:
        ach = flops_of[dominant] / (kernels[dominant]["ms_per_launch"] / 1e3) / 1e12
        roof = dict(kernel=dominant, bound="tensor", achieved=ach, peak=peaks["bf16_tflops"], unit="TFLOP/s",
                    frac=ach / peaks["bf16_tflops"], traffic=profiled_traffic(dominant),
                    peak_source=f"{peaks['source']} bf16 burst")
    elif dominant in bytes_of:
        ach = bytes_of[dominant] / (kernels[dominant]["ms_per_launch"] / 1e3) / 1e9
        roof = dict(kernel=dominant, bound="hbm", achieved=ach, peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=ach / peaks["hbm_gbs"], traffic=None, peak_source=f"{peaks['source']} copy")
    else:
        roof = dict(kernel=dominant, bound="alu", achieved=None, peak=None, unit=None, frac=None, traffic=None)
    whole = max(work["gateup_flops"] + work["down_flops"], 1.0) / (ms / 1e3) / 1e12

    # e2e through the host-buffer entry point (pinned host x and y)
    xh = torch.from_numpy(x_np.view(np.int16).copy()).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    e2e_ms = []
    for i in range(args.steps + 2):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        r = moe.moe_layer_forward_host(dl.w, xh.data_ptr(), T, yh.data_ptr(), ws.data_ptr(), ws_bytes, sp)
        if r != moe.MOE_OK:
            raise moe.MoEError(r, "moe_layer_forward_host")
        b.record(stream)
        b.synchronize()
        if i >= 2:
            e2e_ms.append(a.elapsed_time(b))
    e2e_ms_v = max_over_ranks(dist, sum(e2e_ms) / len(e2e_ms), device)
    e2e = dict(value=sum_over_ranks(dist, float(T), device) / (e2e_ms_v / 1e3), unit="tokens/s",
               h2d_bytes_per_step=T * layer.D * 2, d2h_bytes_per_step=T * layer.D * 2, ms_per_step=e2e_ms_v)

    decode = run_decode(args, moe, synth, torch, device, stream, peaks) if not args.no_decode else None
    headline = dict(T=T, us=ms * 1e3, tokens_per_s=T / (ms / 1e3), bound="tensor",
                    flops=work["gateup_flops"] + work["down_flops"], frac_tensor=whole / peaks["bf16_tflops"],
                    weight_bytes=work["weight_bytes"],
                    frac_hbm=work["weight_bytes"] / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                    experts_touched=work["experts_touched"], samples=args.steps,
                    timing="stream-launched, mean of the timed steps; L2 flushed before each")
    workloads = None
    if not args.no_workloads and rank == 0 and world == 1:
        workloads = run_workloads(args, moe, synth, torch, device, stream, peaks, headline, decode)

    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: T={T} D={layer.D} E={layer.E} top-{layer.k} + 1 shared "
                               f"I={layer.I}, 4-bit g64 codes, bf16 scale/bias"
                               + (f", Zipf({cfg['zipf_s']}) router bias" if cfg["zipf_s"] else "")
                               + f", seed {cfg['seed']}",
                   "T": T, "D": layer.D, "E": layer.E, "k": layer.k, "I": layer.I,
                   "l2": "flushed between steps (512 MiB write outside the timed events)",
                   "parallelism": f"replicas x{world}", "gemm_impl": "tcgen05" if moe.moe_get_option(
                       moe.MOE_OPT_GEMM_IMPL) == 0 else "cuda-core",
                   "experts_touched": work["experts_touched"],
                   "workspace_bytes": dl.workspace_bytes(T),
                   "chunk_tokens": moe.moe_get_option(moe.MOE_OPT_CHUNK_TOKENS)},
        "roofline": roof,
        "layer_tflops": whole,
        "kernels": kernels,
        "e2e": e2e,
        "gpu_launches": launches,
        "wall_s_timed": t_wall,
        "clocks": clk.summary(),
        "decode": decode,
        "workloads": workloads,
        "peaks": peaks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(layer, x_np, args.cpu_seconds)
    return out if rank == 0 else None


def run_decode(args, moe, synth, torch, device, stream, peaks) -> dict:
    """Decode (T=1) µs/token with L2 flushed between steps: stream-launched
    (per-kernel events) and replayed from a CUDA graph (the layer as a decode
    loop would run it). GEMV kernels are measured against HBM bandwidth."""
    import ctypes

    import numpy as np
    layer, x_np = synth.make_config("decode")
    dl = moe.DeviceLayer(layer, device=device)
    x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).to(device)
    y = torch.empty_like(x)
    ws = dl.workspace(1)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, moe.PATH_AUTO)

    def fwd():
        sp = ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
        st = moe.moe_layer_forward(dl.w, x.data_ptr(), 1, y.data_ptr(), ws.data_ptr(), ws.numel(), sp)
        if st != moe.MOE_OK:
            raise moe.MoEError(st, "decode forward")

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        fwd()
    torch.cuda.synchronize(device)
    n = max(args.steps, 50)

    def timed(step, cold=True):
        ms = []
        for _ in range(n):
            if cold:
                flush.zero_()
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return sorted(ms)

    moe.moe_kernel_times()
    moe.moe_set_option(moe.MOE_OPT_KERNEL_TIMING, 1)
    ms = timed(fwd)
    moe.moe_set_option(moe.MOE_OPT_KERNEL_TIMING, 0)
    kt = moe.moe_kernel_times()
    launches = moe.moe_last_launch_count()

    # CUDA-graph replay of the same call
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fwd()
    stream.wait_stream(side)
    torch.cuda.synchronize(device)
    with torch.cuda.graph(g, stream=side):
        fwd()
    torch.cuda.synchronize(device)
    ms_g = timed(g.replay)
    ms_w = timed(g.replay, cold=False)  # warm: the 18 MB working set stays in L2 between steps

    v = dl.view(1, ws)
    idx = moe.ws_tensor(ws, v.topk_idx, (1, layer.k), torch.int32).cpu().numpy()
    work = layer_work(layer, idx)
    med = lambda m: m[len(m) // 2]
    us, us_g = 1e3 * med(ms), 1e3 * med(ms_g)
    kern = {nm: dict(ms_per_launch=t / c, launches=c) for nm, (t, c) in kt.items()}
    # the one-launch kernel that ran (one token, or 2..8 rows), else the two GEMV kernels
    names = next(((nm,) for nm in ("decode_fused", "decode_items", "decode_rows") if nm in kern),
                 ("gemv_gateup", "gemv_down"))
    gemv_ms = sum(kern[nm]["ms_per_launch"] for nm in names if nm in kern)
    ach = work["weight_bytes"] / (gemv_ms / 1e3) / 1e9 if gemv_ms else None
    return {"us_per_token": us_g, "us_per_token_warm": 1e3 * med(ms_w), "us_per_token_stream": us,
            "us_p95_stream": 1e3 * ms[int(0.95 * (n - 1))],
            "us_p95": 1e3 * ms_g[int(0.95 * (n - 1))], "steps": n, "tokens_per_s": 1e6 / us_g,
            "launches_per_step": launches,
            "roofline": dict(kernel="+".join(names), bound="hbm", achieved=ach, peak=peaks["hbm_gbs"],
                             unit="GB/s", frac=(ach / peaks["hbm_gbs"]) if ach else None,
                             traffic=profiled_traffic(names[0]) if len(names) == 1 else None,
                             bytes_per_launch=work["weight_bytes"],
                             peak_source=f"{peaks['source']} copy"),
            "layer_GBps_on_expert_bytes": work["weight_bytes"] / (us_g / 1e6) / 1e9,
            "kernels": kern, "l2": "flushed between steps", "timing": "median; graph replay for us_per_token"}


# --- the oracle (CPU baseline and the reference arm) ------------------------------------------

def cpu_baseline(layer, x_np, seconds: float) -> dict:
    """The oracle, as it stands, on a bounded sample of the workload's tokens."""
    import numpy as np

    from oracle import oracle as O
    ol = O.OracleLayer(layer)
    cores = O.threads_used(0)
    n = cores
    t0 = time.perf_counter()
    O.forward(ol, x_np, tokens=np.arange(n, dtype=np.int32), n_threads=cores)
    dt = time.perf_counter() - t0
    reps = max(1, int(seconds / max(dt, 1e-3)))
    toks = min(x_np.shape[0], n * reps)
    t0 = time.perf_counter()
    O.forward(ol, x_np, tokens=np.arange(toks, dtype=np.int32), n_threads=cores)
    dt = time.perf_counter() - t0
    # and on one core, a small sample
    n1 = max(2, min(16, int(2.0 * toks / dt / cores)))
    t0 = time.perf_counter()
    O.forward(ol, x_np, tokens=np.arange(n1, dtype=np.int32), n_threads=1)
    dt1 = time.perf_counter() - t0
    return {"value": toks / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {toks} of {x_np.shape[0]} tokens of the same layer, fp64 plain C++ oracle, "
                      f"{cores} threads, {dt:.1f} s",
            "one_core": {"value": n1 / dt1, "unit": "tokens/s", "sample": f"first {n1} tokens, 1 thread, {dt1:.1f} s"}}


def run_reference(args) -> dict | None:
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import numpy as np

    from bit_moe_expert_routing_gb300 import synth
    from oracle import oracle as O
    O.build()
    cfg = synth.CONFIGS[args.workload]
    layer, x_np = synth.make_config(args.workload)
    T = x_np.shape[0]
    ol = O.OracleLayer(layer)
    cores = O.threads_used(0)
    per_step = cores  # bounded sample: one token per core per step
    for i in range(args.warmup):
        O.forward(ol, x_np, tokens=(np.arange(per_step) + i * per_step) % T, n_threads=cores)
    t0 = time.perf_counter()
    for i in range(args.steps):
        O.forward(ol, x_np, tokens=(np.arange(per_step) + i * per_step) % T, n_threads=cores)
    dt = time.perf_counter() - t0
    ms = dt / args.steps * 1e3
    value = per_step / (ms / 1e3)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: T={T} D={layer.D} E={layer.E} top-{layer.k} + 1 shared "
                               f"I={layer.I}" + (f", Zipf({cfg['zipf_s']})" if cfg["zipf_s"] else ""),
                   "T": T, "sample_tokens_per_step": per_step},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} tokens per step of the {T}-token workload"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# --- ablations of the source pages' design claims (--ablations) ----------------------------

def run_ablations(args) -> dict:
    """GB300 measurements of the design choices the pages ablate ("Optimizing
    on-device inference for Apple Silicon": "Keep expert routing on the GPU",
    "Match tile size to expert load", "Dequantise weights during matrix
    multiplication"), each against this build's default on the same seeded
    workloads. Every figure is a median over steps with L2 flushed between
    them; one GPU, rank 0 only."""
    import ctypes

    import numpy as np
    import torch

    import bit_moe_expert_routing_gb300 as moe
    from bit_moe_expert_routing_gb300 import build as moe_build, synth

    rank, world, local = dist_env()
    if rank != 0:
        return None
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    moe_build.build()
    moe.lib()
    stream = torch.cuda.current_stream(device)
    sp = ctypes.c_void_p(stream.cuda_stream)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    steps = max(args.steps, 10)
    layers = {}

    def layer_of(name):
        if name not in layers:
            layer, x_np = synth.make_config(name)
            dl = moe.DeviceLayer(layer, device=device)
            x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).to(device)
            layers[name] = (layer, x_np, dl, x, torch.empty_like(x))
        return layers[name]

    def layer_ms(name, opts=None):
        """Median ms of one forward of workload `name` with library options {option: value} set."""
        opts = opts or {}
        layer, x_np, dl, x, y = layer_of(name)
        old = {k: moe.moe_get_option(k) for k in opts}
        try:
            for k, v in opts.items():
                if moe.moe_set_option(k, v) != moe.MOE_OK:
                    raise moe.MoEError(moe.MOE_ERR_ARG, f"option {k}={v}")
            T = x.shape[0]
            ws = dl.workspace(T)
            ms = []
            for i in range(3 + steps):
                flush.zero_()
                torch.cuda._sleep(HOST_LEAD_CYCLES)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                st = moe.moe_layer_forward(dl.w, x.data_ptr(), T, y.data_ptr(), ws.data_ptr(), ws.numel(), sp)
                if st != moe.MOE_OK:
                    raise moe.MoEError(st, "moe_layer_forward")
                b.record(stream)
                b.synchronize()
                if i >= 3:
                    ms.append(a.elapsed_time(b))
            st = moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), sp)
            if st != moe.MOE_OK:
                raise moe.MoEError(st, "device status")
            return sorted(ms)[len(ms) // 2]
        finally:
            for k, v in old.items():
                moe.moe_set_option(k, v)

    moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, moe.PATH_AUTO)
    out = {}
    # 1. routing tables built on the GPU in stream order vs a host round trip
    #    (block count copied back, stream synchronised) before the expert kernels
    out["routing"] = {}
    for name in ("prefill512", "prefill4096_zipf"):
        g = layer_ms(name)
        h = layer_ms(name, {moe.MOE_OPT_HOST_SYNC_ROUTING: 1})
        out["routing"][name] = dict(gpu_resident_ms=g, host_sync_ms=h, speedup=h / g)
    # 2. rows per block-map entry (the GEMM's token tile)
    out["block_rows"] = {}
    for name in ("prefill512", "prefill4096_zipf"):
        out["block_rows"][name] = {str(bm): layer_ms(name, {moe.MOE_OPT_BLOCK_M: bm})
                                   for bm in (16, 32, 64, 128, 192)}
    # 3. operand roles: dequantised weights as the MMA's M (tensor memory, the
    #    default) vs tokens as M (weights in shared memory), and CUDA cores
    out["gemm_impl"] = {}
    for name in ("prefill512", "prefill4096_zipf"):
        out["gemm_impl"][name] = {
            "weights_as_M_tcgen05": layer_ms(name, {moe.MOE_OPT_GEMM_IMPL: moe.GEMM_TENSOR_CORE}),
            "tokens_as_M_tcgen05": layer_ms(name, {moe.MOE_OPT_GEMM_IMPL: moe.GEMM_TENSOR_CORE_SMEM}),
            "cuda_cores": layer_ms(name, {moe.MOE_OPT_GEMM_IMPL: moe.GEMM_CUDA_CORE})}
    # 4. separate dequantisation: the unfused layer (routing; a pass that
    #    expands every selected expert's and the shared expert's weights to
    #    bf16 in HBM; grouped GEMMs reading those bf16 weights through TMA)
    #    against the fused layers: the same shared-memory GEMM dequantising on
    #    chip, and the default tensor-memory GEMM
    layer, x_np, dl, x, y = layer_of("prefill4096_zipf")
    T = x.shape[0]
    ws = dl.workspace(T)
    nb = moe.moe_expanded_weights_bytes(dl.w)
    wbuf = torch.empty(nb, dtype=torch.uint8, device=device)
    ms = []
    moe.moe_kernel_times()
    for i in range(3 + steps):
        flush.zero_()
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        if i == 3:
            moe.moe_set_option(moe.MOE_OPT_KERNEL_TIMING, 1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        st = moe.moe_layer_forward_expanded(dl.w, x.data_ptr(), T, y.data_ptr(), ws.data_ptr(), ws.numel(),
                                            wbuf.data_ptr(), nb, sp)
        if st != moe.MOE_OK:
            raise moe.MoEError(st, "moe_layer_forward_expanded")
        b.record(stream)
        b.synchronize()
        if i >= 3:
            ms.append(a.elapsed_time(b))
    moe.moe_set_option(moe.MOE_OPT_KERNEL_TIMING, 0)
    kt = {nm: 1e3 * tms / steps for nm, (tms, cnt) in moe.moe_kernel_times().items()}  # us per step
    st = moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), sp)
    if st != moe.MOE_OK:
        raise moe.MoEError(st, "device status")
    v = dl.view(T, ws)
    count = moe.ws_tensor(ws, v.count, (layer.E,), torch.int32).cpu().numpy()
    n_exp = int(np.count_nonzero(count)) + 1
    del wbuf
    written = n_exp * 3 * layer.D * layer.I * 2
    read = n_exp * expert_bytes(layer.D, layer.I)
    out["separate_dequant"] = dict(
        workload="prefill4096_zipf", experts=n_exp, unfused_layer_ms=sorted(ms)[len(ms) // 2],
        unfused_kernel_us_per_step={k: round(v, 2) for k, v in kt.items()},
        expansion_bf16_bytes_written=written, expansion_packed_bytes_read=read,
        expansion_hbm_floor_ms=(written + read) / (measured_peaks()["hbm_gbs"] * 1e9) * 1e3,
        fused_same_gemm_ms=layer_ms("prefill4096_zipf", {moe.MOE_OPT_GEMM_IMPL: moe.GEMM_TENSOR_CORE_SMEM}),
        fused_default_ms=layer_ms("prefill4096_zipf"))
    # 5. one token: the single fused kernel vs routing + two GEMV kernels
    out["decode"] = dict(fused_ms=layer_ms("decode", {moe.MOE_OPT_DECODE_FUSED: 1}),
                         separate_ms=layer_ms("decode", {moe.MOE_OPT_DECODE_FUSED: 0}))
    return {"ablations": out, "steps": steps, "l2": "flushed between steps",
            "timing": "median of CUDA-event step times, stream-launched"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the 512-token layer and the small-row GEMV/GEMM sweep")
    ap.add_argument("--sweep-samples", type=int, default=200, help="samples per (row count, path) of the sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ablations", action="store_true",
                    help="print GB300 measurements of the pages' ablated design choices instead")
    args = ap.parse_args(argv)
    if args.impl == "ours":
        args.warmup = max(args.warmup, 3)  # at least three untimed steps
    if args.ablations:
        out = run_ablations(args)
    else:
        out = run_reference(args) if args.impl == "reference" else run_ours(args)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
