#!/usr/bin/env python
"""Benchmark of the DLR layer on GB300.

One step = one pass of the whole DLR hot path over one batch: the layer u -> y on the
B=8, H=256, N=64, L=4096 bank (float32 inputs, synthetic seeded data resident in HBM) through
dlr_scan -- the per-channel table kernel and the tensor-core chunked scan kernel, replayed as
one CUDA graph. L2 is flushed (a 2 x L2 write, then a 1.5 x L2 read so that no dirty line is
left for the step to write back) before every step; the flush is outside the
timed events. The FFT path of the same layer (dlr_kernel + dlr_conv_spectrum + dlr_conv_apply)
and the other workloads are reported as secondary lines.

Prints ONE JSON line (rank 0). Multi-GPU (torchrun): every rank runs its own batch (weak
scaling, no data-path collective); a barrier and a max-over-ranks reduction bracket the timing.

--impl reference times the float64 CPU oracle (the reference arm) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
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

WORKLOAD = "dlr_b8_h256_n64_l4096"
METRIC = "DLR layer elements/s (B*H*L/s) and achieved HBM GB/s vs peak, 1xGB300"
UNIT = "elements/s"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
SCAN_TC_SOURCES = ["state_space_sequence_gb300/csrc/dlr_scan_tc.cu",
                   "state_space_sequence_gb300/csrc/tc_ptx.cuh",
                   "state_space_sequence_gb300/csrc/dlr_common.cuh"]
CONV_SOURCES = ["state_space_sequence_gb300/csrc/dlr_conv.cu",
                "state_space_sequence_gb300/csrc/fft_smem.cuh",
                "state_space_sequence_gb300/csrc/fft_rows.cuh",
                "state_space_sequence_gb300/csrc/dlr_common.cuh"]


def source_hash(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling): seed offset by the rank."""
    return base + 1000 * rank


def aggregate(per_rank_seconds, units_per_rank: int):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    t = max(per_rank_seconds)
    return units_per_rank * len(per_rank_seconds) / t, t


def load_sm_max_mhz() -> float:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return float(json.load(fh).get("sm_max_mhz", 2070.0))
    return 2070.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_tensor_peak():
    """Dense f16/bf16 tensor throughput (TFLOP/s), burst figure: the step is timed alone.
    f16 and bf16 share one nominal rate, so the measured bf16 GEMM stands for both."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured (bf16 burst; f16 has the same rate)"
    return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed loop runs."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-i", str(self.index), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = self.samples
        if self.window is not None:
            inside = [r for r in rows if self.window[0] <= r[0] <= self.window[1]]
            rows = inside or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1][0]) for r in rows if r[1][0].replace(".", "").isdigit()]
        mx = [float(r[1][1]) for r in rows if r[1][1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[1][2 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------------------------
def run_ours(args):
    import torch
    from state_space_sequence_gb300 import dlr, inputs

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    cfg = dict(inputs.WORKLOADS[WORKLOAD])
    B, H, N, L = cfg["B"], cfg["H"], cfg["N"], cfg["L"]
    w = inputs.make_dlr(B, H, N, L, seed=rank_seed(cfg["seed"], rank))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    u = dev(w.u)
    fwd = (dev(w.fwd.log_re), dev(w.fwd.log_im), dev(w.fwd.W))
    ws = torch.empty(dlr.dlr_scan_workspace_size(B, H, N, L), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(u)
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20) or (128 << 20))
    flush = L2Flush(torch, l2)
    stream = torch.cuda.current_stream()

    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step():
        dlr.dlr_scan(u, fwd, out=y, algo="tensor", workspace=ws)

    for _ in range(3):  # eager: loads the module, sets kernel attributes
        step()
    torch.cuda.synchronize()
    # The step's launches are recorded once in a CUDA graph and replayed, so the timing holds no
    # host-side launch gaps.
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        step()
    for _ in range(args.warmup):
        flush()
        g_step.replay()
    torch.cuda.synchronize()
    if dlr.device_status() != 0:
        raise RuntimeError("device status non-zero after warm-up")

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    starts, ends = [], []
    for _ in range(args.steps):
        flush()
        s, e = ev(), ev()
        s.record(stream)
        g_step.replay()
        e.record(stream)
        starts.append(s), ends.append(e)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist is not None:
        dist.barrier()
    sampler.window = (t_wall0, t_wall1)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_s = sum(step_ms) / 1e3
    if dist is not None:
        t = torch.tensor([total_s], dtype=torch.float64, device="cuda")
        gathered = [torch.zeros_like(t) for _ in range(world)]
        dist.all_gather(gathered, t)
        per_rank = [float(g.item()) for g in gathered]
    else:
        per_rank = [total_s]
    units = B * H * L * args.steps
    value, t_max = aggregate(per_rank, units)

    # the dominant kernel alone: dlr_scan_apply with the tables the step left in the workspace
    # (the same launch the step makes after its table kernel), in its own graph and loop
    g_apply = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_apply):
        dlr.dlr_scan_apply(u, ws, N, out=y)
    apply_ms = _time_steps(torch, g_apply.replay, max(20, min(args.steps, 500)), 3, flush,
                           reduce=statistics.fmean)

    # end to end through the public API with host buffers (pinned), copies inside the timing:
    # dlr_scan_host copies u and the parameters in, runs the layer and copies y out in pieces
    # on three streams, ordered after the start event and before the end event on `stream`
    u_h = torch.from_numpy(w.u).pin_memory()
    p_h = tuple(torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W))
    y_h = torch.empty(u_h.shape, dtype=torch.float32).pin_memory()
    ws_h = torch.empty(dlr.dlr_scan_host_workspace_size(B, H, N, L), dtype=torch.uint8,
                       device="cuda")
    e2e_steps = min(args.steps, 200)
    e2e_ms = []
    for i in range(e2e_steps + 3):
        flush()
        s, e = ev(), ev()
        s.record(stream)
        dlr.dlr_scan_host(u_h, p_h, y_h, ws_h, stream=stream)
        e.record(stream)
        if i >= 3:
            e2e_ms.append((s, e))
    torch.cuda.synchronize()
    e2e_total = sum(s.elapsed_time(e) for s, e in e2e_ms) / 1e3
    e2e_value = B * H * L * e2e_steps / e2e_total
    h2d = u_h.numel() * 4 + sum(t.numel() * 4 for t in p_h)
    d2h = y_h.numel() * 4
    if dlr.device_status() != 0:
        raise RuntimeError("device status non-zero after timing")

    sampler.stop()
    clocks = sampler.summary() if rank == 0 else None

    # Roofline of the dominant kernel (dlr_scan_tc_kernel, timed alone above; the table kernel
    # is the rest of the step). Algorithmic bytes: u read + y written once, plus the
    # parameters. The tensor view: 320 multiply-adds per output element (2N chunk states + T
    # Toeplitz + 2N carried-state outputs at N = 64, T = 64), each executed as three f16 MMAs
    # (hi*hi + hi*lo + lo*hi).
    step_avg = total_s / args.steps
    apply_s = apply_ms / 1e3
    layer_bytes = 4 * B * H * L * 2 + 4 * H * N * 4  # u + y + (log_re, log_im, W)
    peak_gbs, peak_kind = load_peaks()
    achieved = layer_bytes / apply_s / 1e9
    achieved_step = layer_bytes / step_avg / 1e9
    macs = B * H * L * (2 * 2 * N + 64)
    tc_flops = 3 * 2 * macs
    tc_peak, tc_kind = load_tensor_peak()
    traffic = None
    if os.path.exists(PROFILE_TRAFFIC):
        with open(PROFILE_TRAFFIC) as fh:
            prof = json.load(fh)
        entry = prof.get("dlr_scan_tc_kernel")
        if entry and entry.get("source_hash") == source_hash(SCAN_TC_SOURCES):
            traffic = entry.get("dram_bytes_per_launch")

    extras = {}
    if rank == 0 and world == 1 and not args.no_extras:
        extras = run_extras(torch, dlr, inputs, flush, load_sm_max_mhz(),
                            props.multi_processor_count)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    cpu = None if world > 1 or args.no_cpu_baseline else cpu_baseline(w)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; DLR init of the pages, u ~ N(0,1))",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "L": L, "path": "scan",
                   "cast": "re", "causal": True, "parallelism": f"replicas x{world}",
                   "l2": "flushed before every step (a 2 x L2 write, then a 1.5 x L2 read so that no dirty lines remain), flush outside the events",
                   "step": "dlr_scan (tensor-core path): per-channel table kernel + chunked "
                           "scan kernel, replayed as one CUDA graph"},
        "layer_hbm": {"algorithmic_bytes": layer_bytes, "achieved_gbs": achieved_step,
                      "frac_of_measured_peak": achieved_step / peak_gbs,
                      "note": "whole step (table kernel + scan kernel)"},
        "roofline": {"kernel": "dlr_scan_tc_kernel (dlr_scan_apply)",
                     "bound": "hbm", "achieved": achieved, "peak": peak_gbs,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak_gbs,
                     "traffic": traffic, "algorithmic_bytes": layer_bytes,
                     "avg_launch_us": apply_s * 1e6, "avg_step_us": step_avg * 1e6,
                     "tensor": {"executed_flops": tc_flops,
                                "achieved": tc_flops / apply_s / 1e12, "peak": tc_peak,
                                "peak_kind": tc_kind, "unit": "TFLOP/s",
                                "frac": tc_flops / apply_s / 1e12 / tc_peak}},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "call": "dlr_scan_host (pinned host buffers)",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "paths": extras,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


class L2Flush:
    """Evicts the step's data from L2 between timed steps: writes a buffer of twice the L2 size,
    then reads another of 1.5 times the L2 size, so that L2 ends up holding unrelated clean lines
    (a write alone would leave up to a whole L2 of dirty lines whose write-back the next timed
    step would pay for)."""

    def __init__(self, torch, l2_bytes: int):
        self.torch = torch
        self.wbuf = torch.empty(2 * l2_bytes // 4 + 1024, dtype=torch.float32, device="cuda")
        self.rbuf = torch.ones(3 * l2_bytes // 8 + 1024, dtype=torch.float32, device="cuda")
        self.acc = torch.empty((), dtype=torch.float32, device="cuda")

    def __call__(self):
        self.wbuf.zero_()
        self.torch.sum(self.rbuf, dim=0, out=self.acc)


def _time_steps(torch, fn, steps, warmup, flush, reduce=statistics.median):
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    ms = []
    for _ in range(steps):
        flush()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        ms.append((s, e))
    torch.cuda.synchronize()
    return reduce([s.elapsed_time(e) for s, e in ms])


def run_extras(torch, dlr, inputs, flush, sm_mhz, sm_count):
    """Secondary lines: the FFT path and the float32 scan on the same bank, and the other
    workloads."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = {}
    w = inputs.make_workload(WORKLOAD)
    B, H, L = w.B, w.H, w.L
    u, fwd = dev(w.u), (dev(w.fwd.log_re), dev(w.fwd.log_im), dev(w.fwd.W))
    y = torch.empty_like(u)
    # FFT layer: dlr_kernel + dlr_conv_spectrum + dlr_conv_apply, one CUDA graph; and the
    # convolution kernel alone (it is bound by FP32 arithmetic: a real FFT of size M counts
    # 2.5 M log2 M flops, forward + inverse 5 M log2 M, plus 6 flops per spectral bin)
    K = torch.empty((H, L), dtype=torch.float32, device="cuda")
    wsf = torch.empty(dlr.dlr_conv_workspace_size(H, L), dtype=torch.uint8, device="cuda")

    def fft_step():
        dlr.dlr_kernel(*fwd, L, "re", out=K)
        dlr.dlr_conv_spectrum(K, workspace=wsf)
        dlr.dlr_conv_apply(u, wsf, out=y)

    for _ in range(3):
        fft_step()
    torch.cuda.synchronize()
    g_fft, g_apply = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_fft):
        fft_step()
    with torch.cuda.graph(g_apply):
        dlr.dlr_conv_apply(u, wsf, out=y)
    ms = _time_steps(torch, g_fft.replay, 20, 3, flush)
    ms_apply = _time_steps(torch, g_apply.replay, 20, 3, flush)
    n = 1 << max(0, int(np.ceil(np.log2(L))))
    M = 2 * n
    apply_flops = B * H * (5 * M * np.log2(M) + 6 * (M // 2 + 1))
    peak_tflops = sm_count * 128 * 2 * sm_mhz * 1e6 / 1e12
    out["fft_" + WORKLOAD] = {
        "ms": ms, "elements_per_s": B * H * L / ms * 1e3,
        "conv_apply_us": ms_apply * 1e3,
        "conv_apply_tflops": apply_flops / ms_apply / 1e9,
        "conv_apply_frac_of_fp32_peak": apply_flops / ms_apply / 1e9 / peak_tflops}
    # the same layer with the spectra evaluated straight from the parameters
    # (dlr_conv_spectrum_direct + dlr_conv_apply: no kernel, no spectrum FFT)
    def direct_step():
        dlr.dlr_conv_spectrum_direct(fwd, None, L=L, workspace=wsf)
        dlr.dlr_conv_apply(u, wsf, out=y)

    ms_d = _time_steps(torch, direct_step, 10, 2, flush)
    ms_s = _time_steps(torch, lambda: dlr.dlr_conv_spectrum_direct(fwd, None, L=L, workspace=wsf),
                       10, 2, flush)
    out["fft_direct_spectrum_" + WORKLOAD] = {
        "ms": ms_d, "elements_per_s": B * H * L / ms_d * 1e3, "spectrum_ms": ms_s}
    del K, wsf
    ms = _time_steps(torch, lambda: dlr.dlr_scan(u, fwd, out=y, algo="fp32"), 20, 3, flush)
    out["scan_fp32_" + WORKLOAD] = {"ms": ms, "elements_per_s": B * H * L / ms * 1e3}
    # the recurrent mode (dlr_step) on the same bank: one sample per call (decode: the state
    # is read and written once, with the per-channel tables), and the whole sequence in one
    # call from a zero state (sequential in the samples)
    N = w.N
    wss = dlr.dlr_step_prepare(fwd)
    xs = torch.zeros((B, H, N, 2), dtype=torch.float32, device="cuda")
    u1, y1 = u[:, :, :1].contiguous(), torch.empty((B, H, 1), dtype=torch.float32, device="cuda")
    us_dec = _time_steps(torch, lambda: dlr.dlr_step(u1, wss, xs, out=y1), 50, 5, flush) * 1e3
    dec_bytes = 2 * B * H * N * 8 + 2 * B * H * 4 + H * N * 24
    ms = _time_steps(torch, lambda: (xs.zero_(), dlr.dlr_step(u, wss, xs, out=y)), 10, 2, flush)
    peak_gbs, peak_kind = load_peaks()
    out["step_" + WORKLOAD] = {
        "decode_us": us_dec, "decode_bytes": dec_bytes,
        "decode_gbs": dec_bytes / us_dec / 1e3,
        "decode_frac": dec_bytes / us_dec / 1e3 / peak_gbs, "peak_kind": peak_kind,
        "sequence_ms": ms, "sequence_elements_per_s": B * H * L / ms * 1e3}
    # the backward pass of the same layer for an output gradient g: the input gradient (the
    # tensor-core scan's reversed pass) and the parameter gradients (the lag correlation of g
    # with u by transforms, then its power sums per state)
    g = torch.randn_like(u)
    du = torch.empty_like(u)
    wsb = torch.empty(dlr.dlr_scan_workspace_size(B, H, N, L), dtype=torch.uint8, device="cuda")
    wsp = torch.empty(dlr.dlr_scan_backward_params_workspace_size(B, H, N, L), dtype=torch.uint8,
                      device="cuda")
    ms_in = _time_steps(torch, lambda: dlr.dlr_scan_backward_input(g, fwd, workspace=wsb,
                                                                   out=du), 10, 2, flush)
    ms_par = _time_steps(torch, lambda: dlr.dlr_scan_backward_params(u, g, fwd, workspace=wsp),
                         10, 2, flush)
    out["backward_" + WORKLOAD] = {
        "input_ms": ms_in, "params_ms": ms_par, "ms": ms_in + ms_par,
        "elements_per_s": B * H * L / (ms_in + ms_par) * 1e3}
    del u, y, xs, wss, g, du, wsb, wsp

    w = inputs.make_workload("dlrprod_bidir_b4_h128_n1024_l16384")
    u = dev(w.u)
    f = (dev(w.fwd.log_re), dev(w.fwd.log_im), dev(w.fwd.W))
    b = (dev(w.bwd.log_re), dev(w.bwd.log_im), dev(w.bwd.W))
    y = torch.empty_like(u)
    ws = torch.empty(dlr.dlr_conv_workspace_size(w.H, w.L, True), dtype=torch.uint8,
                     device="cuda")
    ms = _time_steps(torch, lambda: dlr.dlr_layer(u, f, b, cast="re_im", workspace=ws, out=y),
                     10, 2, flush)
    out["fft_" + w.name] = {"ms": ms, "elements_per_s": w.B * w.H * w.L / ms * 1e3}
    # the kernel generator alone (N >= 256: the tensor-core generator), both directions. Per
    # channel it is a real [L/64 x 2N] x [2N x 128] product (64 lags of Re K and Im K per
    # chunk row), 8 N L flops, executed as three f16 products (hi*hi + hi*lo + lo*hi)
    Kf = torch.empty((w.H, w.L), dtype=torch.float32, device="cuda")
    Kb = torch.empty_like(Kf)
    ms_k = _time_steps(torch, lambda: (dlr.dlr_kernel(*f, w.L, "re_im", out=Kf),
                                       dlr.dlr_kernel(*b, w.L, "re_im", out=Kb)), 10, 3, flush)
    kgen_flops = 2 * 3 * 8 * w.N * w.L * w.H
    tc_peak, tc_kind = load_tensor_peak()
    out["kernel_gen_tc_" + w.name] = {
        "ms": ms_k, "directions": 2, "executed_flops": kgen_flops,
        "tensor": {"achieved": kgen_flops / ms_k / 1e9, "peak": tc_peak, "peak_kind": tc_kind,
                   "unit": "TFLOP/s", "frac": kgen_flops / ms_k / 1e9 / tc_peak}}
    # the same layer's gradients (du and both directions' parameter gradients, DLR-prod cast)
    g = torch.randn_like(u)
    wsg = torch.empty(dlr.dlr_layer_backward_workspace_size(w.B, w.H, w.N, w.L, True, "re_im"),
                      dtype=torch.uint8, device="cuda")
    ms_g = _time_steps(torch, lambda: dlr.dlr_layer_backward(u, g, f, b, cast="re_im",
                                                             workspace=wsg), 5, 2, flush)
    out["backward_" + w.name] = {"ms": ms_g, "elements_per_s": w.B * w.H * w.L / ms_g * 1e3,
                                 "outputs": "du and both directions' parameter gradients"}
    del u, y, ws, Kf, Kb, g, wsg

    w = inputs.make_workload("dlr_b1_h256_n64_l65536_unit8")
    u, fwd = dev(w.u), (dev(w.fwd.log_re), dev(w.fwd.log_im), dev(w.fwd.W))
    y = torch.empty_like(u)
    ms = _time_steps(torch, lambda: dlr.dlr_scan(u, fwd, out=y), 10, 2, flush)
    out["scan_tensor_" + w.name] = {"ms": ms, "elements_per_s": w.B * w.H * w.L / ms * 1e3}
    ws = torch.empty(dlr.dlr_conv_workspace_size(w.H, w.L), dtype=torch.uint8, device="cuda")
    ms = _time_steps(torch, lambda: dlr.dlr_layer(u, fwd, path="fft", workspace=ws, out=y), 10,
                     2, flush)
    out["fft_cluster_" + w.name] = {"ms": ms, "elements_per_s": w.B * w.H * w.L / ms * 1e3}
    ms = _time_steps(torch, lambda: (dlr.dlr_conv_spectrum_direct(fwd, None, L=w.L, workspace=ws),
                                     dlr.dlr_conv_apply(u, ws, out=y)), 5, 2, flush)
    out["fft_cluster_direct_spectrum_" + w.name] = {
        "ms": ms, "elements_per_s": w.B * w.H * w.L / ms * 1e3}
    del u, y, ws

    w = inputs.make_workload("s5_b8_l16384_h512_p256")
    p = w.params
    u = dev(w.u)
    args5 = (dev(p.lam), dev(p.log_delta), dev(p.Bt), dev(p.Ct), dev(p.D))
    ws = torch.empty(dlr.s5_workspace_size(w.B, w.L, w.H, w.P), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty_like(u)
    ms = _time_steps(torch, lambda: dlr.s5_layer(u, *args5, workspace=ws, out=y), 10, 3, flush)
    # both projections as three tf32 products (kind::tf32 runs at half the f16 rate, so the
    # peak is the measured bf16 peak / 2)
    x3_flops = 3 * 2 * 2 * w.B * w.L * w.H * 2 * w.P
    tc_peak, tc_kind = load_tensor_peak()
    out["s5_fp32_tc_" + w.name] = {
        "ms": ms, "elements_per_s": w.B * w.L * w.H / ms * 1e3,
        "tensor": {"executed_tf32_flops": x3_flops, "achieved": x3_flops / ms / 1e9,
                   "peak": tc_peak / 2, "peak_kind": tc_kind + ", halved for tf32",
                   "unit": "TFLOP/s", "frac": x3_flops / ms / 1e9 / (tc_peak / 2)},
        "precision": "float32: projections as tf32 hi*hi + hi*lo + lo*hi with f32 "
                     "accumulation, scan in float32"}
    del ws
    ws = torch.empty(dlr.s5_workspace_size(w.B, w.L, w.H, w.P, "bf16"), dtype=torch.uint8,
                     device="cuda")
    ms = _time_steps(torch, lambda: dlr.s5_layer(u, *args5, prec="bf16", workspace=ws, out=y),
                     10, 3, flush)
    # two projections of 2 * (B L) * H * 2P flops each; algorithmic bytes u in + y out + the
    # parameters (lambda, log_delta, Bt, Ct, D)
    gemm_flops = 2 * 2 * w.B * w.L * w.H * 2 * w.P
    s5_bytes = 4 * (2 * w.B * w.L * w.H + 2 * w.P + w.P + 2 * 2 * w.P * w.H + w.H)
    peak_gbs, peak_kind = load_peaks()
    out["s5_bf16_tc_" + w.name] = {
        "ms": ms, "elements_per_s": w.B * w.L * w.H / ms * 1e3,
        "projection_tflops": gemm_flops / ms / 1e9,
        "hbm": {"algorithmic_bytes": s5_bytes, "achieved_gbs": s5_bytes / ms / 1e6,
                "frac": s5_bytes / ms / 1e6 / peak_gbs, "peak_kind": peak_kind},
        "precision": "bf16 projection operands (u rounded to bf16 in the kernel), V and x "
                     "bf16, scan float32, f32 accumulation"}
    # the discretisation variants on the same workload: the bilinear transform (tensor-core
    # tier) and a step that changes from step to step (float32 tier, irregular gaps)
    ms = _time_steps(torch, lambda: dlr.s5_layer_ex(u, *args5, prec="bf16", disc="bilinear",
                                                    workspace=ws, out=y), 10, 3, flush)
    out["s5_bf16_tc_bilinear_" + w.name] = {"ms": ms,
                                            "elements_per_s": w.B * w.L * w.H / ms * 1e3}
    del ws
    dt = dev(inputs.irregular_gaps(np.random.default_rng(3), w.B, w.L))
    ws = torch.empty(dlr.s5_workspace_size(w.B, w.L, w.H, w.P), dtype=torch.uint8,
                     device="cuda")
    ms = _time_steps(torch, lambda: dlr.s5_layer_tv(u, dt, *args5, workspace=ws, out=y), 5, 2,
                     flush)
    out["s5_fp32_time_varying_" + w.name] = {"ms": ms,
                                             "elements_per_s": w.B * w.L * w.H / ms * 1e3}
    return out


def cpu_baseline(w):
    """The float64 oracle (as it stands) on the full bank, threaded over (b, h) rows; the bank
    is repeated until at least one second of wall time (16+ core-seconds) has been spent."""
    import oracle
    threads = max(1, min(os.cpu_count() or 1, 64))
    par = (w.fwd.log_re, w.fwd.log_im, w.fwd.W)
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.dlr_layer(w.u, par, nthreads=threads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= 1.0 or reps >= 200:
            break
    return {"value": reps * w.B * w.H * w.L / dt, "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": f"full {WORKLOAD} bank x {reps} (sequential float64 recurrence), "
                      f"{dt:.2f} s wall"}


# --------------------------------------------------------------------------------------------
def run_reference(args):
    """Reference arm: the float64 CPU oracle, each step a bounded sample (8 (b,h) rows)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from state_space_sequence_gb300 import inputs
    cfg = dict(inputs.WORKLOADS[WORKLOAD])
    w = inputs.make_dlr(cfg["B"], cfg["H"], cfg["N"], cfg["L"], seed=cfg["seed"])
    rows = 8
    threads = max(1, min(os.cpu_count() or 1, rows))
    u = np.ascontiguousarray(w.u[:1, :rows])
    par = (w.fwd.log_re[:rows], w.fwd.log_im[:rows], w.fwd.W[:rows])
    for _ in range(args.warmup):
        oracle.dlr_layer(u, par, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.dlr_layer(u, par, nthreads=threads)
    dt = time.perf_counter() - t0
    value = rows * cfg["L"] * args.steps / dt
    sample = f"{rows} (b,h) rows of {WORKLOAD} per step (sequential float64 recurrence)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "B": cfg["B"], "H": cfg["H"],
                                        "N": cfg["N"], "L": cfg["L"]},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
