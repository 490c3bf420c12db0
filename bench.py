"""Benchmark: forward implicit-GEMM convolution throughput on GB300.

One step = one conv_fwd call (the whole hot path: dispatch, TMA operand
loads, tcgen05 MMA, epilogue, and split-K reduce when planned) over the
headline workload, the 2048-channel 3x3x3 video convolution (M = 216000
output positions, K = 2048 filters, R = 55296), with inputs resident in HBM.
Throughput is 2*M*K*R / step time.  The same JSON line carries the
end-to-end number (host -> device inputs from pinned memory, conv, output
back to the host, all timed), the roofline fraction of the conv kernel, the
fp64 CPU oracle's rate on a bounded sample (the reference arm), sampled
clocks, and secondary workloads (fp8 with and without its pack, the
>2^31-element temporal conv, the patch embedding).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 launch under torch.distributed.run; each rank runs an independent
replica (the problem has no exchange step) and rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import conv_workloads as cw  # noqa: E402

HEADLINE = "video_conv3d_bf16"
L2_FLUSH_BYTES = 256 << 20
METRIC = "conv fwd TFLOPS (2*M*N*R/time) bf16 & fp8 on 1 GB300; % of dense tensor peak"
# MI355X figure for the same shape (C=K=2048, 3x3x3, M~216k): FlyDSL PR #860, async-DMA commit
PAGE_BASELINE_TFLOPS = {"video_conv3d_bf16": 967.0}


def gemm_dims(wl: cw.Workload):
    """(M, N, R) of the GEMM view of workload wl."""
    if wl.x_layout == "ncdhw":
        N, C, D, H, W = wl.x_shape
    else:
        N, D, H, W, C = wl.x_shape
    if wl.w_layout == "kctrs":
        K, _, T, R, S = wl.w_shape
    else:
        K, T, R, S, _ = wl.w_shape
    ext = []
    for i, (n, f) in enumerate(((D, T), (H, R), (W, S))):
        ext.append((n + 2 * wl.pad[i] - wl.dil[i] * (f - 1) - 1) // wl.stride[i] + 1)
    return N * ext[0] * ext[1] * ext[2], K, C * T * R * S


def flops(wl: cw.Workload) -> float:
    M, N, R = gemm_dims(wl)
    return 2.0 * M * N * R


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_source_sha() -> str:
    """Hash of the library's sources without their // comments and blank
    lines: changes to the code (not to its comments) void measured counters."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "implicit_gemm_convolution_conv3d_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            text = open(os.path.join(csrc, f), encoding="utf-8").read()
            code = [re.sub(r"//.*$", "", line).rstrip() for line in text.split("\n")]
            h.update(f.encode() + b"\0" + "\n".join(c for c in code if c).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes of one step's conv kernel launches (a long reduction runs
    as several launches of whole waves) from the committed ncu summary, or
    None when the kernel sources changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d or d.get("kernel_sha") != kernel_source_sha():
        return None
    return d.get("dram_bytes_per_step")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not self.lines:
            return None
        sm, mx, pw, reasons = [], 0.0, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
                pw.append(float(f[3]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        hi = max(pw) if pw else 0.0
        loaded = [s for s, p in zip(sm, pw) if p >= 0.5 * hi] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": hi}


# GPU cycles of spinning after each flush, before a step's start event: the
# device stays busy while the host enqueues the step, so a step of tens of
# microseconds is timed as the device runs it (not paced by the binding's
# enqueue of its launches); outside the timed region
SLEEP_CYCLES = 200_000


class Timer:
    """Per-step CUDA-event timing on the launching stream, L2 flushed between steps."""

    def __init__(self, steps: int, flush: torch.Tensor):
        self.steps = steps
        self.flush = flush
        self.ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(steps)]

    def run(self, fn):
        stream = torch.cuda.current_stream()
        for i in range(self.steps):
            self.flush.zero_()
            torch.cuda._sleep(SLEEP_CYCLES)
            self.ev[i][0].record(stream)
            fn()
            self.ev[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in self.ev]


def physical_gpu_index(local: int) -> int:
    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    if local < len(vis) and vis[local].isdigit():
        return int(vis[local])
    return local


def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------- workloads

def reads_ncdhw(wl: cw.Workload) -> bool:
    """bf16 workloads whose channel-major activation conv_fwd_ncdhw reads in place."""
    return wl.x_layout == "ncdhw" and wl.dtype == "bf16"


def prepare(pkg, wl: cw.Workload, device):
    """Device-resident operands of workload wl in the layout its conv call takes."""
    x, w = cw.make_inputs(wl, device)
    if wl.dtype == "fp8":
        qx, sx = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(x)
        qw, sw = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(w)
        return {"x": qx, "w": qw, "sx": sx, "sw": sw, "x_bf16_ncdhw": x, "w_ncdhw": w}
    return {"x": x, "w": w, "sx": None, "sw": None}


def conv_step(pkg, wl, ops, out, ws, bias=None, act="none"):
    if reads_ncdhw(wl):
        return lambda: pkg.conv_fwd_ncdhw(ops["x"], ops["w"], wl.stride, wl.pad, wl.dil,
                                          bias=bias, out=out, workspace=ws)
    return lambda: pkg.conv_fwd(ops["x"], ops["w"], wl.stride, wl.pad, wl.dil, scale_x=ops["sx"],
                                scale_w=ops["sw"], out=out, workspace=ws, bias=bias, act=act)


def ndhwc_shape(wl: cw.Workload):
    """The activation's shape in NDHWC order."""
    if wl.x_layout == "ncdhw":
        N, C, D, H, W = wl.x_shape
        return (N, D, H, W, C)
    return tuple(wl.x_shape)


def run_workload(pkg, wl, device, steps, warmup, flush, with_e2e=True, with_bias=False,
                 act="none"):
    """with_bias: the same step through conv_fwd_bias (a per-filter fp32 bias);
    act: then an activation (conv_fwd_bias_act)."""
    ops = prepare(pkg, wl, device)
    x, w = ops["x"], ops["w"]
    ncdhw = reads_ncdhw(wl)
    if ncdhw:
        plan = pkg.conv_fwd_ncdhw_plan(tuple(x.shape), tuple(w.shape), wl.stride, wl.pad, wl.dil)
    else:
        plan = pkg.conv_fwd_plan(tuple(x.shape), tuple(w.shape), wl.stride, wl.pad, wl.dil,
                                 1 if wl.dtype == "fp8" else 0)
    od = pkg.conv_out_dims(ndhwc_shape(wl), tuple(w.shape), wl.stride, wl.pad, wl.dil)
    out = torch.empty(od, dtype=torch.bfloat16, device=device)
    ws = torch.empty(max(plan["workspace_bytes"], 16), dtype=torch.uint8, device=device)
    bias = None
    if with_bias:
        g = torch.Generator(device="cpu").manual_seed(wl.w_seed + 500)
        bias = torch.randn(w.shape[0], generator=g).float().to(device)
    step = conv_step(pkg, wl, ops, out, ws, bias, act)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if pkg.conv_get_device_status() != 0:
        raise RuntimeError("device status reports a timeout")
    times = Timer(steps, flush).run(step)
    if ncdhw:
        # the channel-major plans here run unsliced (reductions under 384 k-steps);
        # a plan whose workspace holds an NDHWC copy of x packs it first
        launches = 1 + (plan["splits"] > 1) + (plan["workspace_bytes"] >= x.numel() * 2)
    else:
        launches = pkg.conv_fwd_kernel_launches(tuple(x.shape), tuple(w.shape), wl.stride,
                                                wl.pad, wl.dil, 1 if wl.dtype == "fp8" else 0,
                                                ws.numel())
    res = {"plan": plan, "ms": times, "flop": flops(wl), "launches_per_step": launches}
    if ncdhw:
        # the alternative: the NCDHW -> NDHWC pass, then conv_fwd
        xn = torch.empty(ndhwc_shape(wl), dtype=torch.bfloat16, device=device)
        cplan = pkg.conv_fwd_plan(tuple(xn.shape), tuple(w.shape), wl.stride, wl.pad, wl.dil)
        cws = torch.empty(max(cplan["workspace_bytes"], 16), dtype=torch.uint8, device=device)

        def pack_then_conv():
            pkg.pack_ncdhw_bf16_to_ndhwc(x, out=xn)
            pkg.conv_fwd(xn, w, wl.stride, wl.pad, wl.dil, out=out, workspace=cws)
        for _ in range(warmup):
            pack_then_conv()
        res["ms_pack_then_conv"] = Timer(steps, flush).run(pack_then_conv)
        res["io_bytes"] = (x.numel() + w.numel() + out.numel()) * 2
        del xn
    if wl.dtype == "fp8":
        # with the pack of the activation (the weight pack is a one-off prep)
        xb = ops["x_bf16_ncdhw"]
        pk_ws = torch.empty(16, dtype=torch.uint8, device=device)

        def full():
            pkg.pack_ncdhw_bf16_to_ndhwc_fp8(xb, out=ops["x"], scale=ops["sx"], workspace=pk_ws)
            step()
        for _ in range(warmup):
            full()
        res["ms_with_pack"] = Timer(steps, flush).run(full)

        def pack_only():
            pkg.pack_ncdhw_bf16_to_ndhwc_fp8(xb, out=ops["x"], scale=ops["sx"], workspace=pk_ws)
        res["ms_pack"] = Timer(steps, flush).run(pack_only)
        res["pack_bytes"] = xb.numel() * 2 * 2 + xb.numel()   # amax read, pack read, fp8 write
        # the activation quantised while the conv loads it (amax pass + one
        # kernel, no pack pass), for T = 1 "same" filters
        try:
            fws = torch.empty(pkg.conv_fwd_ncdhw_fp8_workspace_size(
                tuple(xb.shape), tuple(ops["w"].shape), wl.stride, wl.pad, wl.dil),
                dtype=torch.uint8, device=device)
            fsx = torch.empty(1, dtype=torch.float32, device=device)

            def fused():
                pkg.conv_fwd_ncdhw_fp8(xb, ops["w"], wl.stride, wl.pad, wl.dil, scale_w=ops["sw"],
                                       scale_x=fsx, out=out, workspace=fws)
            for _ in range(warmup):
                fused()
            res["ms_fused"] = Timer(steps, flush).run(fused)
            del fws
        except pkg.ConvError:
            pass
    if with_e2e:
        res["e2e"] = run_e2e(pkg, wl, ops, out, ws, steps, warmup, flush)
    del ops
    return res


def run_e2e(pkg, wl, ops, out, ws, steps, warmup, flush):
    """Same conv through the public API with inputs coming from pinned host
    memory and the output going back to pinned host memory, all timed.  bf16:
    one conv_fwd_from_host call per step (the copies of each slice of output
    rows overlap the other slices' kernels).  fp8: the activation's amax
    needs all of it on the device before the pack, so the copies, the pack
    and the conv run in sequence."""
    # the host holds the activation as the user has it (bf16 NCDHW for the fp8
    # workload, which is packed on the device every step; channel-major x for
    # conv_fwd_ncdhw) and the prepared weight
    dx = ops["x_bf16_ncdhw"] if wl.dtype == "fp8" else ops["x"]
    hx = torch.empty(dx.shape, dtype=dx.dtype, pin_memory=True)
    hx.copy_(dx)
    hw = torch.empty(ops["w"].shape, dtype=ops["w"].dtype, pin_memory=True)
    hw.copy_(ops["w"])
    pk_ws = torch.empty(16, dtype=torch.uint8, device=out.device)
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

    def step():
        if reads_ncdhw(wl):
            dx.copy_(hx, non_blocking=True)
            ops["w"].copy_(hw, non_blocking=True)
            pkg.conv_fwd_ncdhw(dx, ops["w"], wl.stride, wl.pad, wl.dil, out=out, workspace=ws)
            hout.copy_(out, non_blocking=True)
            return
        if wl.dtype != "fp8":
            pkg.conv_fwd_from_host(hx, hw, wl.stride, wl.pad, wl.dil, out_host=hout,
                                   x_dev=ops["x"], w_dev=ops["w"], out_dev=out, workspace=ws)
            return
        dx.copy_(hx, non_blocking=True)
        ops["w"].copy_(hw, non_blocking=True)
        pkg.pack_ncdhw_bf16_to_ndhwc_fp8(dx, out=ops["x"], scale=ops["sx"], workspace=pk_ws)
        pkg.conv_fwd(ops["x"], ops["w"], wl.stride, wl.pad, wl.dil, scale_x=ops["sx"],
                     scale_w=ops["sw"], out=out, workspace=ws)
        hout.copy_(out, non_blocking=True)

    for _ in range(warmup):
        step()
    times = Timer(steps, flush).run(step)
    h2d = hx.numel() * hx.element_size() + hw.numel() * hw.element_size()
    d2h = hout.numel() * hout.element_size()
    return {"ms": times, "h2d": h2d, "d2h": d2h, "link": link_bandwidth(hx, dx, hout, out)}


def link_bandwidth(h_in, d_in, h_out, d_out):
    """Host<->device copy bandwidth of this machine (GB/s): the best of three
    plain copies each way between the e2e leg's own pinned buffers, alone on
    the stream -- the bound the end-to-end number cannot beat."""
    res = {}
    for name, dst, src in (("h2d_gbs", d_in, h_in), ("d2h_gbs", h_out, d_out)):
        dst.copy_(src, non_blocking=True)
        best = 0.0
        for _ in range(3):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record()
            dst.copy_(src, non_blocking=True)
            b.record()
            torch.cuda.synchronize()
            best = max(best, src.numel() * src.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9)
        res[name] = best
    return res


# ---------------------------------------------------------------- CPU oracle arm

def replica_throughput(world: int, flop_per_step: float, ms_max: float) -> float:
    """Whole-job TFLOPS of `world` independent replicas, each doing
    flop_per_step per step, timed by the slowest rank's mean step (ms)."""
    return world * flop_per_step / (ms_max * 1e-3) / 1e12


def cpu_oracle_rate(wl: cw.Workload, x_host, w_host, target_s: float = 10.0):
    """fp64 oracle TFLOPS on a bounded sample of output elements, sized for
    about target_s seconds of work on all host cores."""
    import oracle
    M, N, R = gemm_dims(wl)
    total = M * N
    rng = np.random.default_rng(wl.sample_seed)
    probe = rng.integers(0, total, size=256)
    t0 = time.perf_counter()
    lay = "ncdhw" if wl.x_layout == "ncdhw" else "ndhwc"
    oracle.conv3d_points(x_host, w_host, probe, wl.stride, wl.pad, wl.dil, x_layout=lay)
    per = (time.perf_counter() - t0) / probe.size
    n = int(min(max(256, target_s / max(per, 1e-9)), 5_000_000))
    idx = rng.integers(0, total, size=n)
    t0 = time.perf_counter()
    oracle.conv3d_points(x_host, w_host, idx, wl.stride, wl.pad, wl.dil, x_layout=lay)
    dt = time.perf_counter() - t0
    return {"value": r4(2.0 * n * R / dt / 1e12), "unit": "TFLOPS", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{n} output elements of {wl.name} (each a {R}-term fp64 dot product), "
                      f"{dt:.1f} s"}


def host_inputs(wl: cw.Workload):
    """The workload's operands as the host bytes the oracle reads (generated
    on the CPU with the same seeds and recipe): x as stored (NDHWC, or NCDHW),
    w as KTRSC (values of the bf16 weight before any fp8 pack)."""
    x, w = cw.make_inputs(wl, "cpu")
    if wl.w_layout == "kctrs":
        w = w.permute(0, 2, 3, 4, 1).contiguous()
    xb = x.view(torch.int16).numpy().view(np.uint16)
    wb = w.view(torch.int16).numpy().view(np.uint16)
    return xb, wb


def reference_arm(args):
    dist, rank, world, _ = dist_setup(args)
    if rank != 0:
        return
    wl = cw.BY_NAME[args.workload]
    if wl.dtype == "fp8":
        raise SystemExit("the reference arm times bf16 workloads")
    xb, wb = host_inputs(wl)
    per_step_s = args.ref_seconds if args.ref_seconds > 0 else \
        max(1.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_oracle_rate(wl, xb, wb, target_s=min(per_step_s, 5.0))
    vals, secs = [], []
    last = None
    for _ in range(args.steps):
        t0 = time.perf_counter()
        last = cpu_oracle_rate(wl, xb, wb, target_s=per_step_s)
        secs.append(time.perf_counter() - t0)
        vals.append(last["value"])
    value = statistics.median(vals)
    flop = flops(wl)
    # a step is one bounded sample of the workload's output elements:
    # ms_per_step is the measured wall time of such a step; the time the
    # oracle would take for the whole workload is extrapolated from the rate
    line = {"impl": "reference", "metric": METRIC, "value": r4(value), "unit": "TFLOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": r4(statistics.mean(secs) * 1e3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl),
            "ms_full_workload_extrapolated": r4(flop / (value * 1e12) * 1e3),
            "cpu_baseline": dict(last, value=r4(value)),
            "e2e": {"value": r4(value), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line, separators=(",", ":")))


def workload_config(wl):
    M, N, R = gemm_dims(wl)
    return {"workload": wl.name, "x_shape": list(wl.x_shape), "x_layout": wl.x_layout,
            "w_shape": list(wl.w_shape), "w_layout": wl.w_layout, "stride": list(wl.stride),
            "pad": list(wl.pad), "dil": list(wl.dil), "M": M, "N": N, "R": R,
            "flop_per_step": flops(wl),
            "l2": f"{L2_FLUSH_BYTES >> 20} MB buffer written between timed steps, then "
                  f"{SLEEP_CYCLES} GPU cycles of sleep before each step's start event"}


def run_backward(pkg, wl, device, steps, warmup, flush):
    """Point-output backward passes of workload wl (the patch embedding): one
    conv_bwd_data_point and one conv_bwd_weight_point call per step, each
    with its operand transposes, GEMM and (for dw) split-K reduction."""
    x, w = cw.make_inputs(wl, device)
    N, K = x.shape[0], w.shape[0]
    g = torch.Generator(device=device).manual_seed(wl.sample_seed + 1)
    dy = (torch.randn((N, 1, 1, 1, K), generator=g, device=device) / math.sqrt(K)).to(torch.bfloat16)
    dx, dw = torch.empty_like(x), torch.empty_like(w)
    res = {}
    for which, name in ((0, "dgrad"), (1, "wgrad")):
        need = pkg.conv_bwd_point_workspace_bytes(tuple(x.shape), tuple(w.shape), wl.stride,
                                                  wl.pad, wl.dil, which)
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        if which == 0:
            fn = lambda: pkg.conv_bwd_data_point(dy, w, tuple(x.shape), wl.stride, wl.pad,  # noqa: E731
                                                 wl.dil, dx=dx, workspace=ws)
        else:
            fn = lambda: pkg.conv_bwd_weight_point(x, dy, tuple(w.shape), wl.stride, wl.pad,  # noqa: E731
                                                   wl.dil, dw=dw, workspace=ws)
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        if pkg.conv_get_device_status() != 0:
            raise RuntimeError("device status reports a timeout")
        res[name] = Timer(steps, flush).run(fn)
    return res


# MI355X figures for the patch embedding's backward passes (MIOpen PR #10912,
# test plan and review thread): context, not a target on this hardware
PAGE_BACKWARD_MS = {"dgrad": 0.028, "wgrad": 0.040}
# FlyDSL PR #860, 1x1x1 commit (MI355X): the pointwise conv of a channel-major
# activation through the NCDHW -> NDHWC transpose and the im2col kernel, and
# through torch.matmul on the channel-major tensor
PAGE_NCDHW_MS = {"pointwise_1x1x1_bf16_ncdhw": {"transpose_then_conv": 8.7,
                                                "matmul_on_ncdhw": 3.4}}


# ---------------------------------------------------------------- main arm

def main_arm(args):
    dist, rank, world, local = dist_setup(args)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import implicit_gemm_convolution_conv3d_gb300 as pkg
    pkg.load_library()
    peaks = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    wl = cw.BY_NAME[args.workload]

    barrier(dist)
    with ClockSampler(physical_gpu_index(local)) as clk:
        res = run_workload(pkg, wl, device, args.steps, args.warmup, flush)
    barrier(dist)
    ms = statistics.mean(res["ms"])
    ms_max = max_over_ranks(dist, ms, device)
    e2e_ms = max_over_ranks(dist, statistics.mean(res["e2e"]["ms"]), device)
    value = replica_throughput(world, res["flop"], ms_max)
    e2e_value = replica_throughput(world, res["flop"], e2e_ms)

    secondary = {}
    if not args.no_secondary:
        names = [n for n in ("fp8_conv3d_1x3x3", "temporal_3x1x1_bf16_big", "patch_embed_bf16",
                             "tiny_conv3d_bf16", "vit_patch16_bf16", "vit_patch14_bf16",
                             "temporal_3x1x1_bf16_ncdhw", "pointwise_1x1x1_bf16_ncdhw")
                 if n != wl.name]
        # the bias epilogue on the headline and on the epilogue-heavy patch embedding
        names += [wl.name + "+bias", "patch_embed_bf16+bias", wl.name + "+bias+gelu"]
        for name in names:
            try:
                r = run_workload(pkg, cw.BY_NAME[name.split("+")[0]], device, args.steps,
                                 args.warmup, flush, with_e2e=False,
                                 with_bias="+bias" in name,
                                 act="gelu" if name.endswith("+gelu") else "none")
                secondary[name] = r
            except Exception as e:  # a secondary workload never hides the headline line
                secondary[name] = {"error": f"{type(e).__name__}: {e}"}
            torch.cuda.empty_cache()
        # backward data / weights of the patch embedding
        try:
            pe = cw.BY_NAME["patch_embed_bf16"]
            rb = run_backward(pkg, pe, device, args.steps, args.warmup, flush)
            for name, t in rb.items():
                secondary["patch_embed_bf16_" + name] = {"ms": t, "flop": flops(pe)}
        except Exception as e:
            secondary["patch_embed_bf16_backward"] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()

    if rank != 0:
        return
    peak = peaks["bf16_tflops"] if wl.dtype == "bf16" else 2.0 * peaks["bf16_tflops"]
    achieved = res["flop"] / (ms * 1e-3) / 1e12
    traffic = measured_traffic(wl.name)
    roof = {"bound": "tensor", "achieved": r4(achieved), "peak": peak, "unit": "TFLOP/s",
            "frac": r4(achieved / peak), "traffic": traffic,
            "per": f"one conv_fwd step ({res['launches_per_step']} kernel launches)",
            "peak_source": f"{peaks['source']} bf16 burst (cuBLAS)",
            "kernel": "conv_igemm_kernel (tcgen05, TMA im2col)"}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        xb, wb = host_inputs(wl)
        cpu = cpu_oracle_rate(wl, xb, wb)
    base = PAGE_BASELINE_TFLOPS.get(wl.name)
    line = {"metric": METRIC, "value": r4(value), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r4(ms_max),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": r4(value / base) if base else None,
            "dtype": wl.dtype, "data": "synthetic",
            "config": workload_config(wl),
            "e2e": {"value": r4(e2e_value), "unit": "TFLOPS",
                    "h2d_bytes_per_step": res["e2e"]["h2d"],
                    "d2h_bytes_per_step": res["e2e"]["d2h"], "ms_per_step": r4(e2e_ms),
                    # the host link is shared: single steps can take up to ~2x
                    "ms_median": r4(statistics.median(res["e2e"]["ms"])),
                    "ms_min_max": [r4(min(res["e2e"]["ms"])), r4(max(res["e2e"]["ms"]))],
                    "link_gbs": {k: r4(v) for k, v in res["e2e"]["link"].items()}},
            "gpu_launches": res["launches_per_step"] * args.steps,
            "roofline": roof, "cpu_baseline": cpu, "clocks": clk.summary(),
            "note": "vs_baseline: over the MI355X figure for this shape (967 TFLOPS, "
                    "FlyDSL PR #860), context only; workloads: [TFLOPS, mean ms]",
            "workloads": compact_workloads(secondary),
            "roofline_by_workload": workload_rooflines(secondary, peaks)}
    print(json.dumps(line, separators=(",", ":")))


def r4(v):
    """v rounded to 4 significant digits (the JSON line stays short)."""
    if v is None or not isinstance(v, float) or v == 0.0 or not math.isfinite(v):
        return v
    return float(f"{v:.4g}")


def compact_workloads(secondary):
    """{name: [TFLOPS, mean ms]} of the secondary workloads (errors as text)."""
    out = {}
    for name, r in secondary.items():
        if "error" in r:
            out[name] = r["error"][:80]
            continue
        m = statistics.mean(r["ms"])
        ent = [r4(r["flop"] / (m * 1e-3) / 1e12), r4(m)]
        if "ms_pack_then_conv" in r:   # channel-major: the pack + conv_fwd alternative
            ent.append(r4(statistics.mean(r["ms_pack_then_conv"])))
        out[name] = ent
    return out


def workload_rooflines(secondary, peaks):
    """Roofline entries of the fp8 conv (and its amax + pack), the temporal
    conv and the patch embedding: achieved over the measured peak of the
    kernel's own dtype (e4m3: 2x the bf16 burst, the nominal ratio), and the
    pack's achieved bytes over the measured copy bandwidth."""
    out = {}
    bf16 = peaks["bf16_tflops"]
    for name, peak in (("fp8_conv3d_1x3x3", 2.0 * bf16), ("temporal_3x1x1_bf16_big", bf16),
                       ("patch_embed_bf16", bf16)):
        r = secondary.get(name)
        if not r or "error" in r:
            continue
        m = statistics.mean(r["ms"])
        a = r["flop"] / (m * 1e-3) / 1e12
        ent = {"bound": "tensor", "achieved": r4(a), "peak": r4(peak), "frac": r4(a / peak),
               "ms": r4(m), "ms_median": r4(statistics.median(r["ms"]))}
        if "ms_with_pack" in r:
            mp = statistics.mean(r["ms_with_pack"])
            pk = statistics.mean(r["ms_pack"])
            gbs = r["pack_bytes"] / (pk * 1e-3) / 1e9
            if "ms_fused" in r:   # quantised while loaded: amax pass + fused conv
                mf = statistics.mean(r["ms_fused"])
                ent["fused_ncdhw_ms"] = r4(mf)
                ent["fused_ncdhw_tflops"] = r4(r["flop"] / (mf * 1e-3) / 1e12)
            ent.update({"with_pack_tflops": r4(r["flop"] / (mp * 1e-3) / 1e12),
                        "with_pack_ms": r4(mp),
                        "pack": {"bound": "hbm", "achieved_gbs": r4(gbs), "ms": r4(pk),
                                 "peak_gbs": peaks["hbm_gbs"],
                                 "frac": r4(gbs / peaks["hbm_gbs"])}})
        out[name] = ent
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(cw.BY_NAME))
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=0.0,
                    help="reference arm: seconds of oracle work per step (0: auto)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    else:
        main_arm(args)


if __name__ == "__main__":
    main()
