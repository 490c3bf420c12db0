"""Measured tile sweep for conv_fwd: fills csrc/tile_table.h.

For each workload, every candidate (BN, BK, stages, raster group, split-K,
CTA pair, row sub-tiles) is forced through CONV3D_FORCE_TILE / CONV3D_PAIR /
CONV3D_MSUB, timed with CUDA events (L2 flushed between runs), and the
fastest legal one is printed as a tile-table row.
Candidates whose plan is rejected are skipped.  Run on the GPU:

    python -m implicit_gemm_convolution_conv3d_gb300.sweep_tiles [--workloads a,b] [--quick]
"""
from __future__ import annotations

import argparse
import itertools
import json
import os
import statistics
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import conv_workloads as cw  # noqa: E402
import implicit_gemm_convolution_conv3d_gb300 as pkg  # noqa: E402

CLASS_CODE = {"generic": 0, "temporal": 1, "point_gemm": 2}


def candidates(quick: bool, K: int, k_row_bytes: int, default_bn: int):
    bns = [bn for bn in (256, 224, 192, 160, 128, 96, 64, 32) if bn <= max(32, ((K + 31) // 32) * 32)]
    bks = [bk for bk in (256, 128, 64, 32) if bk <= max(32, k_row_bytes) or (bk == 256 and k_row_bytes > 128)]
    groups = [1, 2, 4, 8, 16, 32]
    if quick:   # default tile width, the two widest k-steps, small raster groups
        bns, bks, groups = [default_bn], bks[:2], [1, 2, 4, 8]
    for bn, bk, grp, pair, msub in itertools.product(bns, bks, groups, (0, 1), (1, 2)):
        yield bn, bk, 0, grp, 1, pair, msub


def time_case(x, w, wl, scale_x, scale_w, spec, flush, reps, pair, msub):
    os.environ["CONV3D_FORCE_TILE"] = spec
    os.environ["CONV3D_PAIR"] = str(pair)
    os.environ["CONV3D_MSUB"] = str(msub)
    try:
        plan = pkg.conv_fwd_plan(tuple(x.shape), tuple(w.shape), wl.stride, wl.pad, wl.dil,
                                 1 if x.dtype == torch.float8_e4m3fn else 0)
    except pkg.ConvError:
        return None, None
    out = torch.empty(pkg.conv_out_dims(tuple(x.shape), tuple(w.shape), wl.stride, wl.pad,
                                        wl.dil), dtype=torch.bfloat16, device=x.device)
    ws = torch.empty(max(16, plan["workspace_bytes"]), dtype=torch.uint8, device=x.device)
    fn = lambda: pkg.conv_fwd(x, w, wl.stride, wl.pad, wl.dil, scale_x=scale_x, scale_w=scale_w,  # noqa: E731
                              out=out, workspace=ws)
    fn()
    torch.cuda.synchronize()
    if pkg.conv_get_device_status() != 0:
        return None, plan
    ts = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts), plan


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workloads", default="video_conv3d_bf16,fp8_conv3d_1x3x3,"
                                           "temporal_3x1x1_bf16_big,patch_embed_bf16")
    ap.add_argument("--quick", action="store_true")
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--json", default="")
    args = ap.parse_args()
    pkg.load_library()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    rows, report = [], {}
    for name in args.workloads.split(","):
        wl = cw.BY_NAME[name]
        x, w = cw.make_inputs(wl, "cuda")
        sx = sw = None
        if wl.dtype == "fp8":
            x, sx = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(x)
            w, sw = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(w)
        elt = 1 if wl.dtype == "fp8" else 2
        K, T, R, S, C = w.shape
        base = pkg.conv_fwd_plan(tuple(x.shape), tuple(w.shape), wl.stride, wl.pad, wl.dil,
                                 1 if wl.dtype == "fp8" else 0)
        row_bytes = C * elt if base["class"] != "point_gemm" else T * R * S * C * elt
        results = []
        for bn, bk, st, grp, spl, pair, msub in candidates(args.quick, K, row_bytes,
                                                           base["tile_n"]):
            spec = f"{bn},{bk},{st},{grp},{spl}"
            ms, plan = time_case(x, w, wl, sx, sw, spec, flush, args.reps, pair, msub)
            if ms is None:
                continue
            tf = 2.0 * cw_flops(wl) / (ms * 1e-3) / 1e12
            results.append((ms, spec, plan, pair, msub))
            print(f"{name:26s} {spec:18s} pair={pair} msub={msub} {ms:9.4f} ms {tf:8.1f} TFLOPS "
                  f"stages={plan['stages']}", flush=True)
        for k in ("CONV3D_FORCE_TILE", "CONV3D_PAIR", "CONV3D_MSUB"):
            os.environ.pop(k, None)
        results.sort(key=lambda r: r[0])
        best_ms, best_spec, best_plan, best_pair, best_msub = results[0]
        bn, bk, _, grp, spl = (int(v) for v in best_spec.split(","))
        M = best_plan_rows(wl)
        rows.append(f"    {{{1 if wl.dtype == 'fp8' else 0}, {CLASS_CODE[best_plan['class']]}, "
                    f"{C}, {K}, {T * R * S}, {M}, {M}, {bn}, {bk}, {best_plan['stages']}, {grp}, "
                    f"{spl}, {best_pair}, {best_msub}}},   // {name}: {best_ms:.3f} ms")
        report[name] = {"best_ms": best_ms, "best": best_spec, "pair": best_pair,
                        "msub": best_msub, "all": [(r[0], r[1], r[3], r[4]) for r in results]}
        del x, w
        torch.cuda.empty_cache()
    print("\n".join(rows))
    if args.json:
        with open(args.json, "w") as f:
            json.dump(report, f, indent=1)


def cw_flops(wl):
    M = best_plan_rows(wl)
    if wl.w_layout == "kctrs":
        K, C, T, R, S = wl.w_shape
    else:
        K, T, R, S, C = wl.w_shape
    return M * K * C * T * R * S


def best_plan_rows(wl):
    if wl.x_layout == "ncdhw":
        N, C, D, H, W = wl.x_shape
    else:
        N, D, H, W, C = wl.x_shape
    if wl.w_layout == "kctrs":
        K, _, T, R, S = wl.w_shape
    else:
        K, T, R, S, _ = wl.w_shape
    od = [(n + 2 * p - d * (f - 1) - 1) // s + 1
          for n, f, s, p, d in zip((D, H, W), (T, R, S), wl.stride, wl.pad, wl.dil)]
    return N * od[0] * od[1] * od[2]


if __name__ == "__main__":
    main()
