"""Measured tile sweep for conv_fwd: fills csrc/tile_table.h.

For each workload, every candidate (BN, BK, stages, raster group, split-K,
CTA pair, row sub-tiles) is forced through the library's plan overrides
(conv_set_overrides) and timed with CUDA events (L2 flushed between runs).
Candidates whose plan is rejected are skipped.  The leaders of that pass
(--ab N) are then timed again in an interleaved A/B: round by round each
leader runs once, so that the power-capped clock drifts alike for all of
them, and the median over the rounds decides.  The winner is printed as a
tile-table row; --md writes the candidates, their medians and the protocol
as a markdown summary.  Run on the GPU:

    python -m implicit_gemm_convolution_conv3d_gb300.sweep_tiles [--workloads a,b] [--quick]
        [--ab 4 --rounds 18] [--json out.json] [--md out.md]
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

CLASS_CODE = {"generic": 0, "temporal": 1, "point_gemm": 2, "patch_gemm": 3}


def candidates(quick: bool, K: int, k_row_bytes: int, default_bn: int):
    bns = [bn for bn in (256, 224, 192, 160, 128, 96, 64, 32) if bn <= max(32, ((K + 31) // 32) * 32)]
    bks = [bk for bk in (256, 128, 64, 32) if bk <= max(32, k_row_bytes) or (bk == 256 and k_row_bytes > 128)]
    groups = [1, 2, 4, 8, 16, 32]
    if quick:   # default tile width, the two widest k-steps, small raster groups
        bns, bks, groups = [default_bn], bks[:2], [1, 2, 4, 8]
    for bn, bk, grp, pair, msub in itertools.product(bns, bks, groups, (0, 1), (1, 2)):
        yield bn, bk, 0, grp, 1, pair, msub


def make_runner(x, w, wl, scale_x, scale_w, spec, pair, msub):
    """(plan, fn) of one forced candidate, or (None, None) if its plan is
    rejected; fn runs one conv_fwd under the candidate's overrides."""
    fp8 = 1 if x.dtype == torch.float8_e4m3fn else 0
    try:
        with pkg.overrides(tile=spec, pair=pair, msub=msub):
            plan = pkg.conv_fwd_plan(tuple(x.shape), tuple(w.shape), wl.stride, wl.pad,
                                     wl.dil, fp8)
    except pkg.ConvError:
        return None, None
    out = torch.empty(pkg.conv_out_dims(tuple(x.shape), tuple(w.shape), wl.stride, wl.pad,
                                        wl.dil), dtype=torch.bfloat16, device=x.device)
    ws = torch.empty(max(16, plan["workspace_bytes"]), dtype=torch.uint8, device=x.device)

    def fn():
        with pkg.overrides(tile=spec, pair=pair, msub=msub):
            pkg.conv_fwd(x, w, wl.stride, wl.pad, wl.dil, scale_x=scale_x, scale_w=scale_w,
                         out=out, workspace=ws)
    return plan, fn


def time_once(fn, flush):
    flush.zero_()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def time_case(x, w, wl, scale_x, scale_w, spec, flush, reps, pair, msub):
    plan, fn = make_runner(x, w, wl, scale_x, scale_w, spec, pair, msub)
    if plan is None:
        return None, None
    fn()
    torch.cuda.synchronize()
    if pkg.conv_get_device_status() != 0:
        return None, plan
    return statistics.median(time_once(fn, flush) for _ in range(reps)), plan


def interleaved_ab(x, w, wl, scale_x, scale_w, leaders, flush, rounds):
    """Medians of `rounds` interleaved runs of each leader (spec, pair, msub)."""
    fns = [make_runner(x, w, wl, scale_x, scale_w, spec, pair, msub)[1]
           for spec, pair, msub in leaders]
    for fn in fns:
        fn()
    torch.cuda.synchronize()
    times = [[] for _ in fns]
    for _ in range(rounds):
        for i, fn in enumerate(fns):
            times[i].append(time_once(fn, flush))
    return [statistics.median(t) for t in times]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workloads", default="video_conv3d_bf16,fp8_conv3d_1x3x3,"
                                           "temporal_3x1x1_bf16_big,patch_embed_bf16")
    ap.add_argument("--quick", action="store_true")
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--json", default="")
    ap.add_argument("--ab", type=int, default=0, help="leaders re-timed in an interleaved A/B")
    ap.add_argument("--rounds", type=int, default=18)
    ap.add_argument("--md", default="")
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
        sweep_rows = []
        for bn, bk, st, grp, spl, pair, msub in candidates(args.quick, K, row_bytes,
                                                           base["tile_n"]):
            spec = f"{bn},{bk},{st},{grp},{spl}"
            ms, plan = time_case(x, w, wl, sx, sw, spec, flush, args.reps, pair, msub)
            if ms is None:
                continue
            tf = 2.0 * cw_flops(wl) / (ms * 1e-3) / 1e12
            results.append((ms, spec, plan, pair, msub))
            sweep_rows.append((ms, spec, pair, msub, plan["stages"]))
            print(f"{name:26s} {spec:18s} pair={pair} msub={msub} {ms:9.4f} ms {tf:8.1f} TFLOPS "
                  f"stages={plan['stages']}", flush=True)
        results.sort(key=lambda r: r[0])
        ab = []
        if args.ab > 1:
            leaders = results[:args.ab]
            med = interleaved_ab(x, w, wl, sx, sw, [(r[1], r[3], r[4]) for r in leaders], flush,
                                 args.rounds)
            # the A/B medians replace the sweep pass's times of the leaders
            ab = sorted(zip(med, leaders), key=lambda t: t[0])
            results = [(m,) + tuple(r[1:]) for m, r in ab]
        best_ms, best_spec, best_plan, best_pair, best_msub = results[0]
        bn, bk, _, grp, spl = (int(v) for v in best_spec.split(","))
        M = best_plan_rows(wl)
        rows.append(f"    {{{1 if wl.dtype == 'fp8' else 0}, {CLASS_CODE[best_plan['class']]}, "
                    f"{C}, {K}, {T * R * S}, {M}, {M}, {bn}, {bk}, {best_plan['stages']}, {grp}, "
                    f"{spl}, {best_pair}, {best_msub}}},   // {name}: {best_ms:.3f} ms")
        report[name] = {"best_ms": best_ms, "best": best_spec, "pair": best_pair,
                        "msub": best_msub, "stages": best_plan["stages"],
                        "sweep": sweep_rows, "ab": [(m, r[1], r[3], r[4]) for m, r in ab]}
        del x, w
        torch.cuda.empty_cache()
    print("\n".join(rows))
    if args.json:
        with open(args.json, "w") as f:
            json.dump(report, f, indent=1)
    if args.md:
        write_markdown(args, report, rows)


def write_markdown(args, report, rows):
    """The sweep as a short markdown summary: per workload, the fastest ten
    candidates of the sweep pass, the interleaved A/B medians, the winner."""
    lines = ["# Tile sweep (sweep_tiles.py)", "",
             f"Command: `python -m implicit_gemm_convolution_conv3d_gb300.sweep_tiles "
             f"--workloads {args.workloads}{' --quick' if args.quick else ''} --reps {args.reps}"
             f"{f' --ab {args.ab} --rounds {args.rounds}' if args.ab else ''} --md <file>`", "",
             f"Protocol: each candidate forced through conv_set_overrides, run once, then "
             f"timed {args.reps} times with CUDA events, a 256 MB buffer written before each "
             f"run (L2 flushed), median kept."
             + (f" The {args.ab} fastest then run round-robin for {args.rounds} rounds "
                f"(one run each per round, same flush), medians compared: under the power "
                f"cap the clock drifts, and interleaving exposes every candidate to the same "
                f"drift." if args.ab else ""), ""]
    for name, r in report.items():
        lines += [f"## {name}", "", "sweep pass (fastest 10 of %d legal candidates):" %
                  len(r["sweep"]), "", "| BN,BK,stages,group,splits | pair | msub | stages | "
                  "median ms |", "|---|---|---|---|---|"]
        for ms, spec, pair, msub, st in sorted(r["sweep"])[:10]:
            lines.append(f"| {spec} | {pair} | {msub} | {st} | {ms:.4f} |")
        if r["ab"]:
            lines += ["", f"interleaved A/B, medians of {args.rounds} rounds:", "",
                      "| BN,BK,stages,group,splits | pair | msub | median ms |",
                      "|---|---|---|---|"]
            for ms, spec, pair, msub in r["ab"]:
                lines.append(f"| {spec} | {pair} | {msub} | {ms:.4f} |")
        lines += ["", f"winner: {r['best']} pair={r['pair']} msub={r['msub']} "
                  f"stages={r['stages']}: {r['best_ms']:.4f} ms", ""]
    lines += ["Tile-table rows printed by the run:", "", "```"] + rows + ["```", ""]
    with open(args.md, "w") as f:
        f.write("\n".join(lines))


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
