"""Host-side logic of bench.py (no GPU): the FLOP convention pinned to the
pages' own ms -> TFLOPS pairs, and the multi-rank (replica) aggregation
exercised with two gloo ranks on CPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import conv_workloads as cw  # noqa: E402


def test_flop_convention_reproduces_the_pages_printed_tflops():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "flop_convention.json")))
    wl = cw.BY_NAME[g["workload"]]
    assert bench.gemm_dims(wl) == (1728000, 1024, 9216)
    for pt in g["printed"]:
        tf = bench.flops(wl) / (pt["ms"] * 1e-3) / 1e12
        assert abs(tf - pt["tflops"]) / pt["tflops"] < g["tolerance_rel"], (pt, tf)


def test_gemm_dims_of_the_workloads():
    assert bench.gemm_dims(cw.BY_NAME["tiny_conv3d_bf16"]) == (256, 32, 432)
    assert bench.gemm_dims(cw.BY_NAME["patch_embed_bf16"]) == (9500, 1280, 588)
    assert bench.gemm_dims(cw.BY_NAME["video_conv3d_bf16"]) == (216000, 2048, 55296)
    assert bench.gemm_dims(cw.BY_NAME["temporal_3x1x1_bf16_big"]) == (3456000, 640, 1920)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    local_ms = [4.0, 5.0][rank]                 # rank 1 is the slow one
    ms_max = bench.max_over_ranks(dist, local_ms, torch.device("cpu"))
    bench.barrier(dist)
    out_q.put((rank, ms_max, bench.replica_throughput(world, 2e12, ms_max)))
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms_max, tflops in res:
        assert ms_max == 5.0
        assert tflops == pytest.approx(2 * 2e12 / 5e-3 / 1e12)


def test_reference_arm_prints_only_on_rank_zero():
    port = str(_free_port())
    env0 = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0", MASTER_ADDR="127.0.0.1",
                MASTER_PORT=port, CUDA_VISIBLE_DEVICES="")
    env1 = dict(env0, RANK="1", LOCAL_RANK="1")
    args = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
            "--steps", "1", "--warmup", "3", "--workload", "tiny_conv3d_bf16",
            "--ref-seconds", "0.2"]
    p0 = subprocess.Popen(args, env=env0, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                          text=True)
    p1 = subprocess.Popen(args, env=env1, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                          text=True)
    out0, err0 = p0.communicate(timeout=300)
    out1, err1 = p1.communicate(timeout=300)
    assert p0.returncode == 0, err0
    assert p1.returncode == 0, err1
    assert out1.strip() == ""
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOPS" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
