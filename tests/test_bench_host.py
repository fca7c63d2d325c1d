"""Host-side checks of bench.py: the multi-rank timing reduction (two gloo ranks on
CPU), the reference arm's JSON line, and the algorithmic byte/flop accounting."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # every rank measured a different time; the job time is the slowest rank's
    v = bench.max_over_ranks(1.5 + rank, world, device=None)
    bench.barrier(world)
    out[rank] = v
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_algorithmic_bytes_closed_form_c1():
    c = W.c1()
    a = bench.algorithmic(c)
    B, N, Hq, Hkv, D, P = 1, 5, 2, 2, 64, 16
    kv = P * Hkv * D * 2 * 2
    assert a["tree_attn_fwd"]["bytes"] >= kv + 2 * B * N * Hq * D * 2
    # |A(i)| for the demo tree: 1, 2, 2, 3, 3 -> 11 tree keys seen in total
    assert a["tree_attn_fwd"]["flops"] == 4 * D * Hq * (N * P + 11)
    assert a["tree_verify_greedy"]["bytes"] >= B * N * 1000 * 4


def test_reference_arm_json_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "c1",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "cpu_baseline", "e2e", "config"):
        assert k in line
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["value"] > 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "c1",
                        "--steps", "1"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_code_digest_ignores_comments_but_not_code(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("// header\n__global__ void k(int* x) {\n  x[0] = 1;  // store\n}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.code_digest(["k.cu"])
    src.write_text("// a different header\n\n__global__ void k(int* x) {\n  x[0] = 1;   // other words\n}\n")
    assert bench.code_digest(["k.cu"]) == d0
    src.write_text("// header\n__global__ void k(int* x) {\n  x[0] = 2;  // store\n}\n")
    assert bench.code_digest(["k.cu"]) != d0



def test_traffic_record_of_an_unknown_workload_is_none():
    assert bench.recorded_traffic("tree_attn_fwd", "no-such-workload") is None
