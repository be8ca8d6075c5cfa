"""Multi-GPU is replicas only: every rank runs the whole step on its own GPU,
no data moves between ranks, and the host aggregates the timings (barrier,
max over ranks, whole-job throughput = units of all ranks / slowest time).
These tests run that host logic with two gloo ranks on the CPU."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import argparse

    import torch.distributed as dist

    import bench as b

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w = b.rank_env()
        # rank-dependent timings: each rank must see the elementwise max
        mx = b.rank_max(dist, [1.0 + rank, 10.0 - rank, 5.0 * (rank + 1)])
        rate = b.job_rate(100.0, 4, w, mx[0])
        # the reference arm: only rank 0 works, the others return at once
        args = argparse.Namespace(warmup=3, steps=1)
        ref = b.run_reference(args, r, w) if r != 0 else "skipped"
        dist.barrier()
        q.put((rank, r, w, mx, rate, ref))
    finally:
        dist.destroy_process_group()


def test_rank_aggregation_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for rank, r, w, mx, rate, ref in out:
        assert (r, w) == (rank, 2)
        assert mx == [2.0, 10.0, 10.0]                 # elementwise max over both ranks
        assert rate == pytest.approx(2 * 100.0 * 4 / 2e-3)
    assert out[1][5] is None                           # rank 1 did no reference work


def test_single_process_helpers():
    assert bench.rank_max(None, [3, 1.5]) == [3.0, 1.5]
    assert bench.job_rate(10.0, 5, 1, 50.0) == pytest.approx(1000.0)
    # weak scaling: N replicas doing the same work in the same time give N times the rate
    assert bench.job_rate(10.0, 5, 4, 50.0) == pytest.approx(4 * bench.job_rate(10.0, 5, 1, 50.0))


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched as the multi-GPU run is: rank 0
    alone prints one JSON line; the other rank exits 0 without output."""
    port = _free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["unit"] == d["unit"]


def test_profile_guard_hashes_code_not_comments(tmp_path):
    """The bench reports profiled DRAM traffic only while the kernel's code
    matches the capture: a comment or blank-line edit keeps the hash, a code
    edit changes it."""
    base = "int f(int x) {  // doubles x\n  return 2 * x;\n}\n"
    a, b, c = tmp_path / "a.cu", tmp_path / "b.cu", tmp_path / "c.cu"
    a.write_text(base)
    b.write_text("// a header comment\n\n" + base.replace("// doubles x", "// twice x") + "\n\n")
    c.write_text(base.replace("2 * x", "3 * x"))
    assert bench.code_hash(str(a)) == bench.code_hash(str(b))
    assert bench.code_hash(str(a)) != bench.code_hash(str(c))
