"""Host logic of the multi-GPU bench path, run on the CPU.

The decode path shards by sequence with no exchange step, so N GPUs run N
independent replicas; the bench's only cross-rank work is a barrier and a
maximum of the per-rank timings (the slowest replica sets the job's time).
These tests run that reduction as two gloo ranks and check the whole-job
throughput formula and that only rank 0 of the reference arm prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench as b

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank 1 has the slower step, rank 0 the slower decode kernel
        ms, dms = b.max_over_ranks([1.0 + rank, 0.5 - 0.1 * rank], world)
        (e2e,) = b.max_over_ranks([3.0 * (rank + 1)], world)
        dist.barrier()
        q.put((rank, ms, dms, e2e, b.job_tokens_per_s(world, 32, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    assert [r[0] for r in res] == [0, 1]
    for _, ms, dms, e2e, value in res:
        assert (ms, dms, e2e) == (2.0, 0.5, 6.0)  # element-wise max, same on every rank
        assert value == pytest.approx(2 * 32 / 2.0e-3)  # both replicas' tokens over the slowest time


def test_single_process_needs_no_group():
    assert bench.max_over_ranks([1.5, 2], 1) == [1.5, 2.0]
    assert bench.job_tokens_per_s(1, 32, 0.1) == pytest.approx(320000.0)
    assert bench.job_tokens_per_s(4, 32, 0.1) == pytest.approx(4 * 320000.0)


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank0():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "3", "--ref-seconds", "1"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
