"""bench.py's multi-rank host logic on the CPU: two gloo ranks.

Rows are independent, so N GPUs run N replicas with no collective on the
data path; what the ranks share is host plumbing -- a barrier, the max of
the timings and the sum of the bytes -- and only rank 0 prints.  These tests
run that plumbing as two local processes with the gloo backend.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(code: str, world: int = 2, timeout: int = 300):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", code], cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=timeout)
        outs.append((p.returncode, o, e))
    return outs


def test_max_and_sum_over_two_gloo_ranks():
    code = (
        "import json, os, bench\n"
        "dist, rank, world, local = bench.dist_setup(2)\n"
        "assert world == 2 and dist is not None\n"
        "t = 10.0 + rank\n"
        "m = bench.max_over_ranks(dist, t)\n"
        "s = bench.sum_over_ranks(dist, 1000.0 * (rank + 1))\n"
        "bench.barrier(dist)\n"
        "print(json.dumps({'rank': rank, 'max': m, 'sum': s}))\n"
        "dist.destroy_process_group()\n")
    outs = _run_ranks(code)
    for rc, o, e in outs:
        assert rc == 0, e
        d = json.loads(o.strip().splitlines()[-1])
        assert d["max"] == 11.0 and d["sum"] == 3000.0


def test_reference_arm_prints_on_rank_zero_only():
    code = ("import bench\n"
            "bench.main(['--impl', 'reference', '--workload', 'tiny-fp32', '--gpus', '2',\n"
            "            '--steps', '2', '--warmup', '1', '--ref-step-seconds', '0.01'])\n")
    outs = _run_ranks(code)
    (rc0, o0, e0), (rc1, o1, e1) = outs
    assert rc0 == 0 and rc1 == 0, (e0, e1)
    line = json.loads(o0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert o1.strip() == ""


def test_row_replicas_are_weak_scaling():
    """Each rank's workload is the whole configuration (its own pool and rows)."""
    code = ("import json, bench, workloads as wl\n"
            "dist, rank, world, local = bench.dist_setup(2)\n"
            "w = wl.WORKLOADS['bf16-long']\n"
            "md = wl.metadata(w)\n"
            "b = bench.algorithmic_bytes(w, md)['kv']\n"
            "tot = bench.sum_over_ranks(dist, float(b))\n"
            "print(json.dumps({'mine': b, 'total': tot}))\n"
            "dist.destroy_process_group()\n")
    outs = _run_ranks(code)
    vals = [json.loads(o.strip().splitlines()[-1]) for rc, o, e in outs]
    assert all(rc == 0 for rc, _, _ in outs)
    assert vals[0]["mine"] == vals[1]["mine"]
    assert vals[0]["total"] == 2 * vals[0]["mine"]
