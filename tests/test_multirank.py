"""The bench's multi-rank host logic on CPU: two ranks over gloo (the N > 1 path runs one
independent replica per GPU, so the only cross-rank steps are the barrier and the max of the
per-rank step times; the reference arm runs on rank 0 alone)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["QSA_ROOT"])
import bench
rank, ws, local = bench.dist_init()
assert ws == 2 and rank == int(os.environ["RANK"])
bench.barrier(ws)
m = bench.max_over_ranks(1.5 + rank, ws)
print(json.dumps({"rank": rank, "max": m}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(code, extra_env=None, timeout=120):
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, QSA_ROOT=ROOT, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            p.kill()
            pytest.fail("rank did not finish")
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_two_ranks_barrier_and_max_over_ranks():
    outs = _run_ranks(_WORKER)
    got = sorted(json.loads(o.strip().splitlines()[-1])["rank"] for o in outs)
    assert got == [0, 1]
    for o in outs:
        assert json.loads(o.strip().splitlines()[-1])["max"] == 2.5


def test_reference_arm_runs_on_rank_zero_only():
    """`bench.py --impl reference` under two ranks: rank 1 exits 0 without work, rank 0 prints one line."""
    code = ("import os, sys; sys.path.insert(0, os.environ['QSA_ROOT']); sys.argv = ['bench.py', '--impl', "
            "'reference', '--steps', '1', '--warmup', '3']; import bench, workloads as W; "
            "W.verify_window = W.tiny_dense_decode; bench.main()")
    outs = _run_ranks(code)
    assert outs[1].strip() == ""
    line = json.loads(outs[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
