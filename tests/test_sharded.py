"""Context-sharded decode (each rank holding a page-aligned range of every slot's cells), host side
on CPU: the phases of sparse_selection_attention_gb300.sharded run on the FP64 oracle give the
oracle's unsharded window (the same selection, and outputs equal up to FP64 rounding), for 1 to 4
ranks run in turn and for 2 ranks exchanging over gloo."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import oracle as O
import workloads as W
from _shard_oracle import OracleBackend
from sparse_selection_attention_gb300 import sharded

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _case():
    # two slots with fills of 9 and 5 pages of 64 cells (ragged last block), rows early in the context
    return W.decode_case(name="shard", seed=77, fills=[560, 300], capacity=640, rows_per_slot=2, n_q_heads=6,
                         n_kv_heads=2, k_cells=192, chunk_cells=48, page_cells=64, bias_prob=0.05,
                         row_pos=[559, 200, 299, 64])


def _check(case, ids, n_sel, out, lse, ref):
    for t in range(case.n_rows):
        assert n_sel[t] == ref["n_sel"][t]
        assert np.array_equal(np.asarray(ids[t][:n_sel[t]]), np.asarray(ref["ids"][t]))
    assert np.allclose(out, ref["out"], rtol=0, atol=1e-12)
    fin = np.isfinite(ref["lse"])
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.allclose(lse[fin], ref["lse"][fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_sharded_phases_equal_unsharded_window(world):
    case = _case()
    ref = O.decode_window(case)
    ids, n_sel, out, lse = sharded.run_ranks_in_turn(
        OracleBackend(), case.pools, list(case.row_pool), case.q, case.row_pos, case.n_q_heads, case.block_cells,
        case.k_cells, case.chunk_cells, case.n_chunks, case.max_blocks, world)
    _check(case, ids, n_sel, out, lse, ref)


def test_page_runs_cover_the_fill():
    for n_filled, pc, world in [(560, 64, 3), (64, 64, 4), (0, 256, 2), (1000, 128, 8)]:
        runs = sharded.page_runs(n_filled, pc, world)
        assert runs[0][0] == 0 and runs[-1][1] == (n_filled + pc - 1) // pc
        assert all(a <= b for a, b in runs) and all(runs[i][1] == runs[i + 1][0] for i in range(world - 1))


_WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["QSA_ROOT"]); sys.path.insert(0, os.path.join(os.environ["QSA_ROOT"], "tests"))
import numpy as np
import torch.distributed as dist
from test_sharded import _case
from _shard_oracle import OracleBackend
from sparse_selection_attention_gb300 import sharded
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()

def gather(x):
    out = [None] * world
    dist.all_gather_object(out, x)
    return out

case = _case()
ids, n_sel, out, lse = sharded.run_window(OracleBackend(), case.pools, list(case.row_pool), case.q, case.row_pos,
                                          case.n_q_heads, case.block_cells, case.k_cells, case.chunk_cells,
                                          case.n_chunks, case.max_blocks, rank, world, gather)
print(json.dumps({"rank": rank, "n_sel": [int(x) for x in n_sel],
                  "ids": [[int(v) for v in ids[t][:n_sel[t]]] for t in range(case.n_rows)],
                  "out": np.asarray(out).ravel().tolist(), "lse": [float(x) for x in np.asarray(lse).ravel()]}),
      flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_exchange_to_the_unsharded_result():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, QSA_ROOT=ROOT, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", _WORKER], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=300)
        assert p.returncode == 0, e
        outs.append(json.loads(o.strip().splitlines()[-1]))
    case = _case()
    ref = O.decode_window(case)
    for res in outs:
        out = np.asarray(res["out"]).reshape(ref["out"].shape)
        lse = np.asarray(res["lse"]).reshape(ref["lse"].shape)
        _check(case, res["ids"], res["n_sel"], out, lse, ref)
