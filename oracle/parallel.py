"""Runs the FP64 oracle over the host's cores (test and baseline infrastructure).

TEST INFRASTRUCTURE ONLY: imported by the tests and by the bench's CPU-baseline
leg, never by the library.  It has no arithmetic of its own: every number comes
from a function of oracle.qsa_oracle, called on a slice of the work (a block of
prompt rows and the q heads of one KV head; one decode row).  Workers are
started with the "spawn" method (safe next to a CUDA context) and rebuild their
inputs from the seeded generators in `workloads`, so no pool is pickled.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from typing import Dict, List, Tuple

import numpy as np

_CASE = None   # the worker's copy of the case


def _build(builder: str, kwargs: Dict):
    import workloads as W
    return getattr(W, builder)(**kwargs)


def _init(builder: str, kwargs: Dict):
    global _CASE
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    _CASE = _build(builder, kwargs)


def _prompt_task(args):
    import oracle.qsa_oracle as O
    call_index, rows, heads = args
    i0, n_q, pos0 = _CASE.calls[call_index]
    out, lse = O.prompt_attention(_CASE.pool, _CASE.q[i0:i0 + n_q], pos0, rows=rows, heads=heads)
    return rows, heads, out[:, heads], lse[:, heads]


def workers(n: int = 0) -> int:
    return n if n > 0 else (os.cpu_count() or 1)


def prompt_call(builder: str, kwargs: Dict, call_index: int, n_workers: int = 0, row_block: int = 128,
                rows: List[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """out [n, Hq, 128] and lse [n, Hq] (float64) of the given rows (default: every row) of one prompt
    call of the case `workloads.<builder>(**kwargs)`, by oracle.prompt_attention over tasks (row block,
    KV head)."""
    case = _build(builder, kwargs)
    _, n_q, _ = case.calls[call_index]
    rows = list(range(n_q)) if rows is None else list(rows)
    Hq, Hkv = case.n_q_heads, case.pool.n_kv_heads
    G = Hq // Hkv
    tasks = [(call_index, rows[r0:r0 + row_block], list(range(h * G, (h + 1) * G)))
             for h in range(Hkv) for r0 in range(0, len(rows), row_block)]
    where = {r: i for i, r in enumerate(rows)}
    out = np.zeros((len(rows), Hq, case.q.shape[2]))
    lse = np.full((len(rows), Hq), -np.inf)
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers(n_workers), initializer=_init, initargs=(builder, kwargs)) as pool:
        for rws, heads, o, l in pool.imap_unordered(_prompt_task, tasks):
            idx = [where[r] for r in rws]
            out[np.ix_(idx, heads)] = o
            lse[np.ix_(idx, heads)] = l
    return out, lse


def _window_task(t: int):
    """One decode row of the worker's case: its pool's block scores, top-k, chunk partials, merge."""
    import oracle.qsa_oracle as O
    case = _CASE
    pool = case.pools[case.row_pool[t]]
    s = O.block_scores(pool, case.q[[t]], case.block_cells)[0]
    sel, _ = O.topk_select(s.astype(np.float32), pool.n_filled, case.block_cells, case.k_cells)
    m, l, o = O.chunk_partials(pool, case.q[t], int(case.row_pos[t]), sel, case.chunk_cells, case.n_chunks)
    O.merge_partials(m, l, o)
    return t


class WindowRunner:
    """A pool of workers holding one decode case; run(n) computes n whole windows (every row of each),
    the rows of all windows spread over the workers."""

    def __init__(self, builder: str, kwargs: Dict, n_workers: int = 0):
        self.n_rows = _build(builder, kwargs).n_rows
        self.n_workers = workers(n_workers)
        self.pool = mp.get_context("spawn").Pool(self.n_workers, initializer=_init, initargs=(builder, kwargs))

    def run(self, n_windows: int) -> None:
        list(self.pool.imap_unordered(_window_task, [t for _ in range(n_windows) for t in range(self.n_rows)]))

    def close(self) -> None:
        self.pool.close()
        self.pool.join()


__all__: List[str] = ["prompt_call", "WindowRunner", "workers"]
