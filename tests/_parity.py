"""Helpers shared by the GPU parity tests: upload seeded cases, run the CUDA
path through the C ABI, and compare with the oracle."""
import json
import os

import numpy as np
import torch

import oracle as O
import sparse_selection_attention_gb300 as qsa

# Gate for float outputs: max |gpu - oracle| / max |oracle| per tensor.
REL_TOL = 1e-5


def rel_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(gpu)), "finite patterns differ"
    assert np.array_equal(ref[~fin], gpu[~fin]), "non-finite values differ"
    if not fin.any():
        return 0.0
    scale = np.abs(ref[fin]).max()
    if scale == 0.0:
        return float(np.abs(gpu[fin]).max())
    return float(np.abs(gpu[fin] - ref[fin]).max() / scale)


def assert_close(gpu, ref, what, tol=REL_TOL):
    e = rel_err(gpu, ref)
    assert e <= tol, f"{what}: max rel err {e:.3e} > {tol:.1e}"
    return e


def upload_case(case, device="cuda"):
    pools = [qsa.DevicePool.upload(p, device) for p in case.pools]
    win = qsa.DecodeWindow(pools, case.row_pool, case.n_q_heads, case.block_cells, case.k_cells,
                           case.chunk_cells, n_chunks=case.n_chunks, max_blocks=case.max_blocks, device=device)
    q = torch.from_numpy(case.q).to(device)
    row_pos = torch.from_numpy(case.row_pos).to(device)
    return win, q, row_pos


def gpu_ids(win):
    ids = win.ids.cpu().numpy()
    n_sel = win.n_sel.cpu().numpy()
    return [ids[t, :n_sel[t]].copy() for t in range(win.n_rows)], n_sel


def run_window_and_check(case):
    win, q, row_pos = upload_case(case)
    win.out.fill_(float("nan"))
    win.lse.fill_(float("nan"))
    win.run_window(q, row_pos)
    torch.cuda.synchronize()
    R = case.n_rows
    scores_gpu = win.scores.cpu().numpy()
    ref = O.decode_window(case, scores_f32=scores_gpu)
    for t in range(R):
        nb = len(ref["scores"][t])
        assert_close(scores_gpu[t, :nb], ref["scores"][t], f"scores row {t}")
    ids, n_sel = gpu_ids(win)
    for t in range(R):
        assert n_sel[t] == ref["n_sel"][t], f"n_sel row {t}"
        assert np.array_equal(ids[t], ref["ids"][t]), f"ids row {t}"
    assert_close(win.out.cpu().numpy(), ref["out"], "out")
    assert_close(win.lse.cpu().numpy(), ref["lse"], "lse")
    return win, q, row_pos


def row_stats(gpu, ref):
    """Row-wise relative error of an output [rows, heads, D]: for every (query, head) vector
    ||gpu - ref|| / ||ref||; returns (mean, max) over the vectors with ||ref|| > 0."""
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1, np.shape(gpu)[-1])
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, np.shape(ref)[-1])
    nr = np.linalg.norm(ref, axis=1)
    ok = nr > 0
    r = np.linalg.norm(gpu - ref, axis=1)[ok] / nr[ok]
    return float(r.mean()), float(r.max())


def report(name, **stats):
    """Prints a parity record; with QSA_PARITY_REPORT set, also appends it to that JSON-lines file."""
    rec = {"case": name, **stats}
    print("PARITY", json.dumps(rec))
    path = os.environ.get("QSA_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")
