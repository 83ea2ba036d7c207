"""Helpers shared by the GPU parity tests: upload seeded cases, run the CUDA
path through the C ABI, and compare with the oracle."""
import numpy as np
import torch

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
