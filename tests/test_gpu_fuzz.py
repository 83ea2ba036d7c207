"""Seeded random decode windows and prompt calls against the FP64 oracle, through the C ABI.

Each case draws its shape at random within the library's limits: one to three pools with ragged
fills and their own capacities, 1-4 rows per pool, 1-8 KV heads (at most 16 warp tasks of 16 cells per block) with 1-6 q heads each, 32-, 64- or
128-cell blocks, pages of 64-256 cells, a top-k of 1-40 blocks, chunks of any multiple of 16
cells, int8 or 4-bit K and V, codes down to -128, and block summaries on some pools' sets.  Every
case runs the four separate calls and the one-call window, and some the window with page-locked
host buffers; the gates are those of the other decode tests (ids bit-exact given the GPU's own
scores, floats within 1e-5 of the output scale)."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_selection_attention_gb300 as qsa
import workloads as W
from _parity import assert_close, gpu_ids

pytestmark = pytest.mark.gpu

N_CASES = 40
N_PROMPT_CASES = 24


def draw_case(seed: int):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.choice([32, 64, 128]))
    hkv_choices = [h for h in (1, 2, 3, 4, 6, 8) if h * (B // 16) <= 16]   # both score kernels
    Hkv = int(rng.choice(hkv_choices))
    G = int(rng.choice([1, 2, 3, 4, 6]))
    n_pools = int(rng.integers(1, 4))
    rows_per_slot = int(rng.integers(1, 5))
    page_cells = int(rng.choice([p for p in (64, 128, 256) if p % B == 0]))
    fills = [int(rng.integers(rows_per_slot, 5001)) for _ in range(n_pools)]
    capacity = max(fills) + int(rng.integers(0, 700))
    k_cells = B * int(rng.integers(1, 41))
    chunk_cells = 16 * int(rng.integers(1, 17))
    v_bits = int(rng.choice([8, 4]))
    k_bits = int(rng.choice([8, 4]))
    code_lo = int(rng.choice([-127, -128]))
    sums = bool(rng.integers(0, 2)) and B % 64 == 0
    host = bool(rng.integers(0, 2))
    case = W.decode_case(name=f"fuzz{seed}", seed=2000 + seed, fills=fills, capacity=capacity,
                         rows_per_slot=rows_per_slot, n_q_heads=G * Hkv, n_kv_heads=Hkv, k_cells=k_cells,
                         chunk_cells=chunk_cells, block_cells=B, page_cells=page_cells, bias_prob=0.05,
                         v_bits=v_bits, k_bits=k_bits, code_lo=code_lo)
    return case, sums, host


def make_window(case, sums):
    pools = [qsa.DevicePool.upload(p) for p in case.pools]
    if sums:
        pools = [p.keep_block_sums() for p in pools]
    return qsa.DecodeWindow(pools, case.row_pool, case.n_q_heads, case.block_cells, case.k_cells, case.chunk_cells,
                            n_chunks=case.n_chunks, max_blocks=case.max_blocks)


def check(case, win, out, lse, what):
    scores = win.scores.cpu().numpy()
    ref = O.decode_window(case, scores_f32=scores)
    for t in range(case.n_rows):
        nb = len(ref["scores"][t])
        assert_close(scores[t, :nb], ref["scores"][t], f"{what}: scores row {t}")
    ids, n_sel = gpu_ids(win)
    for t in range(case.n_rows):
        assert n_sel[t] == ref["n_sel"][t], f"{what}: n_sel row {t}"
        assert np.array_equal(ids[t], ref["ids"][t]), f"{what}: ids row {t}"
    assert_close(out, ref["out"], f"{what}: out")
    assert_close(lse, ref["lse"], f"{what}: lse")


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_window(seed):
    case, sums, host = draw_case(seed)
    win = make_window(case, sums)
    q = torch.from_numpy(case.q).cuda()
    pos = torch.from_numpy(case.row_pos).cuda()
    # the four separate calls
    win.run(q, pos)
    torch.cuda.synchronize()
    check(case, win, win.out.cpu().numpy(), win.lse.cpu().numpy(), "four calls")
    # the one-call window
    win.out.fill_(float("nan"))
    win.lse.fill_(float("nan"))
    win.run_window(q, pos)
    torch.cuda.synchronize()
    check(case, win, win.out.cpu().numpy(), win.lse.cpu().numpy(), "window")
    if host:
        q_h = torch.from_numpy(np.ascontiguousarray(case.q)).pin_memory()
        pos_h = torch.from_numpy(np.ascontiguousarray(case.row_pos)).pin_memory()
        out_h = torch.full(tuple(win.out.shape), float("nan")).pin_memory()
        lse_h = torch.full(tuple(win.lse.shape), float("nan")).pin_memory()
        win.run_window_host(q_h, pos_h, out_h, lse_h)
        torch.cuda.synchronize()
        check(case, win, out_h.numpy(), lse_h.numpy(), "window, host buffers")
    assert qsa.get_device_error() == 0


def draw_prompt_case(seed: int):
    """A prompt call of 1-256 queries at the end of a 64-2,000-cell context (or from position 0),
    1-4 KV heads with 1-8 q heads each, pages of 64-256 cells, int8 or 4-bit K and V."""
    rng = np.random.default_rng(5000 + seed)
    Hkv = int(rng.integers(1, 5))
    G = int(rng.integers(1, 9))
    n_ctx = int(rng.integers(64, 2001))
    n_q = int(rng.integers(1, min(256, n_ctx) + 1))
    if rng.integers(0, 4) == 0:
        n_q = n_ctx   # the whole context is the prompt: queries from position 0
    return W.prompt_case(name=f"pfuzz{seed}", seed=6000 + seed, n_ctx=n_ctx, n_q=n_q, n_q_heads=G * Hkv,
                         n_kv_heads=Hkv, v_bits=int(rng.choice([8, 4])), k_bits=int(rng.choice([8, 4])),
                         page_cells=int(rng.choice([64, 128, 256])), capacity=n_ctx + int(rng.integers(0, 300)),
                         code_lo=int(rng.choice([-127, -128])))


@pytest.mark.parametrize("seed", range(N_PROMPT_CASES))
def test_random_prompt(seed):
    case = draw_prompt_case(seed)
    i0, n, pos0 = case.calls[0]
    pool = qsa.DevicePool.upload(case.pool)
    q = torch.from_numpy(np.ascontiguousarray(case.q[i0:i0 + n])).cuda()
    out = torch.full((n, case.n_q_heads, 128), float("nan"), device="cuda")
    lse = torch.full((n, case.n_q_heads), float("nan"), device="cuda")
    qsa.prompt_attn(pool, q, pos0, out, lse)
    torch.cuda.synchronize()
    assert qsa.get_device_error() == 0
    ref_out, ref_lse = O.prompt_attention(case.pool, case.q, pos0)
    assert_close(out.cpu().numpy(), ref_out, "out")
    assert_close(lse.cpu().numpy(), ref_lse, "lse")
