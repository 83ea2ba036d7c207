"""Block summaries (qsa_pool.k_sums): built by qsa_kv_summarise and kept by qsa_kv_append, they match
the oracle's sums of dequantised K rows per 64-cell block; the decode window and qsa_block_scores that
score from them meet the usual gates (scores within 1e-5 of the oracle's R3 scores, the selection
bit-exact given the GPU's scores, out and lse within 1e-5)."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_selection_attention_gb300 as qsa
import workloads as W
from _parity import assert_close, gpu_ids
from test_gpu_append import new_rows

pytestmark = pytest.mark.gpu


def gpu_summaries(dp, pool):
    """The device summaries of the pool's filled blocks in logical block order, [nb, Hkv, 128]."""
    s = dp.k_sums.cpu().numpy()
    nb = (pool.n_filled + 63) // 64
    return np.stack([s[pool.page_table[b * 64 // pool.page_cells], :, (b * 64 % pool.page_cells) // 64]
                     for b in range(nb)])


@pytest.mark.parametrize("k_bits,v_bits,page_cells,fill", [(8, 8, 256, 1000), (4, 4, 128, 777), (8, 4, 64, 4096)])
def test_summaries_built(k_bits, v_bits, page_cells, fill):
    rng = np.random.default_rng(fill + k_bits)
    pool = W.make_pool(rng, capacity=fill + 300, n_filled=fill, n_kv_heads=4, page_cells=page_cells, v_bits=v_bits,
                       k_bits=k_bits)
    dp = qsa.DevicePool.upload(pool).keep_block_sums()
    torch.cuda.synchronize()
    assert_close(gpu_summaries(dp, pool), O.block_summaries(pool), "block summaries")


def test_summaries_kept_by_appends():
    """Three appends of ragged sizes after a built start: the summaries follow the fill."""
    rng = np.random.default_rng(11)
    pool = W.make_pool(rng, capacity=2048, n_filled=130, n_kv_heads=2, page_cells=128, v_bits=8)
    dp = qsa.DevicePool.upload(pool).keep_block_sums()
    for n in (5, 300, 77):
        k, v = new_rows(rng, n, 2)
        pool = O.append_cells(pool, k, v, pool.n_filled)
        qsa.kv_append(dp, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), dp.n_filled)
        torch.cuda.synchronize()
        assert dp.n_filled == pool.n_filled
        assert_close(gpu_summaries(dp, pool), O.block_summaries(pool), f"summaries after {pool.n_filled} cells")


def upload_with_sums(case):
    pools = [qsa.DevicePool.upload(p).keep_block_sums() for p in case.pools]
    win = qsa.DecodeWindow(pools, case.row_pool, case.n_q_heads, case.block_cells, case.k_cells, case.chunk_cells,
                           n_chunks=case.n_chunks, max_blocks=case.max_blocks)
    return win, torch.from_numpy(case.q).cuda(), torch.from_numpy(case.row_pos).cuda()


def check(case, window: bool):
    win, q, row_pos = upload_with_sums(case)
    (win.run_window if window else win.run)(q, row_pos)
    torch.cuda.synchronize()
    scores = win.scores.cpu().numpy()
    ref = O.decode_window(case, scores_f32=scores)
    for t in range(case.n_rows):
        nb = len(ref["scores"][t])
        assert_close(scores[t, :nb], ref["scores"][t], f"scores row {t}")
    ids, n_sel = gpu_ids(win)
    for t in range(case.n_rows):
        assert n_sel[t] == ref["n_sel"][t] and np.array_equal(ids[t], ref["ids"][t]), f"ids row {t}"
    assert_close(win.out.cpu().numpy(), ref["out"], "out")
    assert_close(win.lse.cpu().numpy(), ref["lse"], "lse")


@pytest.mark.parametrize("window", [True, False])
def test_long_context_scored_from_summaries(window):
    check(W.batched_long_context(), window)


@pytest.mark.parametrize("window", [True, False])
def test_verify_window_scored_from_summaries(window):
    check(W.verify_window(), window)


def test_ragged_128_cell_blocks_and_q4_0():
    case = W.decode_case(name="sums", seed=41, fills=[1000, 333], capacity=1024, rows_per_slot=3, n_q_heads=8,
                         n_kv_heads=2, k_cells=256, chunk_cells=64, block_cells=128, page_cells=128, bias_prob=0.05,
                         v_bits=4, k_bits=4)
    check(case, True)
    check(case, False)
