"""Context-sharded decode on the GPU: the ranks of a window run one after another on this one GPU
(each exchange is a list in rank order, no kernel waits on another), through the library's pool
views, qsa_ids_in_range and qsa_attn_merge_shards.  Gates as for one GPU: the gathered scores within
1e-5 of the oracle's, the selection bit-exact given those scores, out and lse within 1e-5."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_selection_attention_gb300 as qsa
import workloads as W
from _parity import assert_close
from sparse_selection_attention_gb300 import sharded

pytestmark = pytest.mark.gpu


def run_sharded(case, world, block_sums=False):
    pools = [qsa.DevicePool.upload(p) for p in case.pools]
    if block_sums:
        pools = [p.keep_block_sums() for p in pools]
    q = torch.from_numpy(case.q).cuda()
    row_pos = torch.from_numpy(case.row_pos).cuda()
    be = sharded.LibraryBackend()
    ids, n_sel, out, lse = sharded.run_ranks_in_turn(be, pools, list(case.row_pool), q, row_pos, case.n_q_heads,
                                                     case.block_cells, case.k_cells, case.chunk_cells,
                                                     case.n_chunks, case.max_blocks, world)
    torch.cuda.synchronize()
    return be.last_scores.cpu().numpy(), ids.cpu().numpy(), n_sel.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()


def check(case, world, block_sums=False):
    scores, ids, n_sel, out, lse = run_sharded(case, world, block_sums)
    ref = O.decode_window(case, scores_f32=scores)
    for t in range(case.n_rows):
        nb = len(ref["scores"][t])
        assert_close(scores[t, :nb], ref["scores"][t], f"scores row {t}")
        assert n_sel[t] == ref["n_sel"][t]
        assert np.array_equal(ids[t, :n_sel[t]], ref["ids"][t]), f"ids row {t}"
    assert_close(out, ref["out"], "out")
    assert_close(lse, ref["lse"], "lse")


@pytest.mark.parametrize("world", [1, 2, 3])
def test_small_two_pools(world):
    case = W.decode_case(name="shard", seed=77, fills=[560, 300], capacity=640, rows_per_slot=2, n_q_heads=6,
                         n_kv_heads=2, k_cells=192, chunk_cells=48, page_cells=64, bias_prob=0.05,
                         row_pos=[559, 200, 299, 64])
    check(case, world)


@pytest.mark.parametrize("world", [2, 4])
def test_batched_long_context_sharded(world):
    """The long-context window (2 slots x 2 rows, 65,536 / 131,072 cells, top-k 8,192) split over 2 and
    4 ranks."""
    check(W.batched_long_context(), world)


def test_q4_0_sharded():
    case = W.decode_case(name="shard q4_0", seed=79, fills=[1500], capacity=1536, rows_per_slot=3, n_q_heads=8,
                         n_kv_heads=2, k_cells=512, chunk_cells=64, page_cells=128, bias_prob=0.05, v_bits=4,
                         k_bits=4)
    check(case, 3)


def test_sharded_with_block_summaries():
    """Rank views keep the pools' block summaries: the ranks score their blocks from them."""
    check(W.batched_long_context(), 3, block_sums=True)
