"""The decode attention entry point that allocates nothing.

Some callers cannot lend the library a scratch buffer: an engine that
reserves all device memory up front for its KV pool, or a plugin whose
interface carries only input and output pointers.  qsa_decode_attn_noalloc
serves them with a fixed scratch array the library owns.  These tests call it
through the C ABI twice in a row and compare each result with the existing
entry points (qsa_decode_attn + qsa_attn_merge with a caller buffer), within
the tolerance the other parity tests use.  This file is collected last."""
import numpy as np
import pytest
import torch

import sparse_selection_attention_gb300 as qsa
import workloads as W
from _parity import assert_close, upload_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [W.verify_window, W.batched_long_context, W.tiny_dense_decode])
def test_noalloc_matches_caller_scratch_twice(make):
    case = make()
    win, q, row_pos = upload_case(case)
    win.run(q, row_pos)            # caller-scratch path: scores, top-k, attention, merge
    torch.cuda.synchronize()
    ref_out, ref_lse = win.out.cpu().numpy(), win.lse.cpu().numpy()
    for _ in range(2):
        out = torch.full_like(win.out, float("nan"))
        lse = torch.full_like(win.lse, float("nan"))
        qsa.decode_attn_noalloc(win.pools, win.row_pool, q, row_pos, win.ids, win.n_sel, case.k_cells,
                                case.chunk_cells, out, lse)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref_out, "noalloc out")
        assert_close(lse.cpu().numpy(), ref_lse, "noalloc lse")


def _noalloc_vs_caller_scratch(case):
    """One no-allocation call on a fresh pair of outputs, checked against the caller-scratch path."""
    win, q, row_pos = upload_case(case)
    win.run(q, row_pos)
    torch.cuda.synchronize()
    out = torch.full_like(win.out, float("nan"))
    lse = torch.full_like(win.lse, float("nan"))
    qsa.decode_attn_noalloc(win.pools, win.row_pool, q, row_pos, win.ids, win.n_sel, case.k_cells,
                            case.chunk_cells, out, lse)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), win.out.cpu().numpy(), f"noalloc out ({case.name})")
    assert_close(lse.cpu().numpy(), win.lse.cpu().numpy(), f"noalloc lse ({case.name})")


def test_noalloc_ragged_odd_sizes_back_to_back():
    """Odd q-head counts, a last chunk that is only partly filled, and two calls in a row of which the
    second is the smaller: partials the first call left behind in the shared array must not leak into
    the second result."""
    big = W.decode_case(name="odd-big", seed=31, fills=[1500], capacity=1600, rows_per_slot=3, n_q_heads=3,
                        n_kv_heads=1, k_cells=704, chunk_cells=48, page_cells=64, bias_prob=0.05)
    small = W.decode_case(name="odd-small", seed=32, fills=[333], capacity=384, rows_per_slot=1, n_q_heads=1,
                          n_kv_heads=1, k_cells=192, chunk_cells=80, page_cells=64, bias_prob=0.05)
    _noalloc_vs_caller_scratch(big)
    _noalloc_vs_caller_scratch(small)


def test_noalloc_refuses_windows_past_its_scratch():
    case = W.verify_window()
    win, q, row_pos = upload_case(case)
    win.run(q, row_pos)
    torch.cuda.synchronize()
    out = torch.zeros_like(win.out)
    # 16-cell chunks of 4,096 cells: 5 x 24 x 256 x 520 B > 8 MiB
    with pytest.raises(qsa.QsaError) as err:
        qsa.decode_attn_noalloc(win.pools, win.row_pool, q, row_pos, win.ids, win.n_sel, case.k_cells, 16, out)
    assert err.value.status == qsa.QSA_ERR_SCRATCH
    assert torch.count_nonzero(out) == 0
