"""GPU parity of the decode path (block scores -> top-k -> chunk attention ->
merge) against the FP64 oracle, through the C ABI.

Gates: selected ids bit-exact given identical fp32 scores (both directions);
float outputs max |gpu - oracle| / max |oracle| <= 1e-5 per tensor; bitwise
run-to-run determinism."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from _parity import assert_close, gpu_ids, upload_case

pytestmark = pytest.mark.gpu


def run_and_check(case, check_partials=True):
    win, q, row_pos = upload_case(case)
    win.run(q, row_pos)
    torch.cuda.synchronize()
    R = case.n_rows
    scores_gpu = win.scores.cpu().numpy()
    # The oracle ranks the GPU's own fp32 scores: ids must match bit for bit.
    ref = O.decode_window(case, scores_f32=scores_gpu)
    for t in range(R):
        nb = len(ref["scores"][t])
        assert_close(scores_gpu[t, :nb], ref["scores"][t], f"scores row {t}")
    ids, n_sel = gpu_ids(win)
    for t in range(R):
        assert n_sel[t] == ref["n_sel"][t], f"n_sel row {t}"
        assert np.array_equal(ids[t], ref["ids"][t]), f"ids row {t}"
    if check_partials:
        ml, o = win.partial_views()
        ml, o = ml.cpu().numpy(), o.cpu().numpy()
        for t in range(R):
            n_act = (int(n_sel[t]) + case.chunk_cells - 1) // case.chunk_cells
            assert_close(ml[t, :, :n_act, 0], ref["m"][t][:, :n_act], f"chunk m row {t}")
            assert_close(ml[t, :, :n_act, 1], ref["l"][t][:, :n_act], f"chunk l row {t}")
            assert_close(o[t, :, :n_act], ref["o"][t][:, :n_act], f"chunk o row {t}")
    assert_close(win.out.cpu().numpy(), ref["out"], "out")
    assert_close(win.lse.cpu().numpy(), ref["lse"], "lse")
    return win, q, row_pos


def test_tiny_dense_decode():
    """1 query, 2 q heads on 1 KV head, 1,024 cells, top-k = all, 4 chunks of 256."""
    case = W.tiny_dense_decode()
    win, _, _ = run_and_check(case)
    assert int(win.n_sel[0]) == 1024


@pytest.mark.parametrize("fill,page_cells,Hq,Hkv,k,C,v_bits,k_bits", [
    (1000, 128, 6, 2, 256, 64, 8, 8),      # ragged last block, 4 blocks chosen of 16
    (1000, 256, 8, 1, 2048, 48, 8, 8),     # k > all cells: take all; ragged chunks of 48
    (777, 64, 4, 4, 320, 112, 4, 8),       # 4-bit V, group 1, odd chunk size
    (300, 64, 24, 4, 64, 16, 8, 8),        # one block, 16-cell chunks
    (1000, 128, 6, 2, 256, 64, 4, 4),      # q4_0 (4-bit K and V): ragged last block
    (777, 64, 8, 2, 320, 48, 8, 4),        # 4-bit K with int8 V, ragged chunks of 48
])
def test_small_ragged(fill, page_cells, Hq, Hkv, k, C, v_bits, k_bits):
    case = W.decode_case(name="ragged", seed=fill + k, fills=[fill], capacity=fill + 100, rows_per_slot=3,
                         n_q_heads=Hq, n_kv_heads=Hkv, k_cells=k, chunk_cells=C, page_cells=page_cells,
                         v_bits=v_bits, bias_prob=0.05, k_bits=k_bits)
    run_and_check(case)


@pytest.mark.parametrize("fill,Hq,Hkv,k,C", [
    (64, 1, 1, 64, 64),        # one row, one head, one chunk: 1 (row, head, chunk) entry of partials
    (700, 3, 1, 192, 64),      # three q heads on one KV head, three chunks: 9 entries
    (500, 3, 1, 320, 48),      # ragged chunks of 48 over a selection of 320
])
def test_odd_partial_counts(fill, Hq, Hkv, k, C):
    """An odd number of (row, head, chunk) entries: the o region of the partials still starts on a
    16-byte boundary (it starts at the next 256-byte boundary after the (m, l) pairs)."""
    case = W.decode_case(name="odd", seed=fill + Hq, fills=[fill], capacity=fill + 64, rows_per_slot=1,
                         n_q_heads=Hq, n_kv_heads=Hkv, k_cells=k, chunk_cells=C, page_cells=64,
                         bias_prob=0.05)
    run_and_check(case)


def test_codes_of_minus_128():
    """int8 K and V codes drawn in [-128, 127]: scores, selection, partials and outputs stay at parity
    (the one code without a positive twin goes through the exact fp16 conversions)."""
    case = W.decode_case(name="m128", seed=128, fills=[1500], capacity=1600, rows_per_slot=3, n_q_heads=12,
                         n_kv_heads=2, k_cells=512, chunk_cells=64, page_cells=128, bias_prob=0.05, code_lo=-128)
    assert (case.pools[0].k_codes == -128).any() and (case.pools[0].v_codes == -128).any()
    run_and_check(case)
    from _parity import run_window_and_check
    run_window_and_check(case)


@pytest.mark.parametrize("rows_per_slot,Hq,Hkv,B", [
    (10, 16, 8, 64),    # 20 rows (three 8-row tiles), 8 KV heads: two warp tasks per warp
    (6, 8, 2, 128),     # 12 rows, 128-cell blocks
    (4, 32, 4, 32),     # 8 rows, 32-cell blocks, 8 q heads per KV head
])
def test_many_rows_and_block_sizes(rows_per_slot, Hq, Hkv, B):
    case = W.decode_case(name="wide", seed=rows_per_slot * B + Hkv, fills=[2000, 1500], capacity=2048,
                         rows_per_slot=rows_per_slot, n_q_heads=Hq, n_kv_heads=Hkv, k_cells=4 * B,
                         chunk_cells=64, block_cells=B, page_cells=256, bias_prob=0.05)
    run_and_check(case)


def test_rows_with_masked_cells_and_two_pools():
    """Rows early in the context: selected cells past a row's position are masked; a chunk whose cells
    are all masked is empty; the merge skips it."""
    case = W.decode_case(name="masked", seed=5, fills=[900, 1500], capacity=2048, rows_per_slot=2,
                         n_q_heads=12, n_kv_heads=2, k_cells=512, chunk_cells=64, page_cells=128,
                         row_pos=[100, 899, 0, 1499], bias_prob=0.05)
    run_and_check(case)


def test_empty_selection():
    case = W.decode_case(name="k0", seed=9, fills=[500], capacity=512, rows_per_slot=2, n_q_heads=4,
                         n_kv_heads=1, k_cells=0, chunk_cells=64, page_cells=64, n_chunks=2)
    win, q, row_pos = upload_case(case)
    win.run(q, row_pos)
    torch.cuda.synchronize()
    assert win.n_sel.cpu().tolist() == [0, 0]
    assert torch.all(win.out == 0) and torch.all(torch.isinf(win.lse)) and torch.all(win.lse < 0)


def test_verify_window_full_size():
    """5 rows, 24/4 heads, 32,768 cells, k = 4,096, 64-cell chunks (the bench's workload)."""
    run_and_check(W.verify_window())


def test_batched_long_context_full_size():
    """2 slots x 2 rows, capacity 200,000, fills 65,536 / 131,072, k = 8,192, one launch over both pools."""
    run_and_check(W.batched_long_context())


def test_batched_long_context_512_chunk_buffer():
    """Partials sized for 512 chunks per row: chunks 128..511 hold no cells and are never read."""
    case = W.batched_long_context(n_chunks=512)
    win, q, row_pos = upload_case(case)
    win.partials.fill_(float("nan"))   # anything the merge touched past the selection would poison out
    win.run(q, row_pos)
    torch.cuda.synchronize()
    ref = O.decode_window(case, scores_f32=win.scores.cpu().numpy())
    assert_close(win.out.cpu().numpy(), ref["out"], "out")
    assert_close(win.lse.cpu().numpy(), ref["lse"], "lse")


def test_topk_on_oracle_scores_and_adversarial_keys():
    """The GPU top-k ranks the oracle's fp32 scores, and hand-built scores full of ties, signed zeros,
    NaN and infinities, exactly like the oracle's full sort."""
    import sparse_selection_attention_gb300 as qsa
    rng = np.random.default_rng(3)
    B = 64
    rows = []
    case = W.verify_window()
    s64 = O.block_scores(case.pools[0], case.q, B)
    for t in range(case.n_rows):
        rows.append((s64[t].astype(np.float32), 32768, 4096))
    specials = np.array([-np.inf, -1.0, -0.0, 0.0, 1.0, np.inf, np.nan, 2.0], np.float32)
    for n_filled, k in [(64 * 3000, 64 * 700), (64 * 2000 - 5, 64 * 1999), (64 * 37 + 1, 64 * 38), (64 * 500, 64 * 3),
                        (64 * 16384, 64 * 4096), (64 * 16384 - 63, 64 * 1)]:   # QSA_MAX_TOPK_BLOCKS candidates
        nb = (n_filled + B - 1) // B
        rows.append((rng.choice(specials, nb).astype(np.float32), n_filled, k))
        rows.append((rng.integers(-3, 4, nb).astype(np.float32), n_filled, k))
    for scores, n_filled, k in rows:
        nb = (n_filled + B - 1) // B
        s = torch.from_numpy(np.ascontiguousarray(scores[None, :nb])).cuda()
        ids = torch.full((1, k), -7, dtype=torch.int32, device="cuda")
        n_sel = torch.zeros(1, dtype=torch.int32, device="cuda")
        qsa.topk(s, [n_filled], B, k, ids, n_sel)
        want, n = O.topk_select(scores[:nb], n_filled, B, k)
        assert int(n_sel) == n
        assert np.array_equal(ids[0, :n].cpu().numpy(), want)


def test_deterministic_bitwise():
    case = W.verify_window()
    win, q, row_pos = upload_case(case)
    outs = []
    for _ in range(3):
        win.run(q, row_pos)
        torch.cuda.synchronize()
        outs.append((win.scores.clone(), win.ids.clone(), win.partials.clone(), win.out.clone(), win.lse.clone()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    for a, b in zip(outs[0], outs[2]):
        assert torch.equal(a, b)


def test_chunk_size_changes_only_rounding():
    """Another split of the same selection stays within the gate (and equals the oracle)."""
    case = W.verify_window()
    win, q, row_pos = upload_case(case)
    win.run(q, row_pos)
    torch.cuda.synchronize()
    base = win.out.cpu().numpy()
    import sparse_selection_attention_gb300 as qsa
    for C in (128, 256, 1024):
        n_chunks = (case.k_cells + C - 1) // C
        part = torch.zeros(qsa.decode_partials_bytes(case.n_rows, case.n_q_heads, n_chunks) // 4, device="cuda")
        out = torch.zeros_like(win.out)
        qsa.decode_attn(win.pools, win.row_pool, q, row_pos, win.ids, win.n_sel, case.k_cells, C, n_chunks, part)
        qsa.attn_merge(part, win.n_sel, case.n_rows, case.n_q_heads, C, n_chunks, out)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), base, f"chunk {C} vs 64")
