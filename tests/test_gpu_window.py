"""GPU parity of the one-call decode window (qsa_decode_window: q fragments ->
block scores -> top-k -> split attention -> log-sum-exp merge, five chained
launches) against the FP64 oracle, through the C ABI.

Gates as for the four separate calls: ids bit-exact given the GPU's own fp32
scores; scores, out and lse within max |gpu - oracle| / max |oracle| <= 1e-5;
bitwise run-to-run determinism."""
import dataclasses

import numpy as np
import pytest
import torch

import sparse_selection_attention_gb300 as qsa
import workloads as W
from _parity import assert_close, gpu_ids, run_window_and_check, upload_case

pytestmark = pytest.mark.gpu


def test_window_tiny_dense_decode():
    run_window_and_check(W.tiny_dense_decode())


def test_window_verify_window_full_size():
    run_window_and_check(W.verify_window())


def test_window_batched_long_context_full_size():
    run_window_and_check(W.batched_long_context())


@pytest.mark.parametrize("fill,page_cells,Hq,Hkv,k,v_bits,B", [
    (1000, 128, 6, 2, 256, 8, 64),      # ragged last block
    (1000, 256, 8, 1, 2048, 8, 64),     # k above all cells: take all
    (777, 64, 4, 4, 320, 4, 64),        # 4-bit V
    (300, 64, 24, 4, 64, 8, 64),        # one block
    (2000, 256, 32, 4, 512, 8, 128),    # 128-cell blocks, 8 q heads per KV head
    (2000, 256, 16, 8, 256, 8, 32),     # 32-cell blocks, 8 KV heads
    (3000, 256, 16, 16, 1024, 8, 32),   # 16 KV heads x 2 m-tiles: 32 warps per block
])
def test_window_small_ragged(fill, page_cells, Hq, Hkv, k, v_bits, B):
    case = W.decode_case(name="wragged", seed=fill + k + B, fills=[fill], capacity=fill + 100, rows_per_slot=3,
                         n_q_heads=Hq, n_kv_heads=Hkv, k_cells=k, chunk_cells=64, page_cells=page_cells,
                         v_bits=v_bits, block_cells=B, bias_prob=0.05)
    run_window_and_check(case)


def test_window_many_rows_two_pools():
    """20 rows (three 8-row n-tiles) over two pools in one call."""
    case = W.decode_case(name="wmany", seed=77, fills=[2000, 1500], capacity=2048, rows_per_slot=10,
                         n_q_heads=16, n_kv_heads=8, k_cells=256, chunk_cells=64, page_cells=256,
                         bias_prob=0.05)
    run_window_and_check(case)


def test_window_pools_of_mixed_v_formats():
    """An int8-V pool and a 4-bit-V pool in one call: the attention takes the kernel whose warps
    share sub-tiles, which reads each pool in its own format."""
    case = W.decode_case(name="wmixv", seed=55, fills=[1500, 1200], capacity=1536, rows_per_slot=3,
                         n_q_heads=8, n_kv_heads=2, k_cells=256, chunk_cells=64, page_cells=256, bias_prob=0.05)
    rng = np.random.default_rng(56)
    pool4 = W.make_pool(rng, capacity=1536, n_filled=1200, n_kv_heads=2, page_cells=256, v_bits=4, bias_prob=0.05)
    run_window_and_check(dataclasses.replace(case, pools=[case.pools[0], pool4]))


def test_window_4bit_k_with_int8_v():
    """4-bit K (32-dim K-scale groups) with int8 V."""
    case = W.decode_case(name="wk4v8", seed=57, fills=[1800], capacity=1900, rows_per_slot=4, n_q_heads=12,
                         n_kv_heads=2, k_cells=384, chunk_cells=64, page_cells=128, v_bits=8, k_bits=4,
                         bias_prob=0.05)
    run_window_and_check(case)


def test_window_max_rows():
    """QSA_MAX_DECODE_ROWS (32) rows over two pools: four 8-row n-tiles in the block scores."""
    case = W.decode_case(name="wmax", seed=32, fills=[3000, 2600], capacity=3072, rows_per_slot=16,
                         n_q_heads=16, n_kv_heads=4, k_cells=512, chunk_cells=64, page_cells=256, bias_prob=0.05)
    run_window_and_check(case)


def test_window_many_waves_of_blocks_two_pools():
    """1,250 32-cell blocks over two pools (two waves and more of block-score CTAs) and 12 rows (two 8-row
    n-tiles, one q-fragment load per m-tile)."""
    case = W.decode_case(name="wwaves", seed=91, fills=[25000, 15000], capacity=25600, rows_per_slot=6,
                         n_q_heads=16, n_kv_heads=4, k_cells=512, chunk_cells=64, page_cells=256,
                         block_cells=32, bias_prob=0.05)
    run_window_and_check(case)


def test_window_rows_with_masked_cells():
    """Rows early in the context: selected cells past a row's position are masked; splits whose cells are
    all masked are empty and carry no weight in the merge."""
    case = W.decode_case(name="wmasked", seed=5, fills=[900, 1500], capacity=2048, rows_per_slot=2,
                         n_q_heads=12, n_kv_heads=2, k_cells=512, chunk_cells=64, page_cells=128,
                         row_pos=[100, 899, 0, 1499], bias_prob=0.05)
    run_window_and_check(case)


def test_window_empty_selection():
    case = W.decode_case(name="wk0", seed=9, fills=[500], capacity=512, rows_per_slot=2, n_q_heads=4,
                         n_kv_heads=1, k_cells=0, chunk_cells=64, page_cells=64, n_chunks=2)
    win, q, row_pos = upload_case(case)
    win.out.fill_(float("nan"))
    win.run_window(q, row_pos)
    torch.cuda.synchronize()
    assert win.n_sel.cpu().tolist() == [0, 0]
    assert torch.all(win.out == 0) and torch.all(torch.isinf(win.lse)) and torch.all(win.lse < 0)


def test_window_deterministic_and_reusable_workspace():
    """Three calls on one workspace give the same bits, and the
    result matches the four separate calls within the gate."""
    case = W.verify_window()
    win, q, row_pos = upload_case(case)
    outs = []
    for _ in range(3):
        win.run_window(q, row_pos)
        torch.cuda.synchronize()
        outs.append((win.scores.clone(), win.ids.clone(), win.n_sel.clone(), win.out.clone(), win.lse.clone()))
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a, b)
    win.run(q, row_pos)
    torch.cuda.synchronize()
    assert_close(outs[0][3].cpu().numpy(), win.out.cpu().numpy(), "window vs separate calls")


def test_window_replays_from_a_cuda_graph():
    """The window's five chained launches (programmatic dependent launch edges included) captured in
    one CUDA graph: a replay gives the bits of a direct call, and a replay after new q is written into
    the captured buffer gives the bits of a direct call with that q."""
    case = W.verify_window()
    win, q, row_pos = upload_case(case)
    win.run_window(q, row_pos)
    torch.cuda.synchronize()
    direct = [t.clone() for t in (win.scores, win.ids, win.n_sel, win.out, win.lse)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        win.run_window(q, row_pos)
    for t in (win.scores, win.out, win.lse):
        t.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(direct, (win.scores, win.ids, win.n_sel, win.out, win.lse)):
        assert torch.equal(a, b)
    q2 = torch.from_numpy(np.random.default_rng(7).standard_normal(tuple(q.shape)).astype(np.float32)).cuda()
    q.copy_(q2)
    graph.replay()
    torch.cuda.synchronize()
    replayed = [t.clone() for t in (win.scores, win.ids, win.n_sel, win.out, win.lse)]
    win.run_window(q2, row_pos)
    torch.cuda.synchronize()
    for a, b in zip(replayed, (win.scores, win.ids, win.n_sel, win.out, win.lse)):
        assert torch.equal(a, b)
    assert not torch.equal(replayed[3], direct[3])


def test_window_refuses_small_workspace():
    case = W.tiny_dense_decode()
    win, q, row_pos = upload_case(case)
    need = qsa.load().qsa_decode_window_workspace_bytes(case.n_rows, case.n_q_heads, case.pools[0].n_kv_heads,
                                                        case.k_cells)
    assert need > 0
    win._ws = torch.empty((need - 256,), dtype=torch.uint8, device="cuda")
    with pytest.raises(qsa.QsaError) as e:
        win.run_window(q, row_pos)
    assert e.value.status == qsa.QSA_ERR_SCRATCH


@pytest.mark.gpu
@pytest.mark.parametrize("sums", [False, True])
def test_window_with_page_locked_host_buffers(sums):
    """qsa_decode_window_host (q, row positions, out and lse in page-locked host memory, staged by the
    window's first launch) gives the device-buffer call's results bit for bit, on a two-pool ragged
    window, with scores from the codes and from block summaries; pageable host tensors and device
    tensors in the host slots are refused before anything runs."""
    case = W.decode_case(name="host", seed=77, fills=[1000, 3333], capacity=4096, rows_per_slot=2, n_q_heads=12,
                         n_kv_heads=2, k_cells=512, chunk_cells=64)
    dev = torch.device("cuda")
    pools = [qsa.DevicePool.upload(p, dev) for p in case.pools]
    if sums:
        pools = [p.keep_block_sums() for p in pools]
    win = qsa.DecodeWindow(pools, case.row_pool, case.n_q_heads, case.block_cells, case.k_cells, case.chunk_cells,
                           case.n_chunks)
    q = torch.from_numpy(case.q).to(dev)
    pos = torch.from_numpy(case.row_pos.astype(np.int32)).to(dev)
    win.run_window(q, pos)
    torch.cuda.synchronize()
    out_d, lse_d, ids_d = win.out.cpu(), win.lse.cpu(), win.ids.cpu()
    q_h = torch.from_numpy(np.ascontiguousarray(case.q)).pin_memory()
    pos_h = torch.from_numpy(case.row_pos.astype(np.int32)).pin_memory()
    out_h = torch.full(tuple(win.out.shape), float("nan")).pin_memory()
    lse_h = torch.full(tuple(win.lse.shape), float("nan")).pin_memory()
    win.ids.zero_()
    win.run_window_host(q_h, pos_h, out_h, lse_h)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d) and torch.equal(lse_h, lse_d) and torch.equal(win.ids.cpu(), ids_d)
    # refusals: a pageable q, a device out
    lib = qsa.load()
    args = list(win._window_args(win.out, win.out, None))
    args[3], args[4], args[13], args[14] = torch.from_numpy(np.ascontiguousarray(case.q)).data_ptr(), \
        pos_h.data_ptr(), out_h.data_ptr(), lse_h.data_ptr()
    assert lib.qsa_decode_window_host(*args) == qsa.QSA_ERR_ARG
    args[3], args[13] = q_h.data_ptr(), win.out.data_ptr()
    assert lib.qsa_decode_window_host(*args) == qsa.QSA_ERR_ARG
