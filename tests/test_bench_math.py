"""The bench's metric arithmetic (CPU): algorithmic bytes of the decode windows and the prompt's
FLOP counts, checked against values computed independently from the workload definitions (cell
counts x bytes per cell, closed-form pair counts), so that a wrong row size, a missed head or a
dropped causal term in the metric fails here."""
import numpy as np

import bench
import workloads as W


def test_block_score_bytes_of_the_decode_windows():
    # every filled K code (128 B) and its two fp32 scales (8 B) per (cell, KV head)
    for case, want in ((W.verify_window(), 32768 * 4 * 136), (W.batched_long_context(), (65536 + 131072) * 4 * 136),
                       (W.tiny_dense_decode(), 1024 * 1 * 136)):
        a1, _ = bench.algorithmic_bytes(case, [np.zeros(0, np.int32)] * case.n_rows, np.zeros(case.n_rows, np.int32))
        assert a1 == want
    assert (W.verify_window().n_rows, 32768 * 4 * 136) == (5, 17_825_792)
    assert (65536 + 131072) * 4 * 136 == 106_954_752


def test_attention_bytes_count_the_union_of_visible_selected_cells():
    case = W.verify_window()
    # rows share cells: the union is counted once per (cell, KV head), K and V rows with scales (272 B)
    ids = [np.arange(0, 4096, dtype=np.int32) for _ in range(case.n_rows)]
    ids[1] = np.arange(2048, 6144, dtype=np.int32)
    n_sel = np.full(case.n_rows, 4096, np.int32)
    _, a3 = bench.algorithmic_bytes(case, ids, n_sel)
    assert a3 == 6144 * 4 * 272
    # cells past a row's position are not read
    ids = [np.array([0, 1, 32767], np.int32)] + [np.zeros(0, np.int32)] * (case.n_rows - 1)
    n_sel = np.array([3] + [0] * (case.n_rows - 1), np.int32)
    _, a3 = bench.algorithmic_bytes(case, ids, n_sel)
    assert a3 == (3 if 32767 <= case.row_pos[0] else 2) * 4 * 272
    # 4-bit V rows: 64 code bytes and four fp32 scales
    small = W.prompt_case(name="k8v4", seed=1, n_ctx=64, n_q=1, n_q_heads=2, n_kv_heads=1, v_bits=4)
    assert bench.row_bytes(small.pool) == (136, 80)


def test_prompt_flop_counts_of_the_prompt_workloads():
    case = W.prompt_int8()
    issued, logical = bench.prompt_flops(case, case.calls[0])
    pairs = sum(30721 + i for i in range(2048)) * 24       # causal (query, cell) pairs x q heads
    assert pairs == 65_012_736 * 24
    assert logical == pairs * 2 * 2 * 128                 # two products, 2 x 128 FLOP each
    assert issued == 3 * logical                          # three fp16 parts per product
    assert abs(issued - 2.397e12) / 2.397e12 < 1e-3
    # the K8V4 prompt: four calls of 2,048 queries at 122,880.., 32 q heads (its shapes only)
    k8 = W.PromptCase("k8v4", None, None, [(i, 2048, 122880 + i) for i in range(0, 8192, 2048)], 32)
    total = sum(bench.prompt_flops(k8, c)[0] for c in k8.calls)
    assert abs(total - 5.112e13) / 5.112e13 < 1e-3
