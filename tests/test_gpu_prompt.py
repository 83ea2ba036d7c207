"""GPU parity of the tensor-core prompt attention against the FP64 oracle,
through the C ABI: small ragged cases in full, the int8 prompt chunk on every
row and the four K8V4 calls on rows spread over each (the oracle spread over
the host's cores), codes of
-128, the cross-path identity with decode, and the
bounded-wait error path (a wait limit of 0 makes the kernel give up at its
first wait, report through the device error word and leave the context
usable; no fault, trap or hang is involved)."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_selection_attention_gb300 as qsa
import workloads as W
from _parity import assert_close, report, row_stats
from oracle import parallel as OP

pytestmark = pytest.mark.gpu


def run_prompt(case, call):
    i0, n, pos0 = call
    pool = qsa.DevicePool.upload(case.pool)
    q = torch.from_numpy(np.ascontiguousarray(case.q[i0:i0 + n])).cuda()
    out = torch.full((n, case.n_q_heads, 128), float("nan"), device="cuda")
    lse = torch.full((n, case.n_q_heads), float("nan"), device="cuda")
    qsa.prompt_attn(pool, q, pos0, out, lse)
    torch.cuda.synchronize()
    assert qsa.get_device_error() == 0
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("n_ctx,n_q,Hq,Hkv,v_bits,page_cells", [
    (700, 150, 24, 4, 8, 256),     # G = 6: 21 queries per CTA, ragged last CTA and tile
    (513, 40, 8, 2, 4, 64),        # 4-bit V, G = 4
    (64, 64, 2, 1, 8, 64),         # one tile, queries from position 0
    (1000, 37, 6, 6, 8, 128),      # G = 1
    (333, 333, 16, 1, 4, 64),      # G = 16, whole context is the prompt
    (300, 12, 128, 1, 8, 64),      # G = 128 (the largest group): one query per CTA
    # fewer units than SMs: each unit cut into tile ranges merged by log-sum-exp
    (2000, 300, 2, 1, 8, 64),      # G = 2: 5 units of 27..32 tiles, 3 ranges each (ragged range ends)
    (3000, 64, 8, 2, 4, 128),      # 4-bit V, G = 4: 4 units of 47 tiles, 5 ranges each
    (1500, 1500, 4, 4, 8, 64),     # queries from position 0: units from 1 to 24 tiles, cut by the shortest
])
def test_small_prompt_full(n_ctx, n_q, Hq, Hkv, v_bits, page_cells):
    case = W.prompt_case(name="p", seed=n_ctx + n_q, n_ctx=n_ctx, n_q=n_q, n_q_heads=Hq, n_kv_heads=Hkv,
                         v_bits=v_bits, page_cells=page_cells, capacity=n_ctx + 200)
    out, lse = run_prompt(case, case.calls[0])
    ref_out, ref_lse = O.prompt_attention(case.pool, case.q, case.calls[0][2])
    assert_close(out, ref_out, "out")
    assert_close(lse, ref_lse, "lse")


def test_prompt_scratch_covers_images_and_ranges():
    """The scratch of the bench's prompt call: header, one image per tile and KV head, and a whole
    number of 66,560-byte partial-range records (the range count follows the SM count)."""
    case = W.prompt_int8()
    pool = qsa.DevicePool.upload(case.pool)
    i0, n, pos0 = case.calls[0]
    need = qsa.prompt_scratch_bytes(pool, n, pos0, case.n_q_heads)
    images = 256 + case.pool.n_kv_heads * ((pos0 + n - 1) // 64 + 1) * 65536
    assert need >= images and (need - images) % 66560 == 0


def test_prompt_heads_with_far_apart_v_scales():
    """KV heads whose V scales differ by 2^10 in either direction, and one tile of near-zero V scales:
    the V-scale exponent is taken per head and only shifts the reference of p."""
    case = W.prompt_case(name="vs", seed=31, n_ctx=1100, n_q=70, n_q_heads=12, n_kv_heads=3, page_cells=128,
                         capacity=1280)
    case.pool.v_scales[:, 1] *= 1024.0
    case.pool.v_scales[:, 2] /= 1024.0
    phys0 = int(case.pool.page_table[3])
    case.pool.v_scales[phys0, 0, :64] *= 1e-6
    out, lse = run_prompt(case, case.calls[0])
    ref_out, ref_lse = O.prompt_attention(case.pool, case.q, case.calls[0][2])
    assert_close(out, ref_out, "out")
    assert_close(lse, ref_lse, "lse")


def check_rows(name, builder, call_index, rows=None):
    """The given rows (default: every row) of one call of a named prompt workload against the oracle,
    element-wise at the gate, with the row-wise error reported; the rest of the call must be finite."""
    case = getattr(W, builder)()
    out, lse = run_prompt(case, case.calls[call_index])
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    ref_out, ref_lse = OP.prompt_call(builder, {}, call_index, rows=rows)
    if rows is not None:
        out, lse = out[rows], lse[rows]
    e_out = assert_close(out, ref_out, f"{name} out")
    e_lse = assert_close(lse, ref_lse, f"{name} lse")
    mean_row, max_row = row_stats(out, ref_out)
    report(name, rows=int(out.shape[0]), heads=int(out.shape[1]), max_rel_out=e_out, max_rel_lse=e_lse,
           mean_row_rel_out=mean_row, max_row_rel_out=max_row)


def test_prompt_int8_full_size_all_rows():
    """2,048 queries against 32,768 cells, 24/4 heads (the prompt workload of the bench), every row."""
    check_rows("prompt int8 2048 x 32768", "prompt_int8", 0)


@pytest.mark.parametrize("call_index", [0, 1, 2, 3])
def test_prompt_k8v4_every_call(call_index):
    """8,192 queries against 131,072 cells (32/8 heads, int8 K, 4-bit V) in four calls of 2,048: each
    call on 64 rows spread over it (its first and last row among them), every head.  (Every row of a
    call needs about 4.4e12 FP64 multiply-adds in the oracle, longer than a test run allows.)"""
    rows = sorted(set(np.linspace(0, 2047, 62).astype(int).tolist()) | {1, 2046})
    check_rows(f"prompt k8v4 call {call_index}", "prompt_k8v4", call_index, rows=rows)


@pytest.mark.parametrize("v_bits", [8, 4])
def test_prompt_codes_of_minus_128(v_bits):
    """int8 codes drawn in [-128, 127] (K, and V when int8): the code without a positive twin goes
    through the exact conversions like every other."""
    case = W.prompt_case(name="m128", seed=128 + v_bits, n_ctx=900, n_q=120, n_q_heads=12, n_kv_heads=3,
                         v_bits=v_bits, page_cells=128, capacity=1024, code_lo=-128)
    assert (case.pool.k_codes == -128).any()
    out, lse = run_prompt(case, case.calls[0])
    ref_out, ref_lse = O.prompt_attention(case.pool, case.q, case.calls[0][2])
    assert_close(out, ref_out, "out")
    assert_close(lse, ref_lse, "lse")


def test_prompt_row_equals_decode_with_all_cells():
    """Cross-path: a prompt row at position p equals decode with top-k = all cells at p."""
    case = W.prompt_case(name="x", seed=21, n_ctx=640, n_q=5, n_q_heads=24, n_kv_heads=4)
    out, lse = run_prompt(case, case.calls[0])
    dcase = W.DecodeCase("x", [case.pool], np.zeros(5, np.int32), case.q, np.arange(635, 640, dtype=np.int32),
                         24, 64, 640, 64, 10, 10)
    from _parity import upload_case
    win, q, row_pos = upload_case(dcase)
    win.run(q, row_pos)
    torch.cuda.synchronize()
    assert_close(out, win.out.cpu().numpy(), "prompt vs decode out")
    assert_close(lse, win.lse.cpu().numpy(), "prompt vs decode lse")


def test_prompt_deterministic():
    case = W.prompt_case(name="d", seed=2, n_ctx=900, n_q=100, n_q_heads=24, n_kv_heads=4)
    a = run_prompt(case, case.calls[0])
    b = run_prompt(case, case.calls[0])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bounded_wait_reports_and_context_survives():
    case = W.prompt_case(name="w", seed=4, n_ctx=300, n_q=30, n_q_heads=8, n_kv_heads=2)
    pool = qsa.DevicePool.upload(case.pool)
    q = torch.from_numpy(case.q).cuda()
    out = torch.zeros((30, 8, 128), device="cuda")
    try:
        qsa.set_wait_limit_ns(0)
        qsa.prompt_attn(pool, q, case.calls[0][2], out)
        assert qsa.get_device_error() == 1
    finally:
        qsa.set_wait_limit_ns(2_000_000_000)
    assert qsa.get_device_error() == 0          # read-and-clear
    out2, lse2 = run_prompt(case, case.calls[0])  # the context is still usable
    ref_out, _ = O.prompt_attention(case.pool, case.q, case.calls[0][2])
    assert_close(out2, ref_out, "out after error path")
