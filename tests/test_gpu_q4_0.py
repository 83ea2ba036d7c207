"""GPU parity of the q4_0 KV layout (4-bit K and V, one scale per 32 dims) against the oracle,
through the C ABI: the one-call decode window (block scores on 4-bit K, top-k, split attention,
merge), the prompt path and the append.  Gates as for the int8 layouts: ids bit-exact given the
GPU's own fp32 scores, scores / out / lse within max |gpu - oracle| / max |oracle| <= 1e-5."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_selection_attention_gb300 as qsa
import workloads as W
from _parity import assert_close, run_window_and_check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fill,page_cells,Hq,Hkv,k,B,rows", [
    (1000, 128, 6, 2, 256, 64, 3),       # ragged last block
    (3000, 256, 24, 4, 512, 64, 5),      # the verify window's heads and rows
    (2000, 256, 16, 8, 256, 32, 3),      # 32-cell blocks, 8 KV heads
    (2000, 256, 32, 4, 512, 128, 2),     # 128-cell blocks, 8 q heads per KV head
    (1500, 256, 16, 4, 384, 64, 6),      # 12 rows over two pools: two 8-row n-tiles
])
def test_q4_0_window(fill, page_cells, Hq, Hkv, k, B, rows):
    fills = [fill] if rows != 6 else [fill, fill - 300]
    case = W.decode_case(name="q40", seed=fill + k + B + rows, fills=fills, capacity=fill + 100,
                         rows_per_slot=rows, n_q_heads=Hq, n_kv_heads=Hkv, k_cells=k, chunk_cells=64,
                         page_cells=page_cells, v_bits=4, k_bits=4, block_cells=B, bias_prob=0.05)
    run_window_and_check(case)


def test_q4_0_window_verify_size():
    """The verify window's shape (5 rows, 24/4 heads, 32,768 cells, top-k 4,096) in the q4_0 layout."""
    case = W.decode_case(name="q40v", seed=11, fills=[32768], capacity=32768, rows_per_slot=5, n_q_heads=24,
                         n_kv_heads=4, k_cells=4096, chunk_cells=64, v_bits=4, k_bits=4, bias_prob=0.05)
    run_window_and_check(case)


@pytest.mark.parametrize("n_ctx,n_q,Hq,Hkv,page_cells", [
    (700, 150, 24, 4, 256),
    (2000, 300, 8, 2, 64),      # ranges of a cut unit
])
def test_q4_0_prompt(n_ctx, n_q, Hq, Hkv, page_cells):
    case = W.prompt_case(name="q40p", seed=n_ctx + n_q, n_ctx=n_ctx, n_q=n_q, n_q_heads=Hq, n_kv_heads=Hkv,
                         v_bits=4, k_bits=4, page_cells=page_cells, capacity=n_ctx + 64)
    pool = qsa.DevicePool.upload(case.pool)
    i0, n, pos0 = case.calls[0]
    q = torch.from_numpy(case.q).cuda()
    out = torch.full((n, Hq, 128), float("nan"), device="cuda")
    lse = torch.full((n, Hq), float("nan"), device="cuda")
    qsa.prompt_attn(pool, q, pos0, out, lse)
    torch.cuda.synchronize()
    assert qsa.get_device_error() == 0
    ref_out, ref_lse = O.prompt_attention(case.pool, case.q, pos0)
    assert_close(out.cpu().numpy(), ref_out, "out")
    assert_close(lse.cpu().numpy(), ref_lse, "lse")


def test_q4_0_append_bit_exact():
    rng = np.random.default_rng(41)
    pool = W.make_pool(rng, capacity=1024, n_filled=300, n_kv_heads=4, page_cells=256, v_bits=4, k_bits=4)
    k = (rng.standard_normal((200, 4, 128)) * 3).astype(np.float32)
    v = (rng.standard_normal((200, 4, 128)) * 3).astype(np.float32)
    k[0, 0, 32:64] = 0.0
    ref = O.append_cells(pool, k, v, 300)
    dp = qsa.DevicePool.upload(pool)
    qsa.kv_append(dp, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), 300)
    torch.cuda.synchronize()
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        a = getattr(dp, name).cpu().numpy()
        assert np.array_equal(a.view(np.uint8), getattr(ref, name).view(np.uint8)), name
