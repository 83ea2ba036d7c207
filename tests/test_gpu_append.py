"""GPU parity of qsa_kv_append (quantise-on-append of new K/V cells) against the
oracle, through the C ABI: the codes and scales it writes are bit-exact (the
quantiser decides integers in fp32 on both sides), the cells it does not
append are untouched, and attention over appended cells matches the oracle on
the oracle's appended pool."""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_selection_attention_gb300 as qsa
import workloads as W
from _parity import assert_close

pytestmark = pytest.mark.gpu


def new_rows(rng, n, Hkv):
    """Rows of every kind the quantiser must handle: wide magnitudes, an all-zero group, exact
    ties (values on half steps of a scale-1 group) and single spikes."""
    k = (rng.standard_normal((n, Hkv, 128)) * 10.0 ** rng.uniform(-3, 3, size=(n, Hkv, 1))).astype(np.float32)
    v = (rng.standard_normal((n, Hkv, 128)) * 10.0 ** rng.uniform(-3, 3, size=(n, Hkv, 1))).astype(np.float32)
    k[0, 0, :64] = 0.0                                            # zero group
    v[0, 0, 32:64] = 0.0
    if n > 1:
        k[1, 0, :64] = np.arange(64, dtype=np.float32) * 0.5 - 16.0   # half steps: ties to even
        k[1, 0, 63] = 127.0                                           # scale exactly 1
        v[1, 0, :32] = np.arange(32, dtype=np.float32) * 0.25 - 4.0
        v[1, 0, 31] = 7.0                                             # 4-bit: scale exactly 1 (int8: 7 / 127)
    if n > 2:
        k[2, -1, 70] = 1e6                                            # one spike
    return k, v


def device_pool_arrays(dp):
    return [t.cpu().numpy() for t in (dp.k_codes, dp.v_codes, dp.k_scales, dp.v_scales)]


@pytest.mark.parametrize("v_bits,Hkv,page_cells,first,n", [
    (8, 4, 256, 700, 300),     # across a page boundary
    (4, 8, 64, 0, 200),        # 4-bit V, from the first cell, many pages
    (8, 1, 128, 1023, 1),      # one cell, the last of the capacity
    (4, 2, 256, 5, 2048),      # a prompt chunk's worth
])
def test_append_bit_exact(v_bits, Hkv, page_cells, first, n):
    rng = np.random.default_rng(first + n + v_bits)
    capacity = max(1024, first + n)
    pool = W.make_pool(rng, capacity=capacity, n_filled=first, n_kv_heads=Hkv, page_cells=page_cells, v_bits=v_bits)
    k, v = new_rows(rng, n, Hkv)
    ref = O.append_cells(pool, k, v, first)
    dp = qsa.DevicePool.upload(pool)
    qsa.kv_append(dp, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), first)
    torch.cuda.synchronize()
    assert dp.n_filled == first + n
    got = device_pool_arrays(dp)
    for name, a, b in zip(("k_codes", "v_codes", "k_scales", "v_scales"), got,
                          (ref.k_codes, ref.v_codes, ref.k_scales, ref.v_scales)):
        # stale cells carry NaN scales in both pools: compare the bits
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), name


def test_append_near_ties_and_tiny_scales():
    """Values whose quotient by the group scale lies within a few ulps of a half-integer (where a
    product with the reciprocal and the rounded quotient could round apart), and groups so small that
    their scales are subnormal: codes still bit-exact."""
    rng = np.random.default_rng(77)
    n, Hkv = 512, 2
    pool = W.make_pool(rng, capacity=1024, n_filled=0, n_kv_heads=Hkv, page_cells=256, v_bits=4)
    k = np.zeros((n, Hkv, 128), np.float32)
    v = np.zeros((n, Hkv, 128), np.float32)
    for i in range(n):
        for h in range(Hkv):
            for x, grp, qmax in ((k, 64, 127), (v, 32, 7)):
                for g0 in range(0, 128, grp):
                    s = np.float32(10.0 ** rng.uniform(-30, 3))
                    if i % 7 == 0:
                        s = np.float32(10.0 ** rng.uniform(-44, -38))     # subnormal scales
                    steps = rng.integers(-qmax, qmax, size=grp) + 0.5
                    delta = rng.choice([0.0, 2.0 ** -22, -(2.0 ** -22), 2.0 ** -18, -(2.0 ** -18), 2.0 ** -15], size=grp)
                    vals = ((steps + delta) * np.float64(s)).astype(np.float32)
                    vals[int(rng.integers(grp))] = np.float32(qmax * np.float64(s))
                    x[i, h, g0:g0 + grp] = vals
    ref = O.append_cells(pool, k, v, 0)
    dp = qsa.DevicePool.upload(pool)
    qsa.kv_append(dp, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), 0)
    torch.cuda.synchronize()
    got = device_pool_arrays(dp)
    for name, a, b in zip(("k_codes", "v_codes", "k_scales", "v_scales"), got,
                          (ref.k_codes, ref.v_codes, ref.k_scales, ref.v_scales)):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), name


def test_append_then_prompt_matches_oracle():
    """A prompt chunk appended to a pool and then attended (prompt path over the new cells) equals
    the oracle's attention over the oracle's appended pool."""
    rng = np.random.default_rng(12)
    Hkv, Hq, first, n = 4, 24, 1500, 500
    pool = W.make_pool(rng, capacity=2048, n_filled=first, n_kv_heads=Hkv, page_cells=256)
    k, v = new_rows(rng, n, Hkv)
    k = np.clip(k, -50, 50)   # keep the logits in the range of the workloads'
    v = np.clip(v, -50, 50)
    q = rng.standard_normal((n, Hq, 128)).astype(np.float32)
    dp = qsa.DevicePool.upload(pool)
    qsa.kv_append(dp, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), first)
    out = torch.empty((n, Hq, 128), device="cuda")
    lse = torch.empty((n, Hq), device="cuda")
    qsa.prompt_attn(dp, torch.from_numpy(q).cuda(), first, out, lse)
    torch.cuda.synchronize()
    assert qsa.get_device_error() == 0
    ref_pool = O.append_cells(pool, k, v, first)
    rows = [0, 1, 7, 250, n - 1]
    ref_out, ref_lse = O.prompt_attention(ref_pool, q, first, rows=rows)
    assert_close(out.cpu().numpy()[rows], ref_out, "out")
    assert_close(lse.cpu().numpy()[rows], ref_lse, "lse")


def test_append_refuses_past_capacity():
    rng = np.random.default_rng(1)
    pool = W.make_pool(rng, capacity=256, n_filled=200, n_kv_heads=1, page_cells=256)
    dp = qsa.DevicePool.upload(pool)
    k = torch.zeros((100, 1, 128), device="cuda")
    with pytest.raises(qsa.QsaError) as e:
        qsa.kv_append(dp, k, k, 200)
    assert e.value.status == qsa.QSA_ERR_ARG
    assert dp.n_filled == 200
