"""Pins of the CPU oracle against facts other than itself: hand-worked fixtures,
closed forms, special cases that reduce to a library routine, invariants and
brute force on tiny inputs.  Each pin is chosen so that a plausible slip in
the oracle (a dropped term, a wrong index or sign, a swapped operand) fails."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle as O
import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def hand_pool(n_cells, n_kv_heads=1, v_bits=8, page_cells=64, capacity=None, seed=0):
    """A tiny pool with every scale 1.0 and zero codes; callers set codes."""
    capacity = capacity or n_cells
    n_pages = (capacity + page_cells - 1) // page_cells
    D = 128
    vg = 64 if v_bits == 8 else 32
    rng = np.random.default_rng(seed)
    table = rng.permutation(n_pages).astype(np.int32)
    vshape = (n_pages, n_kv_heads, page_cells, D if v_bits == 8 else D // 2)
    return W.Pool(
        k_codes=np.zeros((n_pages, n_kv_heads, page_cells, D), np.int8),
        v_codes=np.zeros(vshape, np.int8 if v_bits == 8 else np.uint8) + (0 if v_bits == 8 else 0x88),
        k_scales=np.ones((n_pages, n_kv_heads, page_cells, 2), np.float32),
        v_scales=np.ones((n_pages, n_kv_heads, page_cells, D // vg), np.float32),
        page_table=table, capacity=capacity, n_filled=n_cells, page_cells=page_cells,
        n_kv_heads=n_kv_heads, head_dim=D, v_bits=v_bits, v_group=vg)


def put(pool, arr_name, c, h, value):
    arr = getattr(pool, arr_name)
    arr[pool.page_table[c // pool.page_cells], h, c % pool.page_cells] = value


def get(pool, arr_name, c, h):
    arr = getattr(pool, arr_name)
    return arr[pool.page_table[c // pool.page_cells], h, c % pool.page_cells]


# ----------------------------------------------------------------- hand fixtures

def test_hand_two_cell_attention_and_merge():
    fx = json.load(open(os.path.join(GOLD, "hand_two_cell.json")))
    pool = hand_pool(2)
    k1 = np.zeros(128, np.int8)
    k1[0] = fx["k_code_cell1_dim0"]
    put(pool, "k_codes", 1, 0, k1)
    for c, v in enumerate(fx["v_code_dim0"]):
        row = np.zeros(128, np.int8)
        row[0] = v
        put(pool, "v_codes", c, 0, row)
    q = np.zeros((1, 128), np.float64)
    q[0, 0] = math.sqrt(128) * math.log(3)
    out, lse = O.attention(pool, q, 1, [0, 1])
    assert out[0, 0] == pytest.approx(fx["expect_out_dim0"], abs=1e-12)
    assert np.all(out[0, 1:] == 0)
    assert lse[0] == pytest.approx(math.log(4), abs=1e-12)
    m, l, o = O.chunk_partials(pool, q, 1, [0, 1], 1, 2)
    exp = [[0.0, 1.0, 4.0], [math.log(3), 1.0, 8.0]]
    for j in range(2):
        assert (m[0, j], l[0, j], o[0, j, 0]) == pytest.approx(tuple(exp[j]), abs=1e-12)
    out2, lse2 = O.merge_partials(m, l, o)
    assert out2[0, 0] == pytest.approx(7.0, abs=1e-12) and lse2[0] == pytest.approx(math.log(4), abs=1e-12)


def test_hand_topk_ties_and_signed_zero():
    fx = json.load(open(os.path.join(GOLD, "topk_ties.json")))
    scores = np.array([float(s) for s in fx["scores"]], np.float32)
    assert math.copysign(1.0, scores[1]) < 0  # -0.0 really is negative zero
    for k, want in fx["expect"].items():
        ids, n = O.topk_select(scores, len(scores), 1, int(k))
        assert list(ids) == want and n == len(want)


def test_hand_nibble_unpacking():
    fx = json.load(open(os.path.join(GOLD, "nibbles.json")))
    pool = hand_pool(1, v_bits=4)
    row = np.full(64, 0x88, np.uint8)
    row[:3] = fx["bytes"]
    put(pool, "v_codes", 0, 0, row)
    V = O.dequantise_v(pool, 0, [0])
    assert list(V[0, :6]) == fx["expect_codes"]
    assert np.all(V[0, 6:] == 0)


# ----------------------------------------------------------------- dequantise

def test_dequantise_scale_groups_and_paging():
    rng = np.random.default_rng(5)
    pool = W.make_pool(rng, capacity=512, n_filled=300, n_kv_heads=2, page_cells=128)
    # A cell's group-1 scale must hit dims 64..127 only, and the page table must be followed.
    c, h = 200, 1
    codes = get(pool, "k_codes", c, h).astype(np.float64)
    ks = get(pool, "k_scales", c, h).astype(np.float64)
    K = O.dequantise_k(pool, h, [c])[0]
    assert np.array_equal(K[:64], codes[:64] * ks[0]) and np.array_equal(K[64:], codes[64:] * ks[1])
    # Physical layout invariance: re-permute pages and the table together.
    perm = rng.permutation(pool.n_pages)
    moved = W.Pool(**{**pool.__dict__})
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        src = getattr(pool, name)
        dst = np.empty_like(src)
        dst[perm] = src
        setattr(moved, name, dst)
    moved.page_table = perm[pool.page_table].astype(np.int32)
    cells = np.arange(0, 300, 7)
    for hh in range(2):
        assert np.array_equal(O.dequantise_k(pool, hh, cells), O.dequantise_k(moved, hh, cells))
        assert np.array_equal(O.dequantise_v(pool, hh, cells), O.dequantise_v(moved, hh, cells))


def test_dequantise_v4_group_of_32():
    pool = hand_pool(1, v_bits=4)
    row = np.full(64, 0x99, np.uint8)      # every code = +1
    put(pool, "v_codes", 0, 0, row)
    put(pool, "v_scales", 0, 0, np.array([1, 2, 3, 4], np.float32))
    V = O.dequantise_v(pool, 0, [0])[0]
    assert list(V[::32]) == [1, 2, 3, 4] and np.all(V[:32] == 1) and np.all(V[96:] == 4)


# ----------------------------------------------------------------- block scores

def test_block_score_closed_form_constant_k():
    """K constant u within the block => S = sum_h (sum_{g in G(h)} q_g) . u_h / sqrt(D)."""
    Hkv, Hq = 2, 6
    pool = hand_pool(100, n_kv_heads=Hkv)        # blocks of 64: one full, one ragged (36 cells)
    rng = np.random.default_rng(1)
    u = rng.integers(-20, 21, size=(Hkv, 128)).astype(np.int8)
    s = np.array([0.25, 0.5], np.float32)        # different group scales
    for c in range(100):
        for h in range(Hkv):
            put(pool, "k_codes", c, h, u[h])
            put(pool, "k_scales", c, h, s)
    q = rng.standard_normal((3, Hq, 128)).astype(np.float32)
    S = O.block_scores(pool, q, 64)
    assert S.shape == (3, 2)
    G = Hq // Hkv
    for t in range(3):
        want = 0.0
        for h in range(Hkv):
            qs = q[t, h * G:(h + 1) * G].astype(np.float64).sum(0)
            uu = u[h].astype(np.float64) * np.repeat(s.astype(np.float64), 64)
            want += qs @ uu / math.sqrt(128)
        assert S[t, 0] == pytest.approx(want, rel=1e-12)
        assert S[t, 1] == pytest.approx(want, rel=1e-12)   # mean, not sum, over the ragged block


def test_block_score_is_mean_of_logits_and_head_mapped():
    """One nonzero cell in a block of n_b => S = logit / n_b, only through its KV head."""
    Hkv, Hq = 2, 4
    pool = hand_pool(64 + 10, n_kv_heads=Hkv)
    kc = np.zeros(128, np.int8)
    kc[5] = 3
    put(pool, "k_codes", 70, 1, kc)              # cell 70: block 1 (10 cells), KV head 1
    q = np.zeros((1, Hq, 128), np.float32)
    q[0, 3, 5] = 2.0                              # q head 3 -> KV head 1
    q[0, 0, 5] = 100.0                            # q head 0 -> KV head 0: must not touch head 1
    S = O.block_scores(pool, q, 64)
    assert S[0, 0] == 0.0
    assert S[0, 1] == pytest.approx(2.0 * 3 / math.sqrt(128) / 10, rel=1e-12)


def test_block_score_linear_in_q():
    case = W.decode_case(name="t", seed=11, fills=[300], capacity=512, rows_per_slot=2, n_q_heads=4,
                         n_kv_heads=2, k_cells=128, chunk_cells=64, page_cells=128)
    pool = case.pools[0]
    q1, q2 = case.q[:1], case.q[1:]
    S1, S2 = O.block_scores(pool, q1, 64), O.block_scores(pool, q2, 64)
    S12 = O.block_scores(pool, (q1.astype(np.float64) + q2), 64)
    assert np.allclose(S12, S1 + S2, rtol=0, atol=1e-12)


# ----------------------------------------------------------------- top-k

def _rank_select(scores, nb, k_blocks):
    """Independent definition: block b is chosen iff fewer than k_blocks blocks rank above it,
    where b' ranks above b iff key(b') > key(b), or equal keys and b' < b."""
    keys = [O.score_key(scores[b]) for b in range(nb)]
    out = []
    for b in range(nb):
        above = sum(1 for c in range(nb) if keys[c] > keys[b] or (keys[c] == keys[b] and c < b))
        if above < k_blocks:
            out.append(b)
    return out


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(2)
    vals = np.array([-np.inf, -2, -1, -0.0, 0.0, 1, 2, np.inf, np.nan], np.float32)
    for trial in range(300):
        nb = int(rng.integers(1, 13))
        B = int(rng.choice([1, 2, 4]))
        n_filled = (nb - 1) * B + int(rng.integers(1, B + 1))
        scores = rng.choice(vals, size=nb) if trial % 2 else rng.standard_normal(nb).astype(np.float32)
        for kb in range(0, nb + 2):
            ids, n = O.topk_select(scores, n_filled, B, kb * B)
            blocks = _rank_select(scores, nb, kb)
            want = [c for b in blocks for c in range(b * B, min((b + 1) * B, n_filled))]
            assert list(ids) == want and n == len(want)


def test_topk_matches_stable_argsort_without_specials():
    rng = np.random.default_rng(3)
    for _ in range(50):
        nb = int(rng.integers(1, 200))
        scores = rng.integers(-5, 6, size=nb).astype(np.float32)  # many ties
        kb = int(rng.integers(0, nb + 1))
        ids, _ = O.topk_select(scores, nb, 1, kb)
        want = np.sort(np.argsort(-scores.astype(np.float64), kind="stable")[:kb])
        assert list(ids) == list(want)


def test_score_key_order():
    xs = np.array([-np.inf, -3.5, -1e-30, -0.0, 0.0, 1e-45, 1.0, 3e38, np.inf], np.float32)
    keys = [O.score_key(x) for x in xs]
    assert keys[3] == keys[4]
    strict = [k for i, k in enumerate(keys) if i != 3]
    assert strict == sorted(strict) and len(set(strict)) == len(strict)
    assert O.score_key(np.float32("nan")) == 0 < keys[0]
    assert O.score_key(-np.float32("nan")) == 0


def test_topk_rejects_k_not_multiple_of_block():
    with pytest.raises(ValueError):
        O.topk_select(np.zeros(4, np.float32), 256, 64, 100)


# ----------------------------------------------------------------- attention

def _small_case(seed=7, fill=700, Hq=6, Hkv=2, v_bits=8):
    return W.decode_case(name="t", seed=seed, fills=[fill], capacity=1024, rows_per_slot=3,
                         n_q_heads=Hq, n_kv_heads=Hkv, k_cells=(fill + 63) // 64 * 64, chunk_cells=64,
                         page_cells=128, v_bits=v_bits)


@pytest.mark.parametrize("v_bits", [8, 4])
def test_attention_matches_scipy_softmax(v_bits):
    case = _small_case(v_bits=v_bits)
    pool = case.pools[0]
    ids = np.arange(0, 700, 3)
    pos = 650
    out, lse = O.attention(pool, case.q[0], pos, ids)
    vis = ids[ids <= pos]
    for g in range(case.n_q_heads):
        h = g // 3
        K = O.dequantise_k(pool, h, vis)
        V = O.dequantise_v(pool, h, vis)
        z = np.einsum("cd,d->c", K, case.q[0, g].astype(np.float64)) / math.sqrt(128)
        assert lse[g] == pytest.approx(scipy.special.logsumexp(z), rel=1e-13)
        assert np.allclose(out[g], scipy.special.softmax(z) @ V, rtol=0, atol=1e-12)


def test_attention_special_cases():
    case = _small_case()
    pool = case.pools[0]
    ids = np.arange(100, 200)
    # q = 0: uniform weights -> mean of V; lse = ln |V_t|
    q0 = np.zeros((6, 128), np.float32)
    out, lse = O.attention(pool, q0, 150, ids)
    V = O.dequantise_v(pool, 1, np.arange(100, 151))
    assert np.allclose(out[4], V.mean(0), atol=1e-13) and lse[4] == pytest.approx(math.log(51))
    # a single visible cell -> exactly its V
    out, lse = O.attention(pool, case.q[0], 100, ids)
    assert np.array_equal(out[5], O.dequantise_v(pool, 1, [100])[0])
    # nothing visible -> 0 and -inf
    out, lse = O.attention(pool, case.q[0], 99, ids)
    assert np.all(out == 0) and np.all(lse == -np.inf)
    # identical q within a group -> identical outputs; different group -> different
    q = np.repeat(case.q[0, :1], 6, axis=0)
    out, _ = O.attention(pool, q, 699, ids)
    assert np.array_equal(out[0], out[2]) and not np.allclose(out[0], out[3])


def test_chunking_and_merge_do_not_change_the_result():
    case = _small_case()
    pool = case.pools[0]
    ids = np.sort(np.random.default_rng(4).choice(700, 333, replace=False))
    pos = 600
    ref_out, ref_lse = O.attention(pool, case.q[1], pos, ids)
    for C in (1, 7, 64, 256, 333, 1000):
        n = (len(ids) + C - 1) // C + 3          # extra chunks past the selection stay empty
        m, l, o = O.chunk_partials(pool, case.q[1], pos, ids, C, n)
        assert np.all(m[:, -3:] == -np.inf)
        out, lse = O.merge_partials(m, l, o)
        assert np.allclose(out, ref_out, rtol=0, atol=1e-12)
        assert np.allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_decode_with_all_cells_equals_prompt_row():
    """Top-k with k >= all cells reduces decode to dense attention, which is the prompt row."""
    case = _small_case(fill=640)
    pool = case.pools[0]
    res = O.decode_window(case)
    pos0 = 600
    pout, plse = O.prompt_attention(pool, case.q, pos0, rows=[0, 1, 2])
    for t in range(3):
        assert list(res["ids"][t]) == list(range(640))
        dout, dlse = O.attention(pool, case.q[t], pos0 + t, res["ids"][t])
        assert np.allclose(dout, pout[t], atol=1e-12) and np.allclose(dlse, plse[t], atol=1e-12)


def test_prompt_row_blocks_and_head_subsets_match_single_rows():
    """The prompt oracle's row blocks (causal mask per row inside a block) and head subsets give, row by
    row, the single-row attention over cells 0 .. position, computed without any mask."""
    case = _small_case(fill=640)
    pool = case.pools[0]
    pos0 = 590
    rows = [0, 3, 4, 9, 10, 11, 49]
    Hq = case.q.shape[1]
    heads = [1, 2, Hq - 1]
    q = np.concatenate([case.q] * 20)[:50]
    out, lse = O.prompt_attention(pool, q, pos0, rows=rows, heads=heads, row_block=3)
    for r, i in enumerate(rows):
        dout, dlse = O.attention(pool, q[i], pos0 + i, list(range(pos0 + i + 1)))
        for g in range(Hq):
            if g in heads:
                assert np.allclose(out[r, g], dout[g], rtol=0, atol=1e-12)
                assert abs(lse[r, g] - dlse[g]) <= 1e-12
            else:
                assert np.all(out[r, g] == 0.0) and lse[r, g] == -np.inf


@pytest.mark.parametrize("B", [64, 128])
def test_block_scores_from_block_summaries(B):
    """R3 is linear in K: the block score equals qbar . (the block's summed K rows) / (n_b sqrt(D)),
    summed over KV heads, with the block's 64-cell summaries added; a summary that dropped a scale or
    a cell, or a block score that dropped 1/n_b, fails it."""
    case = _small_case(fill=700)
    pool = case.pools[0]
    S = O.block_scores(pool, case.q, B)
    sums = O.block_summaries(pool, 64)
    Hq, Hkv = case.q.shape[1], pool.n_kv_heads
    G = Hq // Hkv
    for t in range(case.q.shape[0]):
        for b in range(S.shape[1]):
            n_b = min(B, pool.n_filled - b * B)
            kb = sums[b * B // 64:(b * B + n_b + 63) // 64].sum(axis=0)          # [Hkv, D]
            qbar = case.q[t].astype(np.float64).reshape(Hkv, G, -1).sum(axis=1)  # [Hkv, D]
            v = float((qbar * kb).sum()) / (n_b * np.sqrt(128.0))
            assert abs(v - S[t, b]) <= 1e-12 * max(1.0, abs(S[t, b]))


def test_stale_cells_are_never_read():
    """Cells past the fill carry NaN scales; the whole decode chain stays finite."""
    case = _small_case(fill=700)
    res = O.decode_window(case)
    assert all(np.isfinite(s).all() for s in res["scores"])
    assert np.isfinite(res["out"]).all() and np.isfinite(res["lse"]).all()


def test_workload_recipe():
    """The named workloads have the shapes and value ranges they state."""
    c = W.tiny_dense_decode()
    p = c.pools[0]
    assert c.q.shape == (1, 2, 128) and p.n_filled == 1024 and c.row_pos[0] == 1023
    assert p.k_codes.min() >= -127 and p.k_codes.max() <= 127
    fin = p.k_scales[np.isfinite(p.k_scales)]
    assert fin.min() >= 0.005 and fin.max() <= 0.02
    assert sorted(p.page_table) == list(range(p.n_pages))


# ---------------------------------------------------------------- append (reading R14)

def _group(head, n):
    x = np.zeros(n, np.float32)
    x[:len(head)] = head
    return x


def test_append_groups_worked_by_hand():
    """Hand-worked groups: absmax scale, ties to even (a round-half-away or a scale from the mean
    would change codes 2, 4, -2 or 126), zeros for an all-zero group."""
    g = json.load(open(os.path.join(GOLD, "append_quant.json")))
    for case in g["int8_groups"]:
        codes, scale = O.quantise_group(_group(case["x_head"], 64), 127)
        assert scale == np.float32(case["scale"])
        assert codes[:len(case["codes_head"])].tolist() == case["codes_head"]
        assert not codes[len(case["codes_head"]):].any()
    v = g["v4_group"]
    pool = hand_pool(64, v_bits=4, page_cells=64)
    k_new = np.zeros((1, 1, 128), np.float32)
    v_new = np.zeros((1, 1, 128), np.float32)
    v_new[0, 0, :len(v["x_head"])] = v["x_head"]
    out = O.append_cells(pool, k_new, v_new, 5)
    phys = out.page_table[0]
    assert out.v_scales[phys, 0, 5, 0] == np.float32(v["scale"])
    assert out.v_codes[phys, 0, 5, :2].tolist() == v["bytes_head"]
    assert out.v_codes[phys, 0, 5, 2] == 0x88                       # zeros: code 0 -> nibble 8
    assert (out.k_scales[phys, 0, 5] == 0).all() and not out.k_codes[phys, 0, 5].any()


@pytest.mark.parametrize("qmax", [127, 7])
def test_append_error_bound_and_extreme(qmax):
    """Random fp32 groups: every code within +-qmax, the largest magnitude maps to +-qmax, and the
    dequantised value is within half a step of the input (the bound of rounding to nearest)."""
    rng = np.random.default_rng(3)
    for _ in range(200):
        x = (rng.standard_normal(64) * 10.0 ** rng.uniform(-6, 4)).astype(np.float32)
        codes, scale = O.quantise_group(x, qmax)
        i = int(np.argmax(np.abs(x)))
        assert abs(codes[i]) == qmax and np.sign(codes[i]) == np.sign(x[i])
        assert np.abs(codes).max() <= qmax
        err = np.abs(codes.astype(np.float64) * np.float64(scale) - x.astype(np.float64))
        assert err.max() <= 0.5 * float(scale) * (1 + 1e-5)


@pytest.mark.parametrize("v_bits", [8, 4])
def test_append_cells_round_trip_across_pages(v_bits):
    """Cells appended across a page boundary of a permuted page table come back through the
    dequantisation within half a step per group, and no other cell changes."""
    pool = hand_pool(100, n_kv_heads=2, v_bits=v_bits, page_cells=64, capacity=256, seed=4)
    before = (pool.k_codes.copy(), pool.v_codes.copy(), pool.k_scales.copy(), pool.v_scales.copy())
    rng = np.random.default_rng(5)
    k_new = rng.standard_normal((40, 2, 128)).astype(np.float32)
    v_new = rng.standard_normal((40, 2, 128)).astype(np.float32)
    out = O.append_cells(pool, k_new, v_new, 100)                 # cells 100..139 span pages 1 and 2
    assert out.n_filled == 140 and pool.n_filled == 100
    cells = list(range(100, 140))
    for h in range(2):
        k = O.dequantise_k(out, h, cells)
        v = O.dequantise_v(out, h, cells)
        for x, back, grp, qmax in ((k_new[:, h], k, 64, 127), (v_new[:, h], v, out.v_group, 127 if v_bits == 8 else 7)):
            step = np.repeat(np.abs(x.reshape(40, -1, grp)).max(axis=2) / qmax, grp, axis=1)
            assert (np.abs(back - x) <= 0.5 * step * (1 + 1e-5)).all()
    touched = np.zeros(pool.k_codes.shape[:3], bool)
    for c in cells:
        touched[pool.page_table[c // 64], :, c % 64] = True
    for a, b in zip(before, (out.k_codes, out.v_codes, out.k_scales, out.v_scales)):
        assert np.array_equal(a[~touched], b[~touched])


# ---------------------------------------------------------------- 4-bit K (the q4_0 layout)

def _k4_twin(rng, n_cells=130, Hkv=2):
    """A pool with 4-bit K and V (q4_0 layout) whose two 32-dim K-scale groups inside each 64-dim half
    are equal, and the int8-K twin holding the same codes with one scale per 64 dims."""
    k4 = W.make_pool(rng, capacity=192, n_filled=n_cells, n_kv_heads=Hkv, page_cells=64, v_bits=4, k_bits=4)
    k4.k_scales[..., 1] = k4.k_scales[..., 0]
    k4.k_scales[..., 3] = k4.k_scales[..., 2]
    raw = np.empty(k4.k_codes.shape[:-1] + (128,), np.int8)
    raw[..., 0::2] = (k4.k_codes & 0x0F).astype(np.int8) - 8
    raw[..., 1::2] = (k4.k_codes >> 4).astype(np.int8) - 8
    k8 = W.Pool(raw, k4.v_codes.copy(), k4.k_scales[..., 0::2].copy(), k4.v_scales.copy(), k4.page_table.copy(),
                k4.capacity, k4.n_filled, k4.page_cells, k4.n_kv_heads, k4.head_dim, k4.v_bits, k4.v_group)
    return k4, k8


def test_k4_dequantise_worked_by_hand():
    """Bytes 0x8F, 0x07, 0xF0 of a 4-bit K row are dims 0..5 with codes 7, 0, -1, -8, -8, 7 (the nibble
    fixture), times the scale of their 32-dim group; dims 32.. take the second group's scale."""
    g = json.load(open(os.path.join(GOLD, "nibbles.json")))
    pool = W.make_pool(np.random.default_rng(0), capacity=64, n_filled=64, n_kv_heads=1, page_cells=64,
                       v_bits=4, k_bits=4)
    phys = pool.page_table[0]
    pool.k_codes[phys, 0, 3, :] = 0x88                         # every code 0
    pool.k_codes[phys, 0, 3, :3] = g["bytes"]
    pool.k_codes[phys, 0, 3, 16] = 0xF1                        # dims 32, 33: codes -7, 7
    pool.k_scales[phys, 0, 3, :] = [0.5, 0.25, 2.0, 4.0]
    k = O.dequantise_k(pool, 0, [3])[0]
    assert k[:6].tolist() == [0.5 * c for c in g["expect_codes"]]
    assert k[32:34].tolist() == [-7 * 0.25, 7 * 0.25]
    assert not k[6:32].any() and not k[34:].any()


def test_k4_pool_equals_its_int8_twin():
    """The same codes read as 4-bit K (two equal 32-dim scales) or as int8 K (one 64-dim scale): block
    scores, attention and a prompt row agree to rounding."""
    k4, k8 = _k4_twin(np.random.default_rng(9))
    cells = list(range(130))
    for h in range(2):
        assert np.array_equal(O.dequantise_k(k4, h, cells), O.dequantise_k(k8, h, cells))
    q = np.random.default_rng(10).standard_normal((2, 6, 128)).astype(np.float32)
    np.testing.assert_allclose(O.block_scores(k4, q, 64), O.block_scores(k8, q, 64), rtol=1e-12, atol=1e-12)
    o4, l4 = O.attention(k4, q[0], 129, cells)
    o8, l8 = O.attention(k8, q[0], 129, cells)
    np.testing.assert_allclose(o4, o8, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l4, l8, rtol=1e-12, atol=1e-12)


def test_k4_append_round_trip():
    """4-bit K appended comes back within half a step of its 32-dim group (qmax 7)."""
    pool = W.make_pool(np.random.default_rng(2), capacity=128, n_filled=10, n_kv_heads=1, page_cells=64,
                       v_bits=4, k_bits=4)
    k_new = np.random.default_rng(3).standard_normal((20, 1, 128)).astype(np.float32)
    out = O.append_cells(pool, k_new, k_new, 10)
    back = O.dequantise_k(out, 0, list(range(10, 30)))
    step = np.repeat(np.abs(k_new[:, 0].reshape(20, 4, 32)).max(axis=2) / 7, 32, axis=1)
    assert (np.abs(back - k_new[:, 0]) <= 0.5 * step * (1 + 1e-5)).all()
    assert out.k_scales.shape[-1] == 4
