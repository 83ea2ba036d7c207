"""Plain FP64 oracle of QSA attention over a paged int8 / int8-K 4-bit-V KV cache.

TEST INFRASTRUCTURE ONLY (tests, smoke check, bench CPU baseline).  Slow and
obviously correct: every function takes the method's steps in the order the
pages give them, in float64 numpy, with no blocking, fusion or reordering
beyond what the definition states.  It shares no code with the CUDA library.

Sources (pull-request pages of the "Strata" inference engine):
  [1888]  "#1888 QSA decode attention: split each query's cells across blocks
           on the int8 mma path" -- Summary; What changed.
  [2075]  "#2075 QSA decode attention: PR #540's two-cells-per-step chunk
           kernel on every CUDA card and a bounded merge" -- Summary; Why;
           Bit for bit.
  [600]   "qsa_prompt_attn: tensor-core kernel for Volta (sm_70, mma.m8n8k4)"
           -- description; accuracy table.
  [2806]  "#2806 sycl: decode QSA selection and attention in fewer, shorter
           launches" -- Summary (switch table); What changed.
  [1367]  "#1367 prompt attention: STRATA_PROMPT_ATTN_IMMA=1 - the int8-KV
           kernel on INT8 tensor cores" -- What it does (Operands).

Readings taken where the pages are silent (each also listed in the design
notes of the repository):
  R1  softmax scale 1/sqrt(D), D = 128;
  R2  q head g reads KV head floor(g / G), G = Hq / Hkv (contiguous groups);
  R3  block score S[t,b] = sum_h (1/n_b) sum_{c in b} sum_{g in G(h)}
      q[t,g] . K[c,h] / sqrt(D)  (mean logit of the block, summed over the
      group's q heads, then over KV heads; no causal mask in scoring);
  R4  top-k orders blocks by score descending, ties by block id ascending;
      -0.0 equals +0.0; every NaN ranks below -inf (and equal to other NaNs);
      k_cells must be a multiple of the block size; the first k_cells / B
      blocks are taken (all blocks if fewer exist); the output is the filled
      cells of the chosen blocks in ascending cell id;
  R5  causal rule self-inclusive: a row at position p sees cells c <= p;
  R6  an empty cell set gives out = 0 and lse = -inf; a chunk with no
      visible cell is empty and the merge skips it;
  R7  chunk j of a row is entries [j*C, (j+1)*C) of its selected-id list;
  R8  4-bit V: code = nibble - 8, low nibble = even dim, one scale per
      32-dim group; int8 V and int8 K: one scale per 64-dim group;
  R15 context-sharded decode (a slot's cells split into ranges held by
      different GPUs) selects once per row over the block scores of all
      ranges (one global top-k): the selection, and so the result of
      decode_window, does not depend on the split; each range contributes the
      chunk partials of the selected cells it holds, merged by log-sum-exp;
  R14 appending a cell quantises each group of its K and V rows symmetrically
      by the group's largest magnitude: scale = amax / 127 (int8) or amax / 7
      (4-bit V), code = round-half-to-even(x / scale) clamped to +-127 (+-7),
      amax = 0 giving scale 0 and codes 0; the division and rounding that
      decide the integer codes are taken in fp32 (the stored precision), so
      the codes are exact integers both sides agree on.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np

__all__ = [
    "dequantise_k", "dequantise_v", "kv_head", "block_scores", "score_key",
    "topk_select", "attention", "chunk_partials", "merge_partials",
    "prompt_attention", "decode_window", "quantise_group", "append_cells", "block_summaries",
]


# ---------------------------------------------------------------- dequantise

def _page_slots(pool, cells: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    cells = np.asarray(cells, dtype=np.int64)
    return pool.page_table[cells // pool.page_cells].astype(np.int64), cells % pool.page_cells


def _unpack_nibbles(raw: np.ndarray, head_dim: int) -> np.ndarray:
    """Bytes [n, D/2] -> codes float64 [n, D]: byte j holds dim 2j in its low nibble and 2j + 1 in
    its high nibble, code = nibble - 8 (reading R8)."""
    codes = np.empty((raw.shape[0], head_dim), dtype=np.float64)
    codes[:, 0::2] = (raw & 0x0F).astype(np.int64) - 8
    codes[:, 1::2] = (raw >> 4).astype(np.int64) - 8
    return codes


def dequantise_k(pool, h: int, cells: Sequence[int]) -> np.ndarray:
    """K[c, h, d] = kcode[c, h, d] * kscale[c, h, d // kgroup], float64 [n, D].

    Per-(cell, KV head, 64-dim group) fp32 scale: [600] description ("one
    64-dim group (= one int8 scale group)"); [1367] Operands (int8 K codes used
    as stored).  4-bit K (the q4_0 KV format of [2075] Bit for bit): codes and
    32-dim groups as for 4-bit V."""
    phys, off = _page_slots(pool, np.asarray(cells))
    raw = pool.k_codes[phys, h, off, :]
    k_bits = getattr(pool, "k_bits", 8)
    codes = raw.astype(np.float64) if k_bits == 8 else _unpack_nibbles(raw, pool.head_dim)   # [n, D]
    scales = pool.k_scales[phys, h, off, :].astype(np.float64)                               # [n, D/kgroup]
    return codes * np.repeat(scales, pool.head_dim // scales.shape[1], axis=1)


def dequantise_v(pool, h: int, cells: Sequence[int]) -> np.ndarray:
    """V[c, h, d] = vcode[c, h, d] * vscale[c, h, d // vgroup], float64 [n, D].

    int8 V: group 64.  4-bit V (the K8V4 format named in [1888] and [2075]):
    code = nibble - 8, low nibble holds the even dim, group 32 (reading R8)."""
    phys, off = _page_slots(pool, np.asarray(cells))
    raw = pool.v_codes[phys, h, off, :]
    codes = raw.astype(np.float64) if pool.v_bits == 8 else _unpack_nibbles(raw, pool.head_dim)
    scales = pool.v_scales[phys, h, off, :].astype(np.float64)
    return codes * np.repeat(scales, pool.v_group, axis=1)


# ---------------------------------------------------------------- append (quantise new cells)

def quantise_group(x, qmax: int) -> Tuple[np.ndarray, np.float32]:
    """Codes and scale of one group of fp32 values (reading R14).

    The pages store K/V as int8 (4-bit for K8V4 V) codes with one fp32 scale
    per (cell, KV head, group) ([1367] Operands; [1888], [2075] name the K8V4
    format) and append new cells per row ([2806] What it leaves alone: "K/V and
    indexer appends"), but give no quantiser; the plainest one is symmetric:
    scale = max |x| / qmax, code = x / scale rounded to nearest (ties to even),
    in fp32."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    if amax == 0:
        return np.zeros(x.shape, dtype=np.int64), np.float32(0)
    scale = np.float32(amax / np.float32(qmax))          # fp32 division, rounded to nearest
    q = np.rint(x / scale)                                # fp32 division, then ties-to-even
    return np.clip(q, -qmax, qmax).astype(np.int64), scale


def append_cells(pool, k_new: np.ndarray, v_new: np.ndarray, first_cell: int):
    """A copy of `pool` with cells first_cell .. first_cell + n - 1 written from k_new, v_new (fp32
    [n][Hkv][D]): each of K and V in int8 with one scale per 64 dims, or in 4-bit (code + 8 in a
    nibble, the even dim in the low nibble) with one scale per 32 dims, as the pool stores it.  n_filled becomes
    max(n_filled, first_cell + n)."""
    import copy
    out = copy.deepcopy(pool)
    n = k_new.shape[0]
    for i in range(n):
        cell = first_cell + i
        phys = int(pool.page_table[cell // pool.page_cells])
        off = cell % pool.page_cells
        for h in range(pool.n_kv_heads):
            for x_new, bits, grp, codes_arr, scales_arr in (
                    (k_new, getattr(pool, "k_bits", 8), getattr(pool, "k_group", 64), out.k_codes, out.k_scales),
                    (v_new, pool.v_bits, pool.v_group, out.v_codes, out.v_scales)):
                for g in range(pool.head_dim // grp):
                    codes, scale = quantise_group(x_new[i, h, grp * g:grp * (g + 1)], 127 if bits == 8 else 7)
                    scales_arr[phys, h, off, g] = scale
                    if bits == 8:
                        codes_arr[phys, h, off, grp * g:grp * (g + 1)] = codes
                    else:
                        nib = (codes + 8).astype(np.uint8)
                        for j in range(0, grp, 2):
                            d = grp * g + j
                            codes_arr[phys, h, off, d // 2] = nib[j] | (nib[j + 1] << 4)
    out.n_filled = max(pool.n_filled, first_cell + n)
    return out


def kv_head(g: int, n_q_heads: int, n_kv_heads: int) -> int:
    """Reading R2: contiguous GQA groups, G = Hq / Hkv."""
    return g // (n_q_heads // n_kv_heads)


# ---------------------------------------------------------------- block scores

def block_scores(pool, q_rows: np.ndarray, block_cells: int) -> np.ndarray:
    """Decode block scores of one slot's rows, float64 [R, nb], nb = ceil(n_filled / B).

    The pages name the step (a slot's rows are scored together; a block's
    (query, head) sums are reduced together: [2806] Summary and What changed)
    but print no formula; this is reading R3:
        S[t,b] = sum_h (1/n_b) sum_{c in b} sum_{g in G(h)} q[t,g] . K[c,h] / sqrt(D)
    over the block's filled cells c (n_b of them)."""
    R, Hq, D = q_rows.shape
    Hkv = pool.n_kv_heads
    G = Hq // Hkv
    nb = (pool.n_filled + block_cells - 1) // block_cells
    q64 = q_rows.astype(np.float64)
    out = np.zeros((R, nb), dtype=np.float64)
    for b in range(nb):
        cells = np.arange(b * block_cells, min((b + 1) * block_cells, pool.n_filled))
        n_b = len(cells)
        for h in range(Hkv):
            K = dequantise_k(pool, h, cells)                         # [n_b, D]
            for t in range(R):
                qg = q64[t, h * G:(h + 1) * G, :]                    # [G, D]
                logits = qg @ K.T / math.sqrt(D)                     # [G, n_b]
                out[t, b] += logits.sum() / n_b
    return out


def block_summaries(pool, summary_cells: int = 64) -> np.ndarray:
    """Sum of the dequantised K rows over the filled cells of each summary block of
    `summary_cells` cells, float64 [n_blocks, Hkv, D] (the index of blocks a pool may keep
    beside its cells; by R3's linearity the block score is
    S[t,b] = sum_h qbar[t,h] . (sum of b's summaries)[h] / (n_b sqrt(D)))."""
    Hkv, D = pool.n_kv_heads, pool.head_dim
    nb = (pool.n_filled + summary_cells - 1) // summary_cells
    out = np.zeros((nb, Hkv, D))
    for b in range(nb):
        cells = np.arange(b * summary_cells, min((b + 1) * summary_cells, pool.n_filled))
        for h in range(Hkv):
            out[b, h] = dequantise_k(pool, h, cells).sum(axis=0)
    return out


# ---------------------------------------------------------------- top-k

def score_key(x) -> int:
    """Order-preserving unsigned key of a float32 score (reading R4).

    -0.0 maps to the key of +0.0; every NaN maps to 0, below -inf."""
    f = np.float32(x)
    if np.isnan(f):
        return 0
    if f == 0.0:
        f = np.float32(0.0)
    u = int(np.array(f, dtype=np.float32).view(np.uint32))
    return (~u) & 0xFFFFFFFF if (u & 0x80000000) else (u | 0x80000000)


def topk_select(scores_f32: Sequence[float], n_filled: int, block_cells: int,
                k_cells: int) -> Tuple[np.ndarray, int]:
    """Selected cell ids (int32, ascending) and their count for one row.

    The top-k picks the highest-scoring blocks and hands their cells to the
    attention ([2806] Summary: top-k once per window; integer keys, so the
    same ids whatever the kernel).  Full sort, reading R4."""
    if k_cells % block_cells != 0:
        raise ValueError("k_cells must be a multiple of the block size")
    nb = (n_filled + block_cells - 1) // block_cells
    keys = [score_key(scores_f32[b]) for b in range(nb)]
    order = sorted(range(nb), key=lambda b: (-keys[b], b))
    chosen = sorted(order[: k_cells // block_cells])
    ids: List[int] = []
    for b in chosen:
        ids.extend(range(b * block_cells, min((b + 1) * block_cells, n_filled)))
    return np.array(ids, dtype=np.int32), len(ids)


# ---------------------------------------------------------------- attention

def attention(pool, q_row: np.ndarray, pos: int, ids: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """Exact softmax attention of one row over its selected cells.

    out[g] = sum_c softmax(z)_c V[c], z_c = q[g] . K[c, kv(g)] / sqrt(D),
    lse[g] = log sum_c exp(z_c), over selected cells c <= pos (R1, R2, R5, R6).
    float64; returns out [Hq, D], lse [Hq]."""
    Hq, D = q_row.shape
    Hkv = pool.n_kv_heads
    vis = np.array([c for c in ids if c <= pos], dtype=np.int64)
    out = np.zeros((Hq, D), dtype=np.float64)
    lse = np.full(Hq, -np.inf, dtype=np.float64)
    if len(vis) == 0:
        return out, lse
    for g in range(Hq):
        h = kv_head(g, Hq, Hkv)
        K = dequantise_k(pool, h, vis)
        V = dequantise_v(pool, h, vis)
        z = K @ q_row[g].astype(np.float64) / math.sqrt(D)
        m = z.max()
        p = np.exp(z - m)
        lsum = p.sum()
        out[g] = (p @ V) / lsum
        lse[g] = m + math.log(lsum)
    return out, lse


def chunk_partials(pool, q_row: np.ndarray, pos: int, ids: Sequence[int], chunk_cells: int,
                   n_chunks: int):
    """Per-chunk (m, l, o) of one row: the chunk kernel's output ([2075] Summary:
    chunks of selected cells; [1888] Summary: each query's cells split among blocks).

    m = max logit, l = sum exp(z - m), o = sum exp(z - m) V over the chunk's
    visible cells (R7); an empty chunk has m = -inf, l = 0, o = 0.
    Returns m, l [Hq, n_chunks] and o [Hq, n_chunks, D], float64."""
    Hq, D = q_row.shape
    Hkv = pool.n_kv_heads
    m = np.full((Hq, n_chunks), -np.inf)
    l = np.zeros((Hq, n_chunks))
    o = np.zeros((Hq, n_chunks, D))
    ids = list(ids)
    for j in range(n_chunks):
        cells = np.array([c for c in ids[j * chunk_cells:(j + 1) * chunk_cells] if c <= pos], dtype=np.int64)
        if len(cells) == 0:
            continue
        for g in range(Hq):
            h = kv_head(g, Hq, Hkv)
            K = dequantise_k(pool, h, cells)
            V = dequantise_v(pool, h, cells)
            z = K @ q_row[g].astype(np.float64) / math.sqrt(D)
            m[g, j] = z.max()
            p = np.exp(z - m[g, j])
            l[g, j] = p.sum()
            o[g, j] = p @ V
    return m, l, o


def merge_partials(m: np.ndarray, l: np.ndarray, o: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Log-sum-exp merge of chunk partials in chunk order, skipping empty chunks.

    M = max m_j over non-empty chunks; L = sum_j l_j exp(m_j - M);
    out = sum_j o_j exp(m_j - M) / L; lse = M + log L
    ([1888] What changed: splits merged in split order with the log-sum-exp
    rescale; [2075] Summary and [2806] Summary: the merge skips the chunks
    marked empty and those past the selection).  m, l: [Hq, n]; o: [Hq, n, D]."""
    Hq, n, D = o.shape
    out = np.zeros((Hq, D))
    lse = np.full(Hq, -np.inf)
    for g in range(Hq):
        live = [j for j in range(n) if m[g, j] != -np.inf]
        if not live:
            continue
        M = max(m[g, j] for j in live)
        L = 0.0
        acc = np.zeros(D)
        for j in live:
            w = math.exp(m[g, j] - M)
            L += l[g, j] * w
            acc += o[g, j] * w
        out[g] = acc / L
        lse[g] = M + math.log(L)
    return out, lse


# ---------------------------------------------------------------- prompt

def prompt_attention(pool, q: np.ndarray, q_pos0: int, rows: Sequence[int] = None, heads: Sequence[int] = None,
                     row_block: int = 64):
    """Dense causal prompt attention of a chunk of queries ([1367] What it does;
    [600] description: a chunk of queries against the whole cached context).

    Query i sits at position q_pos0 + i and sees cells 0..q_pos0+i (R5).  The
    computation is the exact attention of the fp32 q on the dequantised K/V;
    the GPU's operand split is rounding inside its error budget.  For each q
    head the logits of up to `row_block` rows come from one matrix product
    with the head's dequantised K; a row's cells past its position are masked
    to -inf before the softmax (so they weigh exactly 0), and the weights
    multiply V in a second product.  `heads` limits the q heads computed
    (others are left at out = 0, lse = -inf).
    Returns out [len(rows), Hq, D] and lse [len(rows), Hq], float64."""
    n_q, Hq, D = q.shape
    Hkv = pool.n_kv_heads
    rows = list(range(n_q)) if rows is None else list(rows)
    heads = list(range(Hq)) if heads is None else list(heads)
    last = q_pos0 + max(rows) + 1 if rows else 0
    out = np.zeros((len(rows), Hq, D))
    lse = np.full((len(rows), Hq), -np.inf)
    for h in range(Hkv):
        group = [g for g in heads if kv_head(g, Hq, Hkv) == h]
        if not group:
            continue
        K = dequantise_k(pool, h, np.arange(last))
        V = dequantise_v(pool, h, np.arange(last))
        for b0 in range(0, len(rows), row_block):
            blk = rows[b0:b0 + row_block]
            pos = q_pos0 + np.asarray(blk)                     # each row's own cell
            n = int(pos.max()) + 1
            hidden = np.arange(n)[None, :] > pos[:, None]      # cells past the row's position
            for g in group:
                z = q[blk, g].astype(np.float64) @ K[:n].T / math.sqrt(D)   # [rows, n]
                z[hidden] = -np.inf
                mx = z.max(axis=1, keepdims=True)
                p = np.exp(z - mx)
                s = p.sum(axis=1)
                out[b0:b0 + len(blk), g] = (p @ V[:n]) / s[:, None]
                lse[b0:b0 + len(blk), g] = mx[:, 0] + np.log(s)
    return out, lse


# ---------------------------------------------------------------- whole window

def decode_window(case, scores_f32: np.ndarray = None):
    """The decode chain of one window, in the pages' order ([2806] What changed:
    scores per slot, one top-k per window, attention over every slot's pools,
    then the merge).  If scores_f32 [R, max_blocks] is given, the top-k ranks
    those (so that selections can be compared given identical scores);
    otherwise the oracle's own scores rounded to float32.
    Returns dict with scores (float64), ids (list), n_sel, m, l, o, out, lse."""
    R = case.n_rows
    Hq, D = case.n_q_heads, case.q.shape[2]
    scores64 = [None] * R
    for p_idx, pool in enumerate(case.pools):
        rows = [t for t in range(R) if case.row_pool[t] == p_idx]
        if not rows:
            continue
        s = block_scores(pool, case.q[rows], case.block_cells)
        for i, t in enumerate(rows):
            scores64[t] = s[i]
    ids, n_sel = [], np.zeros(R, dtype=np.int32)
    m = np.full((R, Hq, case.n_chunks), -np.inf)
    l = np.zeros((R, Hq, case.n_chunks))
    o = np.zeros((R, Hq, case.n_chunks, D))
    out = np.zeros((R, Hq, D))
    lse = np.zeros((R, Hq))
    for t in range(R):
        pool = case.pools[case.row_pool[t]]
        row_scores = scores_f32[t] if scores_f32 is not None else scores64[t].astype(np.float32)
        sel, n = topk_select(row_scores, pool.n_filled, case.block_cells, case.k_cells)
        ids.append(sel)
        n_sel[t] = n
        m[t], l[t], o[t] = chunk_partials(pool, case.q[t], int(case.row_pos[t]), sel,
                                          case.chunk_cells, case.n_chunks)
        out[t], lse[t] = merge_partials(m[t], l[t], o[t])
    return dict(scores=scores64, ids=ids, n_sel=n_sel, m=m, l=l, o=o, out=out, lse=lse)
