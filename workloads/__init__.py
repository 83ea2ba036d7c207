"""Seeded synthetic inputs for QSA attention over a quantised, paged KV cache.

This module only draws random numbers and lays them out in the storage format
that both the CUDA library and the CPU oracle read.  It holds none of the
method's arithmetic (no dequantisation, scoring, selection or attention).

Storage format of one pool (one slot's KV cache), all arrays C-contiguous:

  k_codes   int8    [n_pages, n_kv_heads, page_cells, head_dim]
  v_codes   int8    [n_pages, n_kv_heads, page_cells, head_dim]        (v_bits = 8)
            uint8   [n_pages, n_kv_heads, page_cells, head_dim // 2]   (v_bits = 4;
                    byte j holds dims 2j (low nibble) and 2j+1 (high nibble),
                    each nibble = code + 8)
  k_scales  float32 [n_pages, n_kv_heads, page_cells, head_dim // 64]
  v_scales  float32 [n_pages, n_kv_heads, page_cells, head_dim // v_group]
  page_table int32  [n_pages]   logical page -> physical page

Logical cell c lives in physical page page_table[c // page_cells] at offset
c % page_cells.  Cells at or beyond n_filled are stale: their codes are random
and their scales are NaN, so any read of them poisons a result.

Value recipe (the pages' synthetic workloads: int8 K/V codes, fp32 scales per
(cell, KV head, group), fp32 queries):
  codes uniform integers in [-127, 127] (4-bit V: [-8, 7]);
  scales uniform in [0.005, 0.02];
  q ~ N(0, 1) as float32;
  page table a seeded random permutation of the physical pages;
  optional bias: each filled cell is biased with probability bias_prob; a
  biased cell's K codes of KV head h get rint(3 * sigma * u_h[d]) added and are
  clamped to [-127, 127], sigma = sqrt((255**2 - 1) / 12) (the code
  distribution's standard deviation) and u_h a seeded unit vector per head.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

HEAD_DIM = 128
K_GROUP = 64
SCALE_LO = 0.005
SCALE_HI = 0.02
CODE_SIGMA = math.sqrt((255.0 ** 2 - 1.0) / 12.0)
CODE_SIGMA_4 = math.sqrt((16.0 ** 2 - 1.0) / 12.0)   # spread of 4-bit codes uniform in [-8, 7]


@dataclasses.dataclass
class Pool:
    k_codes: np.ndarray
    v_codes: np.ndarray
    k_scales: np.ndarray
    v_scales: np.ndarray
    page_table: np.ndarray
    capacity: int
    n_filled: int
    page_cells: int
    n_kv_heads: int
    head_dim: int
    v_bits: int
    v_group: int
    k_bits: int = 8
    k_group: int = 64

    @property
    def n_pages(self) -> int:
        return int(self.k_codes.shape[0])


def _pack_nibbles(raw: np.ndarray) -> np.ndarray:
    """4-bit codes in [-8, 7] -> bytes: nibble = code + 8, the even dim in the low nibble."""
    nib = (raw.astype(np.int16) + 8).astype(np.uint8)
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def make_pool(rng: np.random.Generator, *, capacity: int, n_filled: int, n_kv_heads: int,
              head_dim: int = HEAD_DIM, page_cells: int = 256, v_bits: int = 8,
              bias_prob: float = 0.0, k_bits: int = 8, code_lo: int = -127) -> Pool:
    """Draw one paged pool.  Draw order: page table, K codes, K scales, V codes,
    V scales, then (if bias_prob > 0) the bias mask and the bias directions.
    k_bits = 4 (with v_bits = 4: the q4_0 layout) draws K codes in [-8, 7] with
    one scale per 32 dims, packed as the 4-bit V codes are.  int8 codes are
    drawn in [code_lo, 127] (code_lo -128 includes the one code without a
    positive twin)."""
    assert 0 <= n_filled <= capacity
    assert head_dim % K_GROUP == 0 and v_bits in (4, 8) and k_bits in (4, 8)
    n_pages = (capacity + page_cells - 1) // page_cells
    v_group = 64 if v_bits == 8 else 32
    k_group = 64 if k_bits == 8 else 32
    page_table = rng.permutation(n_pages).astype(np.int32)
    shape = (n_pages, n_kv_heads, page_cells, head_dim)
    if k_bits == 8:
        k_codes = rng.integers(code_lo, 128, size=shape, dtype=np.int8)
    else:
        k_codes = _pack_nibbles(rng.integers(-8, 8, size=shape, dtype=np.int8))
    k_scales = rng.uniform(SCALE_LO, SCALE_HI,
                           size=(n_pages, n_kv_heads, page_cells, head_dim // k_group)).astype(np.float32)
    if v_bits == 8:
        v_codes = rng.integers(code_lo, 128, size=shape, dtype=np.int8)
    else:
        v_codes = _pack_nibbles(rng.integers(-8, 8, size=shape, dtype=np.int8))
    v_scales = rng.uniform(SCALE_LO, SCALE_HI,
                           size=(n_pages, n_kv_heads, page_cells, head_dim // v_group)).astype(np.float32)
    pool = Pool(k_codes, v_codes, k_scales, v_scales, page_table, capacity, n_filled,
                page_cells, n_kv_heads, head_dim, v_bits, v_group, k_bits, k_group)
    if bias_prob > 0.0 and n_filled > 0:
        biased = rng.random(n_filled) < bias_prob
        u = rng.standard_normal((n_kv_heads, head_dim))
        u /= np.linalg.norm(u, axis=1, keepdims=True)
        add = np.rint(3.0 * CODE_SIGMA * u).astype(np.int16)  # [Hkv, D]
        cells = np.nonzero(biased)[0]
        phys = page_table[cells // page_cells]
        off = cells % page_cells
        for h in range(n_kv_heads):
            if k_bits == 8:
                cur = k_codes[phys, h, off, :].astype(np.int16) + add[h][None, :]
                k_codes[phys, h, off, :] = np.clip(cur, -127, 127).astype(np.int8)
            else:   # the same direction at the 4-bit code spread
                b = k_codes[phys, h, off, :]
                raw = np.empty(b.shape[:-1] + (head_dim,), np.int16)
                raw[..., 0::2] = (b & 0x0F).astype(np.int16) - 8
                raw[..., 1::2] = (b >> 4).astype(np.int16) - 8
                add4 = np.rint(3.0 * CODE_SIGMA_4 * u[h]).astype(np.int16)
                k_codes[phys, h, off, :] = _pack_nibbles(np.clip(raw + add4[None, :], -8, 7))
    _poison_stale_cells(pool)
    return pool


def _poison_stale_cells(pool: Pool) -> None:
    """Scales of cells at or beyond n_filled become NaN."""
    total = pool.n_pages * pool.page_cells
    if pool.n_filled >= total:
        return
    stale = np.arange(pool.n_filled, total)
    phys = pool.page_table[stale // pool.page_cells]
    off = stale % pool.page_cells
    pool.k_scales[phys, :, off, :] = np.nan
    pool.v_scales[phys, :, off, :] = np.nan


def make_q(rng: np.random.Generator, n_rows: int, n_heads: int, head_dim: int = HEAD_DIM) -> np.ndarray:
    return rng.standard_normal((n_rows, n_heads, head_dim)).astype(np.float32)


@dataclasses.dataclass
class DecodeCase:
    """One decode window: rows (queries) over one or more slots' pools."""
    name: str
    pools: List[Pool]
    row_pool: np.ndarray   # int32 [R]: pool index of each row
    q: np.ndarray          # float32 [R, Hq, D]
    row_pos: np.ndarray    # int32 [R]: the cell each row sits at (causal limit, inclusive)
    n_q_heads: int
    block_cells: int
    k_cells: int
    chunk_cells: int
    max_blocks: int        # row stride of the scores array
    n_chunks: int          # chunks per (row, head) in the partials buffer

    @property
    def n_rows(self) -> int:
        return int(self.q.shape[0])

    def n_filled_rows(self) -> np.ndarray:
        return np.array([self.pools[p].n_filled for p in self.row_pool], dtype=np.int32)


@dataclasses.dataclass
class PromptCase:
    """Prompt chunks: calls[i] = (first query index, number of queries, position of the first)."""
    name: str
    pool: Pool
    q: np.ndarray          # float32 [n_q, Hq, D]
    calls: List[tuple]
    n_q_heads: int


def decode_case(*, name: str, seed: int, fills: List[int], capacity: int, rows_per_slot: int,
                n_q_heads: int, n_kv_heads: int, k_cells: int, chunk_cells: int,
                block_cells: int = 64, page_cells: int = 256, bias_prob: float = 0.0,
                n_chunks: Optional[int] = None, v_bits: int = 8,
                row_pos: Optional[List[int]] = None, k_bits: int = 8, code_lo: int = -127) -> DecodeCase:
    """Pools are drawn slot by slot, then q.  Rows of a slot are contiguous and
    sit at the last positions of its fill unless row_pos is given."""
    rng = np.random.default_rng(seed)
    pools = [make_pool(rng, capacity=capacity, n_filled=f, n_kv_heads=n_kv_heads,
                       page_cells=page_cells, v_bits=v_bits, bias_prob=bias_prob, k_bits=k_bits,
                       code_lo=code_lo) for f in fills]
    row_pool, pos = [], []
    for s, f in enumerate(fills):
        for r in range(rows_per_slot):
            row_pool.append(s)
            pos.append(f - rows_per_slot + r)
    if row_pos is not None:
        pos = list(row_pos)
    q = make_q(rng, len(row_pool), n_q_heads)
    max_blocks = (capacity + block_cells - 1) // block_cells
    if n_chunks is None:
        n_chunks = (k_cells + chunk_cells - 1) // chunk_cells
    return DecodeCase(name, pools, np.array(row_pool, np.int32), q, np.array(pos, np.int32),
                      n_q_heads, block_cells, k_cells, chunk_cells, max_blocks, n_chunks)


def prompt_case(*, name: str, seed: int, n_ctx: int, n_q: int, n_q_heads: int, n_kv_heads: int,
                v_bits: int = 8, calls_of: Optional[int] = None, page_cells: int = 256,
                capacity: Optional[int] = None, k_bits: int = 8, code_lo: int = -127) -> PromptCase:
    """Queries sit at the last n_q positions of the context (causal over them)."""
    rng = np.random.default_rng(seed)
    pool = make_pool(rng, capacity=capacity or n_ctx, n_filled=n_ctx, n_kv_heads=n_kv_heads,
                     page_cells=page_cells, v_bits=v_bits, k_bits=k_bits, code_lo=code_lo)
    q = make_q(rng, n_q, n_q_heads)
    per = calls_of or n_q
    pos0 = n_ctx - n_q
    calls = [(i, min(per, n_q - i), pos0 + i) for i in range(0, n_q, per)]
    return PromptCase(name, pool, q, calls, n_q_heads)


# --- the five named workloads -------------------------------------------------

def tiny_dense_decode() -> DecodeCase:
    """1 query at position 1,023; 2 q heads on 1 KV head; 1,024 filled cells; top-k = all;
    4 chunks of 256 cells; seed 0."""
    return decode_case(name="tiny_dense_decode", seed=0, fills=[1024], capacity=1024, rows_per_slot=1,
                       n_q_heads=2, n_kv_heads=1, k_cells=1024, chunk_cells=256)


def verify_window() -> DecodeCase:
    """5 rows (4 drafts + 1) at positions 32,763..32,767; 24 q heads / 4 KV heads; 32,768 filled
    cells; 64-cell blocks; top-k 4,096 cells; 64-cell chunks; 5 % of cells K-biased; seed 1."""
    return decode_case(name="verify_window", seed=1, fills=[32768], capacity=32768, rows_per_slot=5,
                       n_q_heads=24, n_kv_heads=4, k_cells=4096, chunk_cells=64, bias_prob=0.05)


def batched_long_context(n_chunks: Optional[int] = None) -> DecodeCase:
    """2 slots x 2 rows; capacity 200,000 cells per slot, fills 65,536 and 131,072; 24/4 heads;
    top-k 8,192 cells; 64-cell chunks; 5 % bias; seed 2.  n_chunks=512 sizes the partials for the
    drafter's 32K window, so chunks 128..511 hold no cells."""
    return decode_case(name="batched_long_context", seed=2, fills=[65536, 131072], capacity=200000,
                       rows_per_slot=2, n_q_heads=24, n_kv_heads=4, k_cells=8192, chunk_cells=64,
                       bias_prob=0.05, n_chunks=n_chunks)


def prompt_int8() -> PromptCase:
    """2,048 queries at positions 30,720..32,767 against 32,768 cells; 24/4 heads; int8 K/V; seed 3."""
    return prompt_case(name="prompt_int8", seed=3, n_ctx=32768, n_q=2048, n_q_heads=24, n_kv_heads=4)


def prompt_k8v4() -> PromptCase:
    """8,192 queries at positions 122,880..131,071 against 131,072 cells; 32/8 heads; int8 K,
    4-bit V with per-32-dim scales; four calls of 2,048 queries; seed 4."""
    return prompt_case(name="prompt_k8v4", seed=4, n_ctx=131072, n_q=8192, n_q_heads=32, n_kv_heads=8,
                       v_bits=4, calls_of=2048)


NAMED = {
    "tiny_dense_decode": tiny_dense_decode,
    "verify_window": verify_window,
    "batched_long_context": batched_long_context,
    "prompt_int8": prompt_int8,
    "prompt_k8v4": prompt_k8v4,
}
