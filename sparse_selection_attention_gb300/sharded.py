"""Context-sharded decode window: each rank (one GPU) holds a range of every slot's cells.

The cells of a slot are split into `world` contiguous runs of whole pages; rank r describes its run
of each slot as a pool view (the page table advanced by the run's first page, the fill shortened),
so every kernel of the library runs on a view unchanged.  One window is four phases:

  1. scores   each rank scores the blocks of its views (qsa_block_scores);
     exchange all-gather of the block scores;
  2. select   every rank assembles the slot's whole score row and runs qsa_topk on it: one global
              selection, the same on every rank and equal to a single GPU's;
  3. attend   each rank keeps the selected ids inside its runs (qsa_ids_in_range) and runs the chunk
              attention over them on its views (qsa_decode_attn);
     exchange all-gather of the chunk partials and of the ranks' selection counts;
  4. merge    every rank folds all ranks' partials by log-sum-exp in rank order
              (qsa_attn_merge_shards).

("#1888 QSA decode attention: split each query's cells across blocks on the int8 mma path",
Summary: a query's cells are split, each split yields (m, l, o), and the splits are merged by the
log-sum-exp rescale in split order.)  The phases take a backend (the library on a CUDA device, or
any object with the same methods) and the exchange is the caller's: `run_window` uses
torch.distributed all-gathers; a single process can also run the ranks one after another and
concatenate their results.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence, Tuple


def page_runs(n_filled: int, page_cells: int, world: int) -> List[Tuple[int, int]]:
    """The filled pages of a slot cut into `world` contiguous runs [p0, p1) of near-equal length
    (rank order; a run may be empty when the slot has fewer pages than ranks)."""
    pages = (n_filled + page_cells - 1) // page_cells
    return [(pages * r // world, pages * (r + 1) // world) for r in range(world)]


@dataclass
class ShardPlan:
    """Rank `rank`'s cell ranges [lo, hi) of each pool (multiples of page_cells, hi clipped to the
    fill) and the blocks they start at."""
    rank: int
    world: int
    lo: List[int]
    hi: List[int]
    first_page: List[int]
    local_blocks: int      # block columns of one rank's scores (the most any rank's run needs)

    @staticmethod
    def make(fills: Sequence[int], page_cells: Sequence[int], block_cells: int, rank: int, world: int):
        lo, hi, fp = [], [], []
        most = 1
        for n_filled, pc in zip(fills, page_cells):
            runs = page_runs(n_filled, pc, world)
            p0, p1 = runs[rank]
            lo.append(p0 * pc)
            hi.append(min(p1 * pc, n_filled) if p1 > p0 else p0 * pc)
            fp.append(p0)
            for a, b in runs:
                cells = max(0, min(b * pc, n_filled) - a * pc)
                most = max(most, (cells + block_cells - 1) // block_cells)
        return ShardPlan(rank, world, lo, hi, fp, most)


def phase_scores(backend, plan: ShardPlan, views, row_pool, q, block_cells: int):
    return backend.block_scores(views, row_pool, q, block_cells, plan.local_blocks)


def phase_select(backend, plans: Sequence[ShardPlan], gathered_scores, fills, row_pool, block_cells: int,
                 k_cells: int, max_blocks: int):
    """Every rank's block scores (rank order) -> the whole score rows -> the global selection."""
    return backend.topk_gathered(gathered_scores, plans, fills, row_pool, block_cells, k_cells, max_blocks)


def phase_attend(backend, plan: ShardPlan, views, row_pool, q, row_pos, ids, n_sel, k_cells: int,
                 chunk_cells: int, n_chunks: int):
    lo = [plan.lo[p] for p in row_pool]
    hi = [plan.hi[p] for p in row_pool]
    ids_r, n_sel_r, pos_r = backend.ids_in_range(ids, n_sel, row_pos, lo, hi, k_cells)
    partials = backend.decode_attn(views, row_pool, q, pos_r, ids_r, n_sel_r, k_cells, chunk_cells, n_chunks)
    return partials, n_sel_r


def phase_merge(backend, gathered_partials, gathered_n_sel, n_rows: int, n_q_heads: int, chunk_cells: int,
                n_chunks: int):
    return backend.merge_shards(gathered_partials, gathered_n_sel, n_rows, n_q_heads, chunk_cells, n_chunks)


def run_window(backend, pools, row_pool, q, row_pos, n_q_heads: int, block_cells: int, k_cells: int,
               chunk_cells: int, n_chunks: int, max_blocks: int, rank: int, world: int, all_gather):
    """One window on this rank; `all_gather(x)` returns every rank's x in rank order (a collective
    every rank calls at the same point).  Returns (ids, n_sel, out, lse), the same on every rank."""
    fills = [backend.fill(p) for p in pools]
    pcs = [backend.page_cells(p) for p in pools]
    plans = [ShardPlan.make(fills, pcs, block_cells, r, world) for r in range(world)]
    plan = plans[rank]
    views = [backend.view(p, plan.first_page[i], plan.hi[i] - plan.lo[i]) for i, p in enumerate(pools)]
    local = phase_scores(backend, plan, views, row_pool, q, block_cells)
    ids, n_sel = phase_select(backend, plans, all_gather(local), fills, row_pool, block_cells, k_cells, max_blocks)
    partials, n_sel_r = phase_attend(backend, plan, views, row_pool, q, row_pos, ids, n_sel, k_cells, chunk_cells,
                                     n_chunks)
    out, lse = phase_merge(backend, all_gather(partials), all_gather(n_sel_r), len(row_pool), n_q_heads,
                           chunk_cells, n_chunks)
    return ids, n_sel, out, lse


def run_ranks_in_turn(backend, pools, row_pool, q, row_pos, n_q_heads: int, block_cells: int, k_cells: int,
                      chunk_cells: int, n_chunks: int, max_blocks: int, world: int):
    """All `world` ranks of one window in this process, one after another (each exchange is a list
    in rank order): the same phases and exchange contents as run_window on `world` GPUs."""
    fills = [backend.fill(p) for p in pools]
    pcs = [backend.page_cells(p) for p in pools]
    plans = [ShardPlan.make(fills, pcs, block_cells, r, world) for r in range(world)]
    views = [[backend.view(p, pl.first_page[i], pl.hi[i] - pl.lo[i]) for i, p in enumerate(pools)] for pl in plans]
    local = [phase_scores(backend, plans[r], views[r], row_pool, q, block_cells) for r in range(world)]
    ids, n_sel = phase_select(backend, plans, local, fills, row_pool, block_cells, k_cells, max_blocks)
    att = [phase_attend(backend, plans[r], views[r], row_pool, q, row_pos, ids, n_sel, k_cells, chunk_cells, n_chunks)
           for r in range(world)]
    out, lse = phase_merge(backend, [a[0] for a in att], [a[1] for a in att], len(row_pool), n_q_heads, chunk_cells,
                           n_chunks)
    return ids, n_sel, out, lse


class LibraryBackend:
    """The phases on this process's CUDA device through the library (pools are DevicePool objects,
    q / row_pos device tensors)."""

    def __init__(self, device="cuda"):
        import torch
        self.torch = torch
        self.device = torch.device(device)

    def fill(self, pool) -> int:
        return pool.n_filled

    def page_cells(self, pool) -> int:
        return pool.page_cells

    def view(self, pool, first_page: int, n_cells: int):
        from . import DevicePool
        return DevicePool(pool.k_codes, pool.v_codes, pool.k_scales, pool.v_scales, pool.page_table[first_page:],
                          n_filled=n_cells, capacity=n_cells, page_cells=pool.page_cells, n_kv_heads=pool.n_kv_heads,
                          v_bits=pool.v_bits, head_dim=pool.head_dim, k_bits=pool.k_bits, k_sums=pool.k_sums)

    def block_scores(self, views, row_pool, q, block_cells: int, local_blocks: int):
        from . import block_scores
        scores = self.torch.zeros((len(row_pool), local_blocks), dtype=self.torch.float32, device=self.device)
        if any(v.n_filled > 0 for v in views):
            block_scores(views, row_pool, q, block_cells, scores)
        return scores

    def topk_gathered(self, gathered, plans, fills, row_pool, block_cells: int, k_cells: int, max_blocks: int):
        from . import topk
        torch = self.torch
        R = len(row_pool)
        scores = torch.zeros((R, max_blocks), dtype=torch.float32, device=self.device)
        for s, g in enumerate(gathered):   # each rank's blocks into their columns of the whole row
            for t, pi in enumerate(row_pool):
                b0 = plans[s].lo[pi] // block_cells
                nb = (plans[s].hi[pi] - plans[s].lo[pi] + block_cells - 1) // block_cells
                if nb > 0:
                    scores[t, b0:b0 + nb] = g[t, :nb].to(self.device)
        ids = torch.zeros((R, max(k_cells, 1)), dtype=torch.int32, device=self.device)
        n_sel = torch.zeros((R,), dtype=torch.int32, device=self.device)
        topk(scores, [fills[pi] for pi in row_pool], block_cells, k_cells, ids, n_sel)
        self.last_scores = scores
        return ids, n_sel

    def ids_in_range(self, ids, n_sel, row_pos, lo, hi, k_cells: int):
        from . import _check, _i32_array, _ptr, _stream, load
        torch = self.torch
        R = len(lo)
        ids_r = torch.zeros_like(ids)
        n_sel_r = torch.zeros((R,), dtype=torch.int32, device=self.device)
        pos_r = torch.zeros((R,), dtype=torch.int32, device=self.device)
        _check(load().qsa_ids_in_range(_ptr(ids), _ptr(n_sel), _ptr(row_pos), R, k_cells, _i32_array(lo),
                                       _i32_array(hi), _ptr(ids_r), _ptr(n_sel_r), _ptr(pos_r), _stream(None)),
               "qsa_ids_in_range")
        return ids_r, n_sel_r, pos_r

    def decode_attn(self, views, row_pool, q, row_pos, ids, n_sel, k_cells: int, chunk_cells: int, n_chunks: int):
        from . import decode_attn, decode_partials_bytes
        R, Hq, _ = q.shape
        partials = self.torch.empty((decode_partials_bytes(R, Hq, n_chunks) // 4,), dtype=self.torch.float32,
                                    device=self.device)
        decode_attn(views, row_pool, q, row_pos, ids, n_sel, k_cells, chunk_cells, n_chunks, partials)
        return partials

    def merge_shards(self, gathered_partials, gathered_n_sel, n_rows: int, n_q_heads: int, chunk_cells: int,
                     n_chunks: int):
        from . import _check, _ptr, _stream, load
        torch = self.torch
        parts = torch.cat([p.to(self.device) for p in gathered_partials])
        nsel = torch.stack([n.to(self.device) for n in gathered_n_sel]).contiguous()
        out = torch.empty((n_rows, n_q_heads, 128), dtype=torch.float32, device=self.device)
        lse = torch.empty((n_rows, n_q_heads), dtype=torch.float32, device=self.device)
        _check(load().qsa_attn_merge_shards(_ptr(parts), len(gathered_partials), _ptr(nsel), n_rows, n_q_heads,
                                            chunk_cells, n_chunks, _ptr(out), _ptr(lse), _stream(None)),
               "qsa_attn_merge_shards")
        return out, lse


def torch_all_gather(x):
    """all_gather of one tensor of the same shape on every rank (torch.distributed, any backend)."""
    import torch
    import torch.distributed as dist
    out = [torch.empty_like(x) for _ in range(dist.get_world_size())]
    dist.all_gather(out, x.contiguous())
    return out
