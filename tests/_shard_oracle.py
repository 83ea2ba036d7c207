"""The context-sharded decode phases on the FP64 oracle (numpy pools): the backend the gloo tests
run through sparse_selection_attention_gb300.sharded, so that the orchestration (pool views, the
exchanges, the merge order) is checked on CPU against the oracle's unsharded window."""
import dataclasses

import numpy as np

import oracle as O


class OracleBackend:
    def fill(self, pool):
        return pool.n_filled

    def page_cells(self, pool):
        return pool.page_cells

    def view(self, pool, first_page, n_cells):
        return dataclasses.replace(pool, page_table=pool.page_table[first_page:], n_filled=n_cells,
                                   capacity=n_cells)

    def block_scores(self, views, row_pool, q, block_cells, local_blocks):
        out = np.zeros((len(row_pool), local_blocks), np.float32)
        for pi, v in enumerate(views):
            rows = [t for t, p in enumerate(row_pool) if p == pi]
            if rows and v.n_filled > 0:
                s = O.block_scores(v, q[rows], block_cells).astype(np.float32)
                out[rows, :s.shape[1]] = s
        return out

    def topk_gathered(self, gathered, plans, fills, row_pool, block_cells, k_cells, max_blocks):
        R = len(row_pool)
        scores = np.zeros((R, max_blocks), np.float32)
        for s, g in enumerate(gathered):
            for t, pi in enumerate(row_pool):
                b0 = plans[s].lo[pi] // block_cells
                nb = (plans[s].hi[pi] - plans[s].lo[pi] + block_cells - 1) // block_cells
                scores[t, b0:b0 + nb] = g[t, :nb]
        ids = np.zeros((R, max(k_cells, 1)), np.int64)
        n_sel = np.zeros(R, np.int64)
        for t, pi in enumerate(row_pool):
            sel, n = O.topk_select(scores[t], fills[pi], block_cells, k_cells)
            ids[t, :n] = sel
            n_sel[t] = n
        self.last_scores = scores
        return ids, n_sel

    def ids_in_range(self, ids, n_sel, row_pos, lo, hi, k_cells):
        R = len(lo)
        ids_r = np.zeros_like(ids)
        n_r = np.zeros(R, np.int64)
        for t in range(R):
            sel = ids[t, :n_sel[t]]
            keep = sel[(sel >= lo[t]) & (sel < hi[t])] - lo[t]
            ids_r[t, :len(keep)] = keep
            n_r[t] = len(keep)
        pos_r = np.asarray(row_pos, np.int64) - np.asarray(lo, np.int64)
        return ids_r, n_r, pos_r

    def decode_attn(self, views, row_pool, q, row_pos, ids, n_sel, k_cells, chunk_cells, n_chunks):
        R, Hq, D = q.shape
        m = np.full((R, Hq, n_chunks), -np.inf)
        l = np.zeros((R, Hq, n_chunks))
        o = np.zeros((R, Hq, n_chunks, D))
        for t, pi in enumerate(row_pool):
            m[t], l[t], o[t] = O.chunk_partials(views[pi], q[t], int(row_pos[t]), ids[t, :n_sel[t]], chunk_cells,
                                                n_chunks)
        return (m, l, o)

    def merge_shards(self, gathered_partials, gathered_n_sel, n_rows, n_q_heads, chunk_cells, n_chunks):
        m = np.concatenate([g[0] for g in gathered_partials], axis=2)   # rank order, then chunk order
        l = np.concatenate([g[1] for g in gathered_partials], axis=2)
        o = np.concatenate([g[2] for g in gathered_partials], axis=2)
        out = np.zeros((n_rows, n_q_heads, o.shape[-1]))
        lse = np.zeros((n_rows, n_q_heads))
        for t in range(n_rows):
            out[t], lse[t] = O.merge_partials(m[t], l[t], o[t])
        return out, lse
