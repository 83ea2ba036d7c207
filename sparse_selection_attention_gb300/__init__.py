"""Python binding of the GB300 QSA attention library (``libqsa_gb300.so``).

Argument marshalling only: every function here forwards device pointers,
sizes and the current CUDA stream to the C ABI declared in ``include/qsa.h``,
where all of the computation runs in CUDA kernels.  There is no fallback: if
the library is missing or a call fails, an exception is raised.
PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqsa_gb300.so")

QSA_OK, QSA_ERR_ARG, QSA_ERR_UNSUPPORTED, QSA_ERR_SCRATCH, QSA_ERR_CUDA, QSA_ERR_DEVICE = range(6)
QSA_MAX_CHUNKS = 8192   # chunks per (row, q head) of the chunk partials (qsa.h)
HEAD_DIM = 128
MAX_POOLS = 4
MAX_DECODE_ROWS = 32

EXPORTS = [
    "qsa_block_scores", "qsa_topk", "qsa_decode_partials_bytes", "qsa_decode_attn", "qsa_attn_merge",
    "qsa_prompt_attn", "qsa_prompt_scratch_bytes", "qsa_get_device_error", "qsa_set_wait_limit_ns", "qsa_status_str", "qsa_abi_version",
    "qsa_decode_attn_noalloc", "qsa_decode_window", "qsa_decode_window_workspace_bytes",
    "qsa_decode_window_profile", "qsa_kv_append", "qsa_measure_tc_rate", "qsa_ids_in_range",
    "qsa_attn_merge_shards", "qsa_kv_summarise", "qsa_decode_window_host",
]
QSA_TC_KIND_F16, QSA_TC_KIND_I8 = 0, 1
NOALLOC_SCRATCH_BYTES = 8 << 20


class QsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} (status {status})")


class QsaPoolC(ctypes.Structure):
    _fields_ = [
        ("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
        ("n_filled", ctypes.c_int32), ("capacity", ctypes.c_int32), ("page_cells", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("v_bits", ctypes.c_int32),
        ("k_bits", ctypes.c_int32), ("k_sums", ctypes.c_void_p),
    ]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (build it first with ``_build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"QSA CUDA library not built: {path} is missing; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    i, p, sz, u64 = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint64
    pool_p = ctypes.POINTER(QsaPoolC)
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.qsa_block_scores.argtypes = [pool_p, i, i32p, p, i, i, i, p, i, p]
    lib.qsa_topk.argtypes = [p, i, i32p, i, i, i, p, p, p]
    lib.qsa_decode_partials_bytes.argtypes = [i, i, i]
    lib.qsa_decode_partials_bytes.restype = sz
    lib.qsa_decode_attn.argtypes = [pool_p, i, i32p, p, p, p, p, i, i, i, i, i, p, sz, p]
    lib.qsa_attn_merge.argtypes = [p, p, i, i, i, i, p, p, p]
    lib.qsa_prompt_attn.argtypes = [pool_p, p, i, i, i, p, sz, p, p, p]
    lib.qsa_prompt_scratch_bytes.argtypes = [pool_p, i, i, i]
    lib.qsa_prompt_scratch_bytes.restype = sz
    lib.qsa_decode_attn_noalloc.argtypes = [pool_p, i, i32p, p, p, p, p, i, i, i, i, p, p, p]
    lib.qsa_decode_window.argtypes = [pool_p, i, i32p, p, p, i, i, i, i, p, i, p, p, p, p, p, sz, p]
    lib.qsa_decode_window_profile.argtypes = [pool_p, i, i32p, p, p, i, i, i, i, p, i, p, p, p, p, p, sz, p,
                                              ctypes.POINTER(ctypes.c_float)]
    lib.qsa_decode_window_host.argtypes = [pool_p, i, i32p, p, p, i, i, i, i, p, i, p, p, p, p, p, sz, p]
    lib.qsa_decode_window_workspace_bytes.argtypes = [i, i, i, i]
    lib.qsa_decode_window_workspace_bytes.restype = sz
    lib.qsa_kv_append.argtypes = [pool_p, p, p, i, i, p]
    lib.qsa_get_device_error.argtypes = [i32p, p]
    lib.qsa_set_wait_limit_ns.argtypes = [u64]
    lib.qsa_set_wait_limit_ns.restype = None
    lib.qsa_status_str.argtypes = [i]
    lib.qsa_status_str.restype = ctypes.c_char_p
    lib.qsa_abi_version.argtypes = []
    lib.qsa_measure_tc_rate.argtypes = [i, i, ctypes.POINTER(ctypes.c_double)]
    lib.qsa_ids_in_range.argtypes = [p, p, p, i, i, i32p, i32p, p, p, p, p]
    lib.qsa_attn_merge_shards.argtypes = [p, i, p, i, i, i, i, p, p, p]
    lib.qsa_kv_summarise.argtypes = [pool_p, i, i, p]
    for name in ("qsa_block_scores", "qsa_topk", "qsa_decode_attn", "qsa_attn_merge", "qsa_prompt_attn",
                 "qsa_get_device_error", "qsa_abi_version", "qsa_decode_attn_noalloc", "qsa_decode_window",
                 "qsa_decode_window_profile", "qsa_measure_tc_rate", "qsa_ids_in_range", "qsa_attn_merge_shards",
                 "qsa_kv_summarise", "qsa_decode_window_host"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def status_str(status: int) -> str:
    return load().qsa_status_str(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != QSA_OK:
        raise QsaError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the QSA library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _i32_array(values: Sequence[int]):
    arr = (ctypes.c_int32 * len(values))(*[int(v) for v in values])
    return arr


class DevicePool:
    """One slot's paged KV pool resident on the GPU (layout of include/qsa.h)."""

    def __init__(self, k_codes, v_codes, k_scales, v_scales, page_table, *, n_filled, capacity, page_cells,
                 n_kv_heads, v_bits, head_dim=HEAD_DIM, k_bits=8, k_sums=None):
        self.k_codes, self.v_codes = k_codes, v_codes
        self.k_scales, self.v_scales, self.page_table = k_scales, v_scales, page_table
        self.n_filled, self.capacity, self.page_cells = int(n_filled), int(capacity), int(page_cells)
        self.n_kv_heads, self.v_bits, self.head_dim = int(n_kv_heads), int(v_bits), int(head_dim)
        self.k_bits = int(k_bits)
        self.k_sums = k_sums   # optional block summaries, fp32 [pages][heads][page_cells / 64][128]

    def keep_block_sums(self, stream=None) -> "DevicePool":
        """Allocates the pool's block summaries and builds them for cells 0 .. n_filled - 1; later
        qsa_kv_append calls keep them current."""
        n_pages = self.k_codes.shape[0]
        self.k_sums = torch.zeros((n_pages, self.n_kv_heads, self.page_cells // 64, HEAD_DIM), dtype=torch.float32,
                                  device=self.k_codes.device)
        if self.n_filled > 0:
            kv_summarise(self, 0, self.n_filled, stream)
        return self

    @classmethod
    def upload(cls, pool, device="cuda") -> "DevicePool":
        """Copies a host pool (numpy arrays with the same field names) to the device."""
        t = lambda a: torch.from_numpy(a).to(device)
        return cls(t(pool.k_codes), t(pool.v_codes), t(pool.k_scales), t(pool.v_scales), t(pool.page_table),
                   n_filled=pool.n_filled, capacity=pool.capacity, page_cells=pool.page_cells,
                   n_kv_heads=pool.n_kv_heads, v_bits=pool.v_bits, head_dim=pool.head_dim,
                   k_bits=getattr(pool, "k_bits", 8))

    def c(self) -> QsaPoolC:
        return QsaPoolC(_ptr(self.k_codes), _ptr(self.v_codes), _ptr(self.k_scales), _ptr(self.v_scales),
                        _ptr(self.page_table), self.n_filled, self.capacity, self.page_cells, self.n_kv_heads,
                        self.head_dim, self.v_bits, self.k_bits, _ptr(self.k_sums))


def kv_append(pool: DevicePool, k: torch.Tensor, v: torch.Tensor, first_cell: int, stream=None) -> None:
    """Quantises the new cells' K and V rows (fp32 [n_new][n_kv_heads][128]) into the pool at cells
    first_cell .. first_cell + n_new - 1, then raises the host-side pool.n_filled to cover them."""
    n_new = k.shape[0]
    pc = pool.c()
    _check(load().qsa_kv_append(ctypes.byref(pc), _ptr(k), _ptr(v), int(first_cell), n_new, _stream(stream)),
           "qsa_kv_append")
    pool.n_filled = max(pool.n_filled, int(first_cell) + n_new)


def kv_summarise(pool: DevicePool, first_cell: int, n_cells: int, stream=None) -> None:
    """qsa_kv_summarise: rewrites the pool's block summaries of the 64-cell blocks the cells
    first_cell .. first_cell + n_cells - 1 fall in."""
    pc = pool.c()
    _check(load().qsa_kv_summarise(ctypes.byref(pc), int(first_cell), int(n_cells), _stream(stream)),
           "qsa_kv_summarise")


def _pools_c(pools: Sequence[DevicePool]):
    arr = (QsaPoolC * len(pools))(*[p.c() for p in pools])
    return arr


def block_scores(pools: Sequence[DevicePool], row_pool: Sequence[int], q: torch.Tensor, block_cells: int,
                 scores: torch.Tensor, stream=None) -> None:
    R, Hq, _ = q.shape
    _check(load().qsa_block_scores(_pools_c(pools), len(pools), _i32_array(row_pool), _ptr(q), R, Hq,
                                   block_cells, _ptr(scores), scores.shape[1], _stream(stream)), "qsa_block_scores")


def topk(scores: torch.Tensor, n_filled: Sequence[int], block_cells: int, k_cells: int, ids: torch.Tensor,
         n_sel: torch.Tensor, stream=None) -> None:
    R = len(n_filled)
    _check(load().qsa_topk(_ptr(scores), scores.shape[1], _i32_array(n_filled), R, block_cells, k_cells,
                           _ptr(ids), _ptr(n_sel), _stream(stream)), "qsa_topk")


def partials_o_offset(n: int) -> int:
    """Byte offset of o in a chunk-partials buffer of n (row, head, chunk) entries (qsa.h layout)."""
    return (8 * n + 255) // 256 * 256


def decode_partials_bytes(n_rows: int, n_q_heads: int, n_chunks: int) -> int:
    return int(load().qsa_decode_partials_bytes(n_rows, n_q_heads, n_chunks))


def decode_attn(pools: Sequence[DevicePool], row_pool: Sequence[int], q: torch.Tensor, row_pos: torch.Tensor,
                ids: torch.Tensor, n_sel: torch.Tensor, k_cells: int, chunk_cells: int, n_chunks: int,
                partials: torch.Tensor, stream=None) -> None:
    R, Hq, _ = q.shape
    _check(load().qsa_decode_attn(_pools_c(pools), len(pools), _i32_array(row_pool), _ptr(q), _ptr(row_pos),
                                  _ptr(ids), _ptr(n_sel), R, Hq, k_cells, chunk_cells, n_chunks, _ptr(partials),
                                  partials.numel() * partials.element_size(), _stream(stream)), "qsa_decode_attn")


def attn_merge(partials: torch.Tensor, n_sel: torch.Tensor, n_rows: int, n_q_heads: int, chunk_cells: int,
               n_chunks: int, out: torch.Tensor, lse: Optional[torch.Tensor] = None, stream=None) -> None:
    _check(load().qsa_attn_merge(_ptr(partials), _ptr(n_sel), n_rows, n_q_heads, chunk_cells, n_chunks, _ptr(out),
                                 _ptr(lse), _stream(stream)), "qsa_attn_merge")


def prompt_scratch_bytes(pool: DevicePool, n_q: int, q_pos0: int, n_q_heads: int) -> int:
    """Scratch bytes of a prompt call on the current device (0 for invalid arguments)."""
    pc = pool.c()
    return int(load().qsa_prompt_scratch_bytes(ctypes.byref(pc), n_q, q_pos0, n_q_heads))


def prompt_attn(pool: DevicePool, q: torch.Tensor, q_pos0: int, out: torch.Tensor,
                lse: Optional[torch.Tensor] = None, scratch: Optional[torch.Tensor] = None, stream=None) -> None:
    """Causal prompt attention.  `scratch` (uint8, device) must hold prompt_scratch_bytes(); when it is
    None a buffer of that size is allocated for this call."""
    n_q, Hq, _ = q.shape
    pc = pool.c()
    if scratch is None:
        need = prompt_scratch_bytes(pool, n_q, q_pos0, Hq)
        scratch = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(load().qsa_prompt_attn(ctypes.byref(pc), _ptr(q), n_q, q_pos0, Hq, _ptr(scratch), scratch.numel(),
                                  _ptr(out), _ptr(lse), _stream(stream)), "qsa_prompt_attn")


def decode_attn_noalloc(pools: Sequence[DevicePool], row_pool: Sequence[int], q: torch.Tensor,
                        row_pos: torch.Tensor, ids: torch.Tensor, n_sel: torch.Tensor, k_cells: int,
                        chunk_cells: int, out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                        stream=None) -> None:
    """Chunk attention + merge with the library's own fixed scratch, for callers that cannot allocate
    device memory (an engine whose memory is all reserved up front, a plugin with no allocator).
    Calls that overlap on the GPU share that scratch and race; the first call on a device should come
    before any stream capture."""
    R, Hq, _ = q.shape
    _check(load().qsa_decode_attn_noalloc(_pools_c(pools), len(pools), _i32_array(row_pool), _ptr(q),
                                          _ptr(row_pos), _ptr(ids), _ptr(n_sel), R, Hq, k_cells, chunk_cells,
                                          _ptr(out), _ptr(lse), _stream(stream)), "qsa_decode_attn_noalloc")


def get_device_error(stream=None) -> int:
    code = ctypes.c_int32(0)
    st = load().qsa_get_device_error(ctypes.byref(code), _stream(stream))
    if st not in (QSA_OK, QSA_ERR_DEVICE):
        raise QsaError(st, "qsa_get_device_error")
    return int(code.value)


def set_wait_limit_ns(ns: int) -> None:
    load().qsa_set_wait_limit_ns(int(ns))


def measure_tc_rate(kind: int, passes: int = 10000) -> float:
    """qsa_measure_tc_rate: dense tcgen05 operations per second of this GPU for QSA_TC_KIND_I8 or
    QSA_TC_KIND_F16 (synchronous; a few milliseconds)."""
    r = ctypes.c_double(0.0)
    _check(load().qsa_measure_tc_rate(int(kind), int(passes), ctypes.byref(r)), "qsa_measure_tc_rate")
    return float(r.value)


def abi_version() -> int:
    return int(load().qsa_abi_version())


class DecodeWindow:
    """Device buffers of one decode window and the four calls of its hot path
    (block scores -> top-k -> chunk attention -> merge), all on one stream."""

    def __init__(self, pools: List[DevicePool], row_pool: Sequence[int], n_q_heads: int, block_cells: int,
                 k_cells: int, chunk_cells: int, n_chunks: Optional[int] = None, max_blocks: Optional[int] = None,
                 device="cuda"):
        self.pools, self.row_pool = pools, [int(x) for x in row_pool]
        self.n_rows, self.n_q_heads = len(self.row_pool), int(n_q_heads)
        self.block_cells, self.k_cells, self.chunk_cells = int(block_cells), int(k_cells), int(chunk_cells)
        self.n_chunks = int(n_chunks or (k_cells + chunk_cells - 1) // chunk_cells)
        cap = max(p.capacity for p in pools)
        self.max_blocks = int(max_blocks or (cap + block_cells - 1) // block_cells)
        self.n_filled = [pools[p].n_filled for p in self.row_pool]
        R = self.n_rows
        self.scores = torch.zeros((R, self.max_blocks), dtype=torch.float32, device=device)
        self.ids = torch.zeros((R, max(self.k_cells, 1)), dtype=torch.int32, device=device)
        self.n_sel = torch.zeros((R,), dtype=torch.int32, device=device)
        nbytes = decode_partials_bytes(R, self.n_q_heads, self.n_chunks)
        self.partials = torch.zeros((nbytes // 4,), dtype=torch.float32, device=device)
        self.out = torch.zeros((R, self.n_q_heads, HEAD_DIM), dtype=torch.float32, device=device)
        self.lse = torch.zeros((R, self.n_q_heads), dtype=torch.float32, device=device)

        # ctypes arguments that do not change between steps, built once.
        self._c_pools = _pools_c(pools)
        self._c_row_pool = _i32_array(self.row_pool)
        self._c_n_filled = _i32_array(self.n_filled)
        self._nbytes = nbytes
        self._ws = None

    def scores_step(self, q: torch.Tensor, stream=None) -> None:
        _check(load().qsa_block_scores(self._c_pools, len(self.pools), self._c_row_pool, _ptr(q), self.n_rows,
                                       self.n_q_heads, self.block_cells, self.scores.data_ptr(), self.max_blocks,
                                       _stream(stream)), "qsa_block_scores")

    def topk_step(self, stream=None) -> None:
        _check(load().qsa_topk(self.scores.data_ptr(), self.max_blocks, self._c_n_filled, self.n_rows,
                               self.block_cells, self.k_cells, self.ids.data_ptr(), self.n_sel.data_ptr(),
                               _stream(stream)), "qsa_topk")

    def attn_step(self, q: torch.Tensor, row_pos: torch.Tensor, stream=None) -> None:
        _check(load().qsa_decode_attn(self._c_pools, len(self.pools), self._c_row_pool, _ptr(q), _ptr(row_pos),
                                      self.ids.data_ptr(), self.n_sel.data_ptr(), self.n_rows, self.n_q_heads,
                                      self.k_cells, self.chunk_cells, self.n_chunks, self.partials.data_ptr(),
                                      self._nbytes, _stream(stream)), "qsa_decode_attn")

    def merge_step(self, stream=None) -> None:
        _check(load().qsa_attn_merge(self.partials.data_ptr(), self.n_sel.data_ptr(), self.n_rows, self.n_q_heads,
                                     self.chunk_cells, self.n_chunks, self.out.data_ptr(), self.lse.data_ptr(),
                                     _stream(stream)), "qsa_attn_merge")

    def run_window(self, q: torch.Tensor, row_pos: torch.Tensor, stream=None) -> None:
        """The whole window in one call (qsa_decode_window): scores, ids, n_sel, out and lse."""
        _check(load().qsa_decode_window(*self._window_args(q, row_pos, stream)), "qsa_decode_window")

    def run_window_host(self, q_host: torch.Tensor, row_pos_host: torch.Tensor, out_host: torch.Tensor,
                        lse_host: Optional[torch.Tensor] = None, stream=None) -> None:
        """qsa_decode_window_host: the window with q, row_pos, out and lse in page-locked host memory
        (CPU tensors with pin_memory()); scores, ids and n_sel stay on the device.  The results are in
        out_host / lse_host once the stream has run the call."""
        for t in (q_host, row_pos_host, out_host) + ((lse_host,) if lse_host is not None else ()):
            if t.device.type != "cpu" or not t.is_pinned() or not t.is_contiguous():
                raise ValueError("run_window_host takes contiguous page-locked CPU tensors")
        args = list(self._window_args(self.out, self.out, stream))
        args[3], args[4] = q_host.data_ptr(), row_pos_host.data_ptr()
        args[13], args[14] = out_host.data_ptr(), (lse_host.data_ptr() if lse_host is not None else None)
        _check(load().qsa_decode_window_host(*args), "qsa_decode_window_host")

    def _window_args(self, q, row_pos, stream):
        if self._ws is None:
            nbytes = int(load().qsa_decode_window_workspace_bytes(self.n_rows, self.n_q_heads,
                                                                  self.pools[0].n_kv_heads, self.k_cells))
            self._ws = torch.empty((max(nbytes, 256),), dtype=torch.uint8, device=self.out.device)
        return (self._c_pools, len(self.pools), self._c_row_pool, _ptr(q), _ptr(row_pos), self.n_rows,
                self.n_q_heads, self.block_cells, self.k_cells, self.scores.data_ptr(), self.max_blocks,
                self.ids.data_ptr(), self.n_sel.data_ptr(), self.out.data_ptr(), self.lse.data_ptr(),
                self._ws.data_ptr(), self._ws.numel(), _stream(stream))

    def run_window_profile(self, q: torch.Tensor, row_pos: torch.Tensor, stream=None) -> List[float]:
        """qsa_decode_window_profile: the window's five launches without overlap; returns their times in
        microseconds (q fragments, block scores, top-k, split attention, merge).  Synchronises."""
        us = (ctypes.c_float * 5)()
        _check(load().qsa_decode_window_profile(*self._window_args(q, row_pos, stream), us),
               "qsa_decode_window_profile")
        return [float(x) for x in us]

    def run(self, q: torch.Tensor, row_pos: torch.Tensor, stream=None) -> None:
        """block scores -> top-k -> chunk attention -> merge, enqueued on one stream."""
        self.scores_step(q, stream)
        self.topk_step(stream)
        self.attend(q, row_pos, stream)

    def attend(self, q: torch.Tensor, row_pos: torch.Tensor, stream=None) -> None:
        self.attn_step(q, row_pos, stream)
        self.merge_step(stream)

    def partial_views(self):
        """(ml [R, Hq, n_chunks, 2], o [R, Hq, n_chunks, 128]) views of the partials buffer."""
        R, H, n = self.n_rows, self.n_q_heads, self.n_chunks
        o0 = partials_o_offset(R * H * n) // 4
        ml = self.partials[: R * H * n * 2].view(R, H, n, 2)
        o = self.partials[o0:o0 + R * H * n * HEAD_DIM].view(R, H, n, HEAD_DIM)
        return ml, o
