"""The C-ABI library loads, exports every symbol include/qsa.h declares, and its
host-side validation rejects bad calls before anything is enqueued.  No test
here launches a kernel or needs a GPU."""
import ctypes
import os
import re

import pytest

import sparse_selection_attention_gb300 as qsa
from sparse_selection_attention_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return qsa.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "qsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("qsa_block_scores", "qsa_topk", "qsa_decode_attn", "qsa_attn_merge", "qsa_prompt_attn"):
        assert n in names
    assert sorted(qsa.EXPORTS) == sorted(names)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_pure_host_calls(lib):
    assert qsa.abi_version() == 109
    assert qsa.status_str(qsa.QSA_ERR_SCRATCH) == "scratch buffer too small"
    assert qsa.decode_partials_bytes(5, 24, 64) == 4 * 5 * 24 * 64 * 130
    # o starts at the next 256-byte boundary after the (m, l) pairs, whatever their count
    assert qsa.decode_partials_bytes(1, 1, 1) == 256 + 4 * 128
    assert qsa.decode_partials_bytes(1, 3, 3) == 256 + 4 * 9 * 128
    assert qsa.decode_partials_bytes(0, 24, 64) == 0


def _pool(**kw):
    base = dict(k_codes=16, v_codes=32, k_scales=48, v_scales=64, page_table=80, n_filled=100, capacity=256,
                page_cells=256, n_kv_heads=4, head_dim=128, v_bits=8, k_bits=8, k_sums=None)
    base.update(kw)
    return qsa.QsaPoolC(*[base[f] for f, _ in qsa.QsaPoolC._fields_])


def _scores_call(lib, pools, row_pool, R=2, Hq=24, B=64, q=16, scores=32, max_blocks=4):
    arr = (qsa.QsaPoolC * len(pools))(*pools)
    rp = (ctypes.c_int32 * len(row_pool))(*row_pool)
    return lib.qsa_block_scores(arr, len(pools), rp, q, R, Hq, B, scores, max_blocks, None)


def test_block_scores_validation(lib):
    ok_pool = _pool()
    assert _scores_call(lib, [_pool(k_codes=None)], [0, 0]) == qsa.QSA_ERR_ARG
    assert _scores_call(lib, [_pool(k_codes=17)], [0, 0]) == qsa.QSA_ERR_ARG          # misaligned
    assert _scores_call(lib, [_pool(head_dim=64)], [0, 0]) == qsa.QSA_ERR_UNSUPPORTED
    assert _scores_call(lib, [ok_pool], [0, 1]) == qsa.QSA_ERR_ARG                     # row -> missing pool
    assert _scores_call(lib, [ok_pool], [0, 0], Hq=25) == qsa.QSA_ERR_ARG              # Hq % Hkv
    assert _scores_call(lib, [ok_pool], [0, 0], Hq=40) == qsa.QSA_ERR_UNSUPPORTED      # group 10 > 8
    assert _scores_call(lib, [ok_pool], [0, 0], B=48) == qsa.QSA_ERR_ARG
    assert _scores_call(lib, [ok_pool], [0, 0], max_blocks=1) == qsa.QSA_ERR_ARG        # 2 blocks needed
    assert _scores_call(lib, [ok_pool] * 5, [0, 0]) == qsa.QSA_ERR_UNSUPPORTED          # > 4 pools


def test_topk_validation(lib):
    nf = (ctypes.c_int32 * 2)(100, 200)
    assert lib.qsa_topk(16, 4, nf, 2, 64, 100, 32, 48, None) == qsa.QSA_ERR_ARG    # k not multiple of B
    assert lib.qsa_topk(16, 3, nf, 2, 64, 128, 32, 48, None) == qsa.QSA_ERR_ARG    # 4 blocks > max_blocks 3
    assert lib.qsa_topk(None, 4, nf, 2, 64, 128, 32, 48, None) == qsa.QSA_ERR_ARG
    big = (ctypes.c_int32 * 1)(64 * 40000)
    assert lib.qsa_topk(16, 40000, big, 1, 64, 128, 32, 48, None) == qsa.QSA_ERR_UNSUPPORTED
    many = (ctypes.c_int32 * 33)(*([100] * 33))
    assert lib.qsa_topk(16, 4, many, 33, 64, 128, 32, 48, None) == qsa.QSA_ERR_UNSUPPORTED


def test_decode_attn_validation(lib):
    pools = (qsa.QsaPoolC * 1)(_pool())
    rp = (ctypes.c_int32 * 2)(0, 0)
    need = qsa.decode_partials_bytes(2, 24, 4)
    args = lambda **kw: [pools, 1, rp, 16, 32, 48, 64, 2, 24, kw.get("k", 256), kw.get("C", 64),
                         kw.get("n", 4), kw.get("part", 80), kw.get("nbytes", need), None]
    assert lib.qsa_decode_attn(*args(nbytes=need - 4)) == qsa.QSA_ERR_SCRATCH
    assert lib.qsa_decode_attn(*args(n=3)) == qsa.QSA_ERR_ARG          # fewer chunks than k / C
    assert lib.qsa_decode_attn(*args(C=40)) == qsa.QSA_ERR_ARG
    assert lib.qsa_decode_attn(*args(part=84)) == qsa.QSA_ERR_ARG      # misaligned scratch
    assert lib.qsa_decode_attn(*args(part=None)) == qsa.QSA_ERR_ARG
    assert lib.qsa_attn_merge(None, 16, 2, 24, 64, 4, 32, None, None) == qsa.QSA_ERR_ARG
    assert lib.qsa_attn_merge(16, 16, 2, 24, 40, 4, 32, None, None) == qsa.QSA_ERR_ARG


def test_prompt_validation(lib):
    pool = _pool(n_filled=1000, capacity=1024)
    need = lib.qsa_prompt_scratch_bytes(ctypes.byref(pool), 100, 900, 24)
    # one tile image per tile and head; no partial ranges without a device (its SM count decides them)
    assert need == 256 + 4 * (999 // 64 + 1) * 65536
    assert lib.qsa_prompt_scratch_bytes(ctypes.byref(_pool(v_bits=4, n_filled=1000, capacity=1024)), 100, 900, 24) == need
    assert lib.qsa_prompt_scratch_bytes(ctypes.byref(pool), 100, 900, 26) == 0      # not a multiple of the KV heads
    assert lib.qsa_prompt_scratch_bytes(ctypes.byref(pool), 0, 900, 24) == 0
    ok = dict(scratch=1 << 20, nbytes=need)

    def call(pl, q_pos0, n_q, Hq=24, scratch=None, nbytes=None):
        a = dict(ok, **({} if scratch is None else {"scratch": scratch}), **({} if nbytes is None else {"nbytes": nbytes}))
        return lib.qsa_prompt_attn(ctypes.byref(pl), 16, n_q, q_pos0, Hq, a["scratch"], a["nbytes"], 32, None, None)
    assert call(pool, 950, 100) == qsa.QSA_ERR_ARG                   # past n_filled
    assert call(pool, -1, 100) == qsa.QSA_ERR_ARG
    assert call(pool, 0, 100, Hq=26) == qsa.QSA_ERR_ARG               # not a multiple of the KV heads
    assert call(_pool(page_cells=96), 0, 10) == qsa.QSA_ERR_ARG       # pages of a multiple of 64 cells only
    assert call(pool, 0, 0) == qsa.QSA_OK                             # nothing to do
    assert call(pool, 900, 100, nbytes=need - 1) == qsa.QSA_ERR_SCRATCH
    assert call(pool, 900, 100, scratch=(1 << 20) + 16) == qsa.QSA_ERR_SCRATCH   # not 256-byte aligned
    assert lib.qsa_prompt_attn(ctypes.byref(pool), 16, 100, 900, 24, None, need, 32, None, None) == qsa.QSA_ERR_SCRATCH

def test_kv_append_validation(lib):
    pool = _pool(n_filled=100, capacity=256)
    call = lambda pl, first, n, k=16, v=32: lib.qsa_kv_append(ctypes.byref(pl), k, v, first, n, None)
    assert call(pool, 200, 57) == qsa.QSA_ERR_ARG                   # past the capacity
    assert call(pool, -1, 1) == qsa.QSA_ERR_ARG
    assert call(pool, 0, -1) == qsa.QSA_ERR_ARG
    assert call(pool, 10, 5, k=24) == qsa.QSA_ERR_ARG               # k not 16-byte aligned
    assert call(pool, 10, 5, v=0) == qsa.QSA_ERR_ARG                # v missing
    assert call(_pool(page_cells=96), 0, 1) == qsa.QSA_ERR_ARG       # pages of a multiple of 64 cells only
    assert call(_pool(head_dim=64), 0, 1) == qsa.QSA_ERR_UNSUPPORTED
    assert call(pool, 200, 0) == qsa.QSA_OK                          # nothing to append: nothing launched


def test_four_bit_k_validation(lib):
    """4-bit K (k_bits 4) is served by every call; k_bits other than 8 and 4 is an argument error; the
    pools of one call share k_bits (checked before anything is launched)."""
    k4 = _pool(k_bits=4, v_bits=4)
    assert _scores_call(lib, [_pool(k_bits=5)], [0, 0]) == qsa.QSA_ERR_ARG
    assert _scores_call(lib, [_pool(), k4], [0, 1]) == qsa.QSA_ERR_ARG          # mixed k_bits in one call


def test_chunk_cap_and_noalloc_refusals(lib):
    """Chunk counts past QSA_MAX_CHUNKS are refused by the attention, the merge and the no-allocation
    entry point alike; the no-allocation call checks every argument of both of its steps (a NULL out
    among them) before it looks anything up or enqueues anything."""
    pools = (qsa.QsaPoolC * 1)(_pool(n_filled=256, capacity=256))
    rp = (ctypes.c_int32 * 1)(0)
    cap = qsa.QSA_MAX_CHUNKS
    k = 16 * (cap + 1)
    need = qsa.decode_partials_bytes(1, 4, cap + 1)
    assert lib.qsa_decode_attn(pools, 1, rp, 16, 32, 48, 64, 1, 4, k, 16, cap + 1, 256, need, None) == \
        qsa.QSA_ERR_UNSUPPORTED
    assert lib.qsa_attn_merge(256, 64, 1, 4, 16, cap + 1, 512, None, None) == qsa.QSA_ERR_UNSUPPORTED
    assert lib.qsa_attn_merge(260, 64, 1, 4, 16, 4, 512, None, None) == qsa.QSA_ERR_ARG   # misaligned partials
    noalloc = lambda out, k_cells, C=16, Hq=4: lib.qsa_decode_attn_noalloc(pools, 1, rp, 16, 32, 48, 64, 1, Hq,
                                                                        k_cells, C, out, None, None)
    assert noalloc(None, 256) == qsa.QSA_ERR_ARG
    assert noalloc(512, 200000) == qsa.QSA_ERR_UNSUPPORTED      # 12,500 chunks of 16 cells
    assert noalloc(512, 2 ** 31 - 1, C=1024) == qsa.QSA_ERR_UNSUPPORTED   # no int overflow in the chunk count
    assert noalloc(512, 16 * cap, Hq=8) == qsa.QSA_ERR_SCRATCH  # 8 x 8,192 chunks of partials > 8 MiB


def test_tc_rate_validation(lib):
    """Argument checks of the rate measurement, taken before anything is launched."""
    r = ctypes.c_double(0.0)
    assert lib.qsa_measure_tc_rate(2, 10, ctypes.byref(r)) == qsa.QSA_ERR_ARG
    assert lib.qsa_measure_tc_rate(qsa.QSA_TC_KIND_I8, 0, ctypes.byref(r)) == qsa.QSA_ERR_ARG
    assert lib.qsa_measure_tc_rate(qsa.QSA_TC_KIND_F16, 10, None) == qsa.QSA_ERR_ARG


def test_window_host_refuses_buffers_that_are_not_page_locked(lib):
    """qsa_decode_window_host takes q, row_pos, out and lse in page-locked host memory only: pageable
    host arrays (and NULL) are refused with QSA_ERR_ARG before the pools are even looked at."""
    q = (ctypes.c_float * (2 * 128))()
    pos = (ctypes.c_int32 * 1)()
    out = (ctypes.c_float * (2 * 128))()
    addr = lambda a: ctypes.cast(a, ctypes.c_void_p).value
    call = lambda qq, pp, oo: lib.qsa_decode_window_host(None, 1, None, qq, pp, 1, 2, 64, 64, None, 1, None, None, oo,
                                                         None, None, 0, None)
    assert call(addr(q), addr(pos), addr(out)) == qsa.QSA_ERR_ARG
    assert call(None, addr(pos), addr(out)) == qsa.QSA_ERR_ARG
    assert call(addr(q), addr(pos), None) == qsa.QSA_ERR_ARG
