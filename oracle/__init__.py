"""ctypes wrapper of the CPU oracle (``liboracle.so``).

TEST INFRASTRUCTURE ONLY: imported by the test-suite, by the package smoke
check and by the benchmark's CPU-baseline leg.  The product path never
imports it.  All arrays are numpy arrays in host memory.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

BF16, FP8, MXFP4 = 0, 1, 2
MX_FIELD_BYTES = 8704
FP8_INDEX_FIELD_BYTES = 16896
BF16_INDEX_FIELD_BYTES = 32768

_lib = None


def lib():
    """The oracle library: the built ``liboracle.so``, or the library named by
    ``BSP_ORACLE_LIB`` (the planted-mistake test loads variants of the oracle
    this way)."""
    global _lib
    if _lib is None:
        path = os.environ.get("BSP_ORACLE_LIB") or _build.build()
        _lib = C.CDLL(path)
        _declare(_lib)
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def _declare(L):
    vp, i32, i64, f32 = C.c_void_p, C.c_int, C.c_int64, C.c_float
    L.orc_e4m3_encode.argtypes = [f32]
    L.orc_e4m3_encode.restype = C.c_uint8
    L.orc_e4m3_decode.argtypes = [C.c_uint8]
    L.orc_e4m3_decode.restype = C.c_double
    L.orc_e2m1_encode.argtypes = [C.c_double]
    L.orc_e2m1_encode.restype = C.c_uint8
    L.orc_e2m1_decode.argtypes = [C.c_uint8]
    L.orc_e2m1_decode.restype = C.c_double
    L.orc_e8m0_decode.argtypes = [C.c_uint8]
    L.orc_e8m0_decode.restype = C.c_double
    L.orc_bf16_encode.argtypes = [f32]
    L.orc_bf16_encode.restype = C.c_uint16
    L.orc_bf16_decode.argtypes = [C.c_uint16]
    L.orc_bf16_decode.restype = f32
    L.orc_mx_scale_byte.argtypes = [vp, i32]
    L.orc_mx_scale_byte.restype = C.c_uint8
    L.orc_cast_e4m3.argtypes = [vp, vp, i64]
    L.orc_kv_block_bytes.argtypes = [i32, i32]
    L.orc_kv_block_bytes.restype = i64
    L.orc_index_field_bytes.argtypes = [i32]
    L.orc_index_field_bytes.restype = i64
    L.orc_l1_offset.argtypes = [i32, i32, i32, i64, i32, i32, i32]
    L.orc_l1_offset.restype = i64
    L.orc_mx_field_offset.argtypes = [i32, i64, i32, i32]
    L.orc_mx_field_offset.restype = i64
    L.orc_kv_page_write.argtypes = [i32, i32, vp, f32, f32, i32, i32, vp, vp, vp, vp, vp, i32]
    L.orc_row_lengths_decode.argtypes = [vp, i32, i32, i32, vp, vp]
    L.orc_row_lengths_prefill.argtypes = [vp, vp, i32, i32, vp, vp]
    L.orc_index_score.argtypes = [i32, i32, vp, i64, vp, i32, vp, i32, vp, vp, i32, i32, vp, vp, vp, i32]
    L.orc_topk_select.argtypes = [vp, i32, i32, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, i32]
    L.orc_topk_select_blocks.argtypes = [vp, i32, i32, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, i32]
    L.orc_sparse_attention.argtypes = [i32, i32, vp, f32, f32, vp, i32, i32, vp, vp, i32, i32, f32, vp, vp, i32]
    L.orc_dense_attention.argtypes = [i32, i32, vp, f32, f32, vp, i32, i32, vp, i32, vp, vp, i32, f32, vp, vp, i32]
    L.orc_num_threads.restype = i32
    L.orc_set_num_threads.argtypes = [i32]
    L.orc_set_num_threads.restype = None


def _subset(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(rows, dtype=np.int32)
    return r, len(r)


# ---- codecs ---------------------------------------------------------------
def e4m3_encode(x):
    return int(lib().orc_e4m3_encode(float(x)))


def e4m3_decode(b):
    return float(lib().orc_e4m3_decode(int(b)))


def e2m1_encode(x):
    return int(lib().orc_e2m1_encode(float(x)))


def e2m1_decode(n):
    return float(lib().orc_e2m1_decode(int(n)))


def e8m0_decode(b):
    return float(lib().orc_e8m0_decode(int(b)))


def bf16_encode(x):
    return int(lib().orc_bf16_encode(float(x)))


def bf16_decode(b):
    return float(lib().orc_bf16_decode(int(b)))


def mx_scale_byte(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    return int(lib().orc_mx_scale_byte(_p(x), len(x)))


def cast_e4m3(x_bf16):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_cast_e4m3(_p(x), _p(out), x.size)
    return out


# ---- layouts --------------------------------------------------------------
def kv_block_bytes(kv_dtype, hkv):
    return int(lib().orc_kv_block_bytes(kv_dtype, hkv))


def index_field_bytes(idx_dtype):
    return int(lib().orc_index_field_bytes(idx_dtype))


def l1_offset(kv_dtype, hkv, side, page_id, h, t, d):
    return int(lib().orc_l1_offset(kv_dtype, hkv, side, page_id, h, t, d))


def mx_field_offset(hkv, block, side, h):
    return int(lib().orc_mx_field_offset(hkv, block, side, h))


# ---- pipeline steps -------------------------------------------------------
def kv_page_write(kv_dtype, hkv, kv_cache, k_scale, v_scale, idx_dtype, hidx, idx_cache, k, v, idx_k, slot):
    """In place: kv_cache / idx_cache are uint8 numpy buffers."""
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    ik = None if idx_k is None else np.ascontiguousarray(idx_k, dtype=np.uint16)
    slot = np.ascontiguousarray(slot, dtype=np.int64)
    lib().orc_kv_page_write(kv_dtype, hkv, _p(kv_cache), k_scale, v_scale, idx_dtype, hidx,
                            _p(idx_cache), _p(k), _p(v), _p(ik), _p(slot), len(slot))


def row_lengths_decode(seq_lens, q_len, num_heads):
    s = np.ascontiguousarray(seq_lens, dtype=np.int32)
    rows = len(s) * q_len * num_heads
    rs = np.empty(rows, np.int32)
    rl = np.empty(rows, np.int32)
    lib().orc_row_lengths_decode(_p(s), len(s), q_len, num_heads, _p(rs), _p(rl))
    return rs, rl


def row_lengths_prefill(query_req_id, query_abs_pos, num_heads):
    a = np.ascontiguousarray(query_req_id, dtype=np.int32)
    b = np.ascontiguousarray(query_abs_pos, dtype=np.int32)
    rows = len(a) * num_heads
    rs = np.empty(rows, np.int32)
    rl = np.empty(rows, np.int32)
    lib().orc_row_lengths_prefill(_p(a), _p(b), len(a), num_heads, _p(rs), _p(rl))
    return rs, rl


def index_score(idx_dtype, hidx, idx_cache, q, q_dtype, block_table, row_seq, row_len, max_pages,
                rows=None, want_absdot=False, block_stride=None):
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    rs = np.ascontiguousarray(row_seq, dtype=np.int32)
    rl = np.ascontiguousarray(row_len, dtype=np.int32)
    q = np.ascontiguousarray(q)
    n = len(rs)
    scores = np.full((n, max_pages), np.nan, dtype=np.float32)
    absdot = np.zeros((n, max_pages), dtype=np.float32) if want_absdot else None
    sub, nsub = _subset(rows)
    if block_stride is None:
        block_stride = hidx * index_field_bytes(idx_dtype)
    lib().orc_index_score(idx_dtype, hidx, _p(idx_cache), block_stride, _p(q), q_dtype, _p(bt), bt.shape[1],
                          _p(rs), _p(rl), n, max_pages, _p(scores), _p(absdot), _p(sub), nsub)
    return (scores, absdot) if want_absdot else scores


def topk_select(scores, row_seq, row_len, block_table, id_rule, k_pages, force_tail=True, rows=None):
    sc = np.ascontiguousarray(scores, dtype=np.float32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    rs = np.ascontiguousarray(row_seq, dtype=np.int32)
    rl = np.ascontiguousarray(row_len, dtype=np.int32)
    n = sc.shape[0]
    ti = np.full((n, k_pages), -2, np.int32)
    sb = np.full((n, k_pages), -2, np.int32)
    ctx = np.full(n, -2, np.int32)
    sub, nsub = _subset(rows)
    lib().orc_topk_select(_p(sc), n, sc.shape[1], _p(rs), _p(rl), _p(bt), bt.shape[1], id_rule, k_pages,
                          1 if force_tail else 0, _p(ti), _p(sb), _p(ctx), _p(sub), nsub)
    return ti, sb, ctx


def topk_select_blocks(scores, row_seq, row_len, block_table, id_rule, k_pages, force_tail=True, rows=None):
    """128-token blocks as the unit of selection (k_pages // 8 blocks a row)."""
    sc = np.ascontiguousarray(scores, dtype=np.float32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    rs = np.ascontiguousarray(row_seq, dtype=np.int32)
    rl = np.ascontiguousarray(row_len, dtype=np.int32)
    n = sc.shape[0]
    ti = np.full((n, k_pages), -2, np.int32)
    sb = np.full((n, k_pages), -2, np.int32)
    ctx = np.full(n, -2, np.int32)
    sub, nsub = _subset(rows)
    lib().orc_topk_select_blocks(_p(sc), n, sc.shape[1], _p(rs), _p(rl), _p(bt), bt.shape[1], id_rule, k_pages,
                                 1 if force_tail else 0, _p(ti), _p(sb), _p(ctx), _p(sub), nsub)
    return ti, sb, ctx


def sparse_attention(kv_dtype, hkv, kv_cache, k_scale, v_scale, q, q_dtype, group, sparse_bt, sparse_ctx,
                     sm_scale, rows=None):
    q = np.ascontiguousarray(q)
    sb = np.ascontiguousarray(sparse_bt, dtype=np.int32)
    ctx = np.ascontiguousarray(sparse_ctx, dtype=np.int32)
    n = len(ctx)
    out = np.zeros((n * group, 128), dtype=np.uint16)
    sub, nsub = _subset(rows)
    lib().orc_sparse_attention(kv_dtype, hkv, _p(kv_cache), k_scale, v_scale, _p(q), q_dtype, group, _p(sb),
                               _p(ctx), n, sb.shape[1], sm_scale, _p(out), _p(sub), nsub)
    return out


def dense_attention(kv_dtype, hkv, kv_cache, k_scale, v_scale, q, q_dtype, group, block_table, row_seq,
                    row_len, sm_scale, rows=None):
    q = np.ascontiguousarray(q)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    rs = np.ascontiguousarray(row_seq, dtype=np.int32)
    rl = np.ascontiguousarray(row_len, dtype=np.int32)
    n = len(rs)
    out = np.zeros((n * group, 128), dtype=np.uint16)
    sub, nsub = _subset(rows)
    lib().orc_dense_attention(kv_dtype, hkv, _p(kv_cache), k_scale, v_scale, _p(q), q_dtype, group, _p(bt),
                              bt.shape[1], _p(rs), _p(rl), n, sm_scale, _p(out), _p(sub), nsub)
    return out


def num_threads():
    return int(lib().orc_num_threads())


def set_num_threads(n):
    """Threads of the oracle's later OpenMP loops (for a one-core timing)."""
    lib().orc_set_num_threads(int(n))


def bf16_to_f32(a):
    """Vectorised bf16-bits -> float32 (a view, for test comparisons)."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)
