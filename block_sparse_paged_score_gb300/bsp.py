"""ctypes binding of libbsp (include/bsp.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch CUDA tensors; the stream is torch's current stream unless
one is given.  A call whose library is missing raises -- there is no CPU
fallback.
"""
import ctypes as C
import math
import os

import torch

from . import build as _build

BF16, FP8_E4M3, MXFP4 = 0, 1, 2
FORCE_TAIL = 1
REUSE_SELECTION = 2  # decode step: attend with another layer's sparse_bt / sparse_ctx
SELECT_BLOCKS = 4  # top-k: 128-token blocks are the unit of selection
DEVERR = {1: "page id", 2: "block id", 4: "group sequence", 8: "timeout", 16: "slot"}
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace too small", 4: "CUDA error"}


class BspError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn}: {STATUS.get(status, status)} (status {status})")
        self.status = status


class KvCacheDesc(C.Structure):
    _fields_ = [("dtype", C.c_int32), ("num_kv_heads", C.c_int32), ("k_base", C.c_void_p), ("v_base", C.c_void_p),
                ("id_stride_bytes", C.c_int64), ("num_ids", C.c_int64), ("num_blocks", C.c_int64),
                ("k_scale", C.c_float), ("v_scale", C.c_float)]


class IndexCacheDesc(C.Structure):
    _fields_ = [("dtype", C.c_int32), ("num_heads", C.c_int32), ("base", C.c_void_p),
                ("block_stride_bytes", C.c_int64), ("num_blocks", C.c_int64)]


class DecodeStepArgs(C.Structure):
    _fields_ = [("kv", C.POINTER(KvCacheDesc)), ("idx", C.POINTER(IndexCacheDesc)),
                ("k_new", C.c_void_p), ("v_new", C.c_void_p), ("idx_k_new", C.c_void_p), ("slot", C.c_void_p),
                ("num_new_tokens", C.c_int32),
                ("q", C.c_void_p), ("q_dtype", C.c_int32), ("q_cast", C.c_void_p), ("num_q_heads", C.c_int32),
                ("idx_q", C.c_void_p), ("idx_q_dtype", C.c_int32), ("idx_q_cast", C.c_void_p),
                ("seq_lens", C.c_void_p), ("num_seqs", C.c_int32), ("q_len", C.c_int32),
                ("block_table", C.c_void_p), ("bt_stride", C.c_int32), ("max_pages", C.c_int32),
                ("k_pages", C.c_int32), ("flags", C.c_int32), ("sm_scale", C.c_float),
                ("row_seq", C.c_void_p), ("row_len", C.c_void_p), ("scores", C.c_void_p), ("topk_idx", C.c_void_p),
                ("sparse_bt", C.c_void_p), ("sparse_ctx", C.c_void_p), ("out", C.c_void_p), ("ws", C.c_void_p),
                ("ws_bytes", C.c_size_t), ("dev_err", C.c_void_p), ("sel_counters", C.c_void_p)]


_lib = None
SYMBOLS = {
    "bsp_kv_cache_interleaved": [C.c_int32, C.c_int32, C.c_void_p, C.c_int64, C.c_float, C.c_float,
                                 C.POINTER(KvCacheDesc)],
    "bsp_index_cache_packed": [C.c_int32, C.c_int32, C.c_void_p, C.c_int64, C.POINTER(IndexCacheDesc)],
    "bsp_kv_page_write": [C.POINTER(KvCacheDesc), C.POINTER(IndexCacheDesc), C.c_void_p, C.c_void_p, C.c_void_p,
                          C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p],
    "bsp_cast_e4m3": [C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p],
    "bsp_row_lengths_decode": [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p],
    "bsp_row_lengths_prefill": [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p],
    "bsp_index_score": [C.POINTER(IndexCacheDesc), C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p,
                        C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p],
    "bsp_index_score_prefill": [C.POINTER(IndexCacheDesc), C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p,
                                C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                C.c_void_p, C.c_void_p],
    "bsp_topk_select": [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                        C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p],
    "bsp_sparse_pa_decode": [C.POINTER(KvCacheDesc), C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                             C.c_int32, C.c_int32, C.c_float, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p,
                             C.c_void_p],
    "bsp_sparse_pa_decode_noalloc": [C.POINTER(KvCacheDesc), C.c_void_p, C.c_int32, C.c_int32, C.c_void_p,
                                     C.c_void_p, C.c_int32, C.c_int32, C.c_float, C.c_void_p, C.c_void_p,
                                     C.c_void_p],
    "bsp_sparse_pa_prefill": [C.POINTER(KvCacheDesc), C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                              C.c_int32, C.c_int32, C.c_float, C.c_void_p, C.c_void_p, C.c_void_p],
    "bsp_sparse_pa_decode_workspace_bytes": [C.c_int32, C.c_int32, C.c_int32],
    "bsp_sparse_pa_decode_splits": [C.c_int32, C.c_int32, C.c_int32],
    "bsp_sparse_decode_step": [C.POINTER(DecodeStepArgs), C.c_void_p, C.c_void_p],
    "bsp_kv_block_bytes": [C.c_int32, C.c_int32],
    "bsp_index_field_bytes": [C.c_int32],
    "bsp_status_str": [C.c_int32],
    "bsp_last_cuda_error": [],
    "bsp_launch_count": [],
    "bsp_version": [],
}
RESTYPES = {"bsp_sparse_pa_decode_workspace_bytes": C.c_size_t, "bsp_kv_block_bytes": C.c_int64,
            "bsp_index_field_bytes": C.c_int64, "bsp_status_str": C.c_char_p, "bsp_launch_count": C.c_int64}


def library_path():
    return _build.LIB


def lib(build_if_missing=True):
    """Load libbsp.so (building it first when the CUDA toolkit is here)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libbsp.so is not built ({path}); run __graft_entry__.build()")
        L = C.CDLL(path)
        for name, args in SYMBOLS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = RESTYPES.get(name, C.c_int32)
        _lib = L
    return _lib


def _check(fn, status):
    if status != 0:
        raise BspError(fn, status)


def _ptr(t):
    """The device address of a CUDA tensor: caches, tables, lengths, score
    rows, selections and workspaces must live in device memory."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libbsp takes a CUDA tensor here (only per-token inputs and outputs may be pinned host "
                         "tensors)")
    return t.data_ptr()


def _io_ptr(t):
    """The address of a per-token input or output: a CUDA tensor, or a pinned
    host tensor (pinned memory is mapped into the device's address space;
    the kernels read or write it once, in place)."""
    if t is None:
        return None
    if not t.is_cuda and not t.is_pinned():
        raise ValueError("libbsp takes CUDA tensors or pinned host tensors")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def launch_count():
    return int(lib().bsp_launch_count())


def kv_block_bytes(dtype, hkv):
    return int(lib().bsp_kv_block_bytes(dtype, hkv))


def index_field_bytes(dtype):
    return int(lib().bsp_index_field_bytes(dtype))


class KvCache:
    """An interleaved (bf16/fp8) or MXFP4 K/V cache in a caller-owned uint8 tensor."""

    def __init__(self, dtype, num_kv_heads, num_blocks, k_scale=1.0, v_scale=1.0, buffer=None, device="cuda"):
        nbytes = num_blocks * kv_block_bytes(dtype, num_kv_heads)
        self.buffer = buffer if buffer is not None else torch.zeros(nbytes, dtype=torch.uint8, device=device)
        assert self.buffer.numel() >= nbytes
        self.dtype, self.num_kv_heads, self.num_blocks = dtype, num_kv_heads, num_blocks
        self.desc = KvCacheDesc()
        _check("bsp_kv_cache_interleaved",
               lib().bsp_kv_cache_interleaved(dtype, num_kv_heads, _ptr(self.buffer), num_blocks, k_scale, v_scale,
                                              C.byref(self.desc)))


class IndexCache:
    """A packed index-key cache (one field per block and index head)."""

    def __init__(self, dtype, num_heads, num_blocks, buffer=None, device="cuda"):
        nbytes = num_blocks * num_heads * index_field_bytes(dtype)
        self.buffer = buffer if buffer is not None else torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.dtype, self.num_heads, self.num_blocks = dtype, num_heads, num_blocks
        self.desc = IndexCacheDesc()
        _check("bsp_index_cache_packed",
               lib().bsp_index_cache_packed(dtype, num_heads, _ptr(self.buffer), num_blocks, C.byref(self.desc)))


def kv_page_write(kv, idx, k, v, idx_k, slot, dev_err=None, stream=None):
    _check("bsp_kv_page_write",
           lib().bsp_kv_page_write(C.byref(kv.desc), C.byref(idx.desc) if idx is not None else None, _io_ptr(k),
                                   _io_ptr(v), _io_ptr(idx_k), _io_ptr(slot), slot.numel(), _ptr(dev_err),
                                   _stream(stream)))


def cast_e4m3(x, out=None, stream=None):
    out = out if out is not None else torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check("bsp_cast_e4m3", lib().bsp_cast_e4m3(_io_ptr(x), _io_ptr(out), x.numel(), _stream(stream)))
    return out


def row_lengths_decode(seq_lens, q_len, num_heads, row_seq=None, row_len=None, stream=None):
    rows = seq_lens.numel() * q_len * num_heads
    row_seq = row_seq if row_seq is not None else torch.empty(rows, dtype=torch.int32, device=seq_lens.device)
    row_len = row_len if row_len is not None else torch.empty(rows, dtype=torch.int32, device=seq_lens.device)
    _check("bsp_row_lengths_decode", lib().bsp_row_lengths_decode(_io_ptr(seq_lens), seq_lens.numel(), q_len, num_heads,
                                                                  _ptr(row_seq), _ptr(row_len), _stream(stream)))
    return row_seq, row_len


def row_lengths_prefill(query_req_id, query_abs_pos, num_heads, row_seq=None, row_len=None, stream=None):
    rows = query_req_id.numel() * num_heads
    dev = query_req_id.device
    row_seq = row_seq if row_seq is not None else torch.empty(rows, dtype=torch.int32, device=dev)
    row_len = row_len if row_len is not None else torch.empty(rows, dtype=torch.int32, device=dev)
    _check("bsp_row_lengths_prefill",
           lib().bsp_row_lengths_prefill(_ptr(query_req_id), _ptr(query_abs_pos), query_req_id.numel(), num_heads,
                                         _ptr(row_seq), _ptr(row_len), _stream(stream)))
    return row_seq, row_len


def index_score(idx, idx_q, q_dtype, block_table, row_seq, row_len, q_group, max_pages, scores=None, dev_err=None,
                stream=None):
    rows = row_seq.numel()
    scores = scores if scores is not None else torch.empty((rows, max_pages), dtype=torch.float32,
                                                           device=idx_q.device)
    _check("bsp_index_score",
           lib().bsp_index_score(C.byref(idx.desc), _ptr(idx_q), q_dtype, _ptr(block_table), block_table.shape[1],
                                 _ptr(row_seq), _ptr(row_len), rows, q_group, max_pages, _ptr(scores), _ptr(dev_err),
                                 _stream(stream)))
    return scores


def prefill_tiles(cu_tokens_host):
    """Host upper bound on the 128-row tiles of the prefill chunks."""
    sizes = [int(b) - int(a) for a, b in zip(cu_tokens_host[:-1], cu_tokens_host[1:])]
    return sum((s + 127) // 128 for s in sizes)


def index_score_prefill(idx, idx_q, q_dtype, block_table, row_seq, row_len, cu_tokens, num_chunks, max_tiles,
                        max_pages, scores=None, dev_err=None, stream=None):
    rows = row_seq.numel()
    scores = scores if scores is not None else torch.empty((rows, max_pages), dtype=torch.float32,
                                                           device=idx_q.device)
    _check("bsp_index_score_prefill",
           lib().bsp_index_score_prefill(C.byref(idx.desc), _ptr(idx_q), q_dtype, _ptr(block_table),
                                         block_table.shape[1], _ptr(row_seq), _ptr(row_len), rows, _ptr(cu_tokens),
                                         num_chunks, max_tiles, max_pages, _ptr(scores), _ptr(dev_err),
                                         _stream(stream)))
    return scores


def topk_select(scores, row_seq, row_len, block_table, kv_dtype, k_pages, flags=FORCE_TAIL, topk_idx=None,
                sparse_bt=None, sparse_ctx=None, stream=None):
    rows, max_pages = scores.shape
    dev = scores.device
    topk_idx = topk_idx if topk_idx is not None else torch.empty((rows, k_pages), dtype=torch.int32, device=dev)
    sparse_bt = sparse_bt if sparse_bt is not None else torch.empty((rows, k_pages), dtype=torch.int32, device=dev)
    sparse_ctx = sparse_ctx if sparse_ctx is not None else torch.empty(rows, dtype=torch.int32, device=dev)
    _check("bsp_topk_select",
           lib().bsp_topk_select(_ptr(scores), rows, max_pages, _ptr(row_seq), _ptr(row_len), _ptr(block_table),
                                 block_table.shape[1], kv_dtype, k_pages, flags, _ptr(topk_idx), _ptr(sparse_bt),
                                 _ptr(sparse_ctx), _stream(stream)))
    return topk_idx, sparse_bt, sparse_ctx


def decode_workspace_bytes(num_rows, k_pages, group):
    return int(lib().bsp_sparse_pa_decode_workspace_bytes(num_rows, k_pages, group))


def decode_splits(kv_dtype, num_rows, k_pages):
    """CTAs per row of a decode attention call with these sizes (> 8: the
    splits merge through the workspace)."""
    return int(lib().bsp_sparse_pa_decode_splits(kv_dtype, num_rows, k_pages))


def decode_workspace(num_rows, k_pages, group, device="cuda"):
    """A zeroed split-K workspace (its arrival counters must start at zero)."""
    n = decode_workspace_bytes(num_rows, k_pages, group)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def sparse_pa_decode(kv, q, q_dtype, num_q_heads, sparse_bt, sparse_ctx, k_pages, sm_scale=None, out=None, ws=None,
                     dev_err=None, stream=None):
    rows = sparse_ctx.numel()
    sm_scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(128)
    out = out if out is not None else torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    if ws is None:
        ws = decode_workspace(rows, k_pages, num_q_heads // kv.num_kv_heads, q.device)
    _check("bsp_sparse_pa_decode",
           lib().bsp_sparse_pa_decode(C.byref(kv.desc), _io_ptr(q), q_dtype, num_q_heads, _ptr(sparse_bt),
                                      _ptr(sparse_ctx), rows, k_pages, sm_scale, _io_ptr(out), _ptr(ws), ws.numel(),
                                      _ptr(dev_err), _stream(stream)))
    return out


def sparse_pa_decode_noalloc(kv, q, q_dtype, num_q_heads, sparse_bt, sparse_ctx, k_pages, sm_scale=None, out=None,
                             dev_err=None, stream=None):
    """bsp_sparse_pa_decode without a caller workspace (the library's own
    fixed scratch; see include/bsp.h for the size limit and the sharing rule)."""
    rows = sparse_ctx.numel()
    sm_scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(128)
    out = out if out is not None else torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    _check("bsp_sparse_pa_decode_noalloc",
           lib().bsp_sparse_pa_decode_noalloc(C.byref(kv.desc), _io_ptr(q), q_dtype, num_q_heads, _ptr(sparse_bt),
                                              _ptr(sparse_ctx), rows, k_pages, sm_scale, _io_ptr(out), _ptr(dev_err),
                                              _stream(stream)))
    return out


def sparse_pa_prefill(kv, q, q_dtype, num_q_heads, sparse_bt, sparse_ctx, k_pages, sm_scale=None, out=None,
                      dev_err=None, stream=None):
    rows = sparse_ctx.numel()
    sm_scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(128)
    out = out if out is not None else torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    _check("bsp_sparse_pa_prefill",
           lib().bsp_sparse_pa_prefill(C.byref(kv.desc), _io_ptr(q), q_dtype, num_q_heads, _ptr(sparse_bt),
                                       _ptr(sparse_ctx), rows, k_pages, sm_scale, _io_ptr(out), _ptr(dev_err),
                                       _stream(stream)))
    return out


def sparse_decode_step(args, events=None, stream=None):
    """Run bsp_sparse_decode_step on a filled DecodeStepArgs (see DecodeStep)."""
    ev = None
    if events is not None:
        ev = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check("bsp_sparse_decode_step", lib().bsp_sparse_decode_step(C.byref(args), ev, _stream(stream)))
