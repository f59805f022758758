"""The C ABI library builds, loads and exports every call include/bsp.h
declares; host-side argument validation answers without touching a GPU."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "bsp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(bsp_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_paged_score_gb300 import build
    path = build.build()
    return C.CDLL(path)


def test_header_declares_the_five_steps():
    names = declared_functions()
    for n in ("bsp_kv_page_write", "bsp_index_score", "bsp_topk_select", "bsp_sparse_pa_decode",
              "bsp_sparse_pa_prefill", "bsp_index_score_prefill", "bsp_sparse_decode_step"):
        assert n in names, n


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header():
    from block_sparse_paged_score_gb300 import bsp
    assert set(declared_functions()) <= set(bsp.SYMBOLS), set(declared_functions()) - set(bsp.SYMBOLS)


def test_host_validation_without_a_gpu():
    from block_sparse_paged_score_gb300 import bsp
    L = bsp.lib()
    assert L.bsp_status_str(2) == b"unsupported size or dtype"
    assert L.bsp_kv_block_bytes(bsp.FP8_E4M3, 1) == 32768
    assert L.bsp_kv_block_bytes(bsp.MXFP4, 1) == 2 * 8704
    assert L.bsp_index_field_bytes(bsp.FP8_E4M3) == 16896
    d = bsp.KvCacheDesc()
    fake = 1 << 20  # a host-side descriptor only; never dereferenced here
    assert L.bsp_kv_cache_interleaved(bsp.FP8_E4M3, 1, fake, 128, 0.5, 0.5, C.byref(d)) == 0
    assert d.num_ids == 2040 and d.v_base - d.k_base == 8 * 2048 and d.id_stride_bytes == 2048
    assert L.bsp_kv_cache_interleaved(bsp.MXFP4, 2, fake, 4, 1, 1, C.byref(d)) == 0
    assert d.id_stride_bytes == 4 * 8704 and d.v_base - d.k_base == 2 * 8704 and d.num_ids == 32
    assert L.bsp_kv_cache_interleaved(bsp.FP8_E4M3, 1, fake + 8, 128, 0.5, 0.5, C.byref(d)) == 1  # misaligned
    ic = bsp.IndexCacheDesc()
    assert L.bsp_index_cache_packed(bsp.FP8_E4M3, 1, fake, 16, C.byref(ic)) == 0
    # q_group out of range and a prefill scorer with bf16 queries are refused before any launch
    assert L.bsp_index_score(C.byref(ic), fake, bsp.FP8_E4M3, fake, 4, fake, fake, 4, 9, 8, fake, None, None) == 2
    ic2 = bsp.IndexCacheDesc()
    assert L.bsp_index_cache_packed(bsp.MXFP4, 1, fake, 16, C.byref(ic2)) == 0
    assert L.bsp_index_score_prefill(C.byref(ic2), fake, bsp.BF16, fake, 4, fake, fake, 4, fake, 1, 1, 8, fake,
                                     None, None) == 2
    assert L.bsp_topk_select(fake, 4, 8, fake, fake, fake, 1, 0, 0, 1, fake, fake, fake, None) == 1  # k_pages 0
    # the allocation-free attention runs the attention's own checks first: a
    # group of 3 query heads per KV head is refused before any CUDA call
    d2 = bsp.KvCacheDesc()
    assert L.bsp_kv_cache_interleaved(bsp.FP8_E4M3, 2, fake, 16, 0.5, 0.5, C.byref(d2)) == 0
    assert L.bsp_sparse_pa_decode_noalloc(C.byref(d2), fake, bsp.BF16, 6, fake, fake, 4, 8, C.c_float(0.1), fake,
                                          None, None) == 2
    assert L.bsp_sparse_pa_decode_noalloc(C.byref(d2), fake, bsp.BF16, 32, fake, fake, 3, 8, C.c_float(0.1), fake,
                                          None, None) == 1  # rows not a multiple of the KV heads


def test_binding_refuses_pageable_host_tensors():
    """Tensors reach the library as device addresses: CUDA tensors, or, for
    the per-token inputs and outputs only, pinned host tensors (mapped into
    the device's address space).  A pageable host tensor has no device
    address and is refused before any call, in either role."""
    import torch
    from block_sparse_paged_score_gb300 import bsp
    assert bsp._ptr(None) is None and bsp._io_ptr(None) is None
    with pytest.raises(ValueError):
        bsp._ptr(torch.empty(4))
    with pytest.raises(ValueError):
        bsp._io_ptr(torch.empty(4))


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="fake device addresses must never reach a GPU")
def test_invalid_decode_step_enqueues_nothing():
    """bsp_sparse_decode_step checks every stage's arguments (scorer,
    selector, attention and its workspace) before its first event or launch:
    an invalid step returns its status with nothing enqueued.  Without a GPU
    any launch would fail with BSP_ERR_CUDA, so each documented status below
    shows that the call returned before its first launch."""
    from block_sparse_paged_score_gb300 import bsp
    L = bsp.lib()
    fake = 1 << 20  # host-side descriptors and addresses only; never dereferenced
    kv, ic = bsp.KvCacheDesc(), bsp.IndexCacheDesc()
    assert L.bsp_kv_cache_interleaved(bsp.FP8_E4M3, 1, fake, 64, 0.5, 0.5, C.byref(kv)) == 0
    assert L.bsp_index_cache_packed(bsp.FP8_E4M3, 1, fake, 64, C.byref(ic)) == 0

    def args(**kw):
        a = bsp.DecodeStepArgs()
        a.kv, a.idx = C.pointer(kv), C.pointer(ic)
        for f in ("k_new", "v_new", "idx_k_new", "slot", "q", "q_cast", "idx_q", "idx_q_cast", "seq_lens",
                  "block_table", "row_seq", "row_len", "scores", "topk_idx", "sparse_bt", "sparse_ctx", "out", "ws",
                  "dev_err"):
            setattr(a, f, fake)
        a.num_new_tokens, a.num_seqs, a.q_len, a.num_q_heads = 1, 1, 1, 16
        a.q_dtype, a.idx_q_dtype = bsp.BF16, bsp.FP8_E4M3
        a.bt_stride, a.max_pages, a.k_pages, a.flags, a.sm_scale = 8, 64, 16, bsp.FORCE_TAIL, 0.088
        a.ws_bytes, a.sel_counters = 1 << 30, None
        for k, v in kw.items():
            setattr(a, k, v)
        return a

    cases = [
        (dict(num_q_heads=3), 2),                   # 3 query heads per KV head (attention)
        (dict(k_pages=4096), 2),                    # more pages than the selector takes
        (dict(max_pages=100), 1),                   # wider than the block table covers (scorer)
        (dict(k_pages=2048, ws_bytes=16), 3),       # one row split 64 ways needs a workspace
        (dict(out=None), 1),                        # no output (attention)
        (dict(scores=None), 1),                     # no score rows (scorer)
        (dict(topk_idx=None), 1),                   # no selection output (selector)
        (dict(sel_counters=fake + 2), 1),           # misaligned counters (fused selection)
        (dict(idx_q_cast=None), 1),                 # e4m3 index queries need their cast buffer
        (dict(q_dtype=bsp.FP8_E4M3, q_cast=None), 1),
        (dict(flags=bsp.FORCE_TAIL | bsp.REUSE_SELECTION, num_q_heads=3), 2),
        (dict(num_seqs=1 << 29, q_len=8), 2),     # more rows than an int32 counts
    ]
    n0 = L.bsp_launch_count()
    for kw, want in cases:
        assert L.bsp_sparse_decode_step(C.byref(args(**kw)), None, None) == want, kw
    assert L.bsp_launch_count() == n0
