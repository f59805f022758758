"""Guard bands and sentinels around every output (GPU required).

Each buffer a call writes sits inside a larger allocation: canary bytes on
both sides and, between them, a sentinel that the call never produces (NaN
for scores and for the bf16 attention output, the e4m3 NaN code for the
casts, 0x7EEEEEEE for ids and lengths).  After the call the canaries must be
intact (nothing written outside the buffer) and no sentinel may be left where
the call defines every element (nothing left unwritten).  The caches are
wrapped the same way, zero inside as a fresh cache.  Without a memory checker
on the GPU, this is the overrun and coverage check of every kernel: the
writer, the casts and row lengths, both decode scorers, the prefill scorers,
the selector, the decode and prefill attention, and the one-call decode step.
"""
import numpy as np
import pytest
import torch

from block_sparse_paged_score_gb300 import workloads as W

from harness import MINI, SM_SCALE

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side: a multiple of 256 keeps the inside aligned
CANARY = 0x5A
NAN32, NAN16, E4M3_NAN, ID_SENTINEL = 0x7FC00000, 0x7FC0, 0x7F, 0x7EEEEEEE
INT_VIEW = {1: torch.uint8, 2: torch.int16, 4: torch.int32}


class Guarded:
    """A tensor of `shape` and `dtype` inside canary bytes, filled with the
    bit pattern `sentinel` (None: zeros)."""

    def __init__(self, shape, dtype, sentinel=None):
        es = torch.empty((), dtype=dtype).element_size()
        self.n = int(np.prod(shape))
        self.nbytes = self.n * es
        self.raw = torch.full((self.nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        inner = self.raw[GUARD:GUARD + self.nbytes]
        self.bits = inner.view(INT_VIEW[es])
        self.sentinel = sentinel
        self.bits.fill_(0 if sentinel is None else sentinel)
        self.t = inner.view(dtype).view(shape)

    def guards_intact(self):
        return bool((self.raw[:GUARD] == CANARY).all()) and bool((self.raw[GUARD + self.nbytes:] == CANARY).all())

    def left(self):
        """Elements still holding the sentinel."""
        return int((self.bits == self.sentinel).sum())


def check(name, g, complete=True):
    assert g.guards_intact(), f"{name}: a write landed outside the buffer"
    if complete:
        assert g.left() == 0, f"{name}: {g.left()} of {g.n} elements left unwritten"


def t(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def guarded_caches(w, bsp):
    kvg = Guarded((w.num_blocks * bsp.kv_block_bytes(w.kv_dtype, w.hkv),), torch.uint8)
    idxg = Guarded((w.num_blocks * w.hidx * bsp.index_field_bytes(w.idx_dtype),), torch.uint8)
    kv = bsp.KvCache(w.kv_dtype, w.hkv, w.num_blocks, w.k_scale, w.v_scale, buffer=kvg.t)
    idx = bsp.IndexCache(w.idx_dtype, w.hidx, w.num_blocks, buffer=idxg.t)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k, v, ik, slot in w.context_batches():
        bsp.kv_page_write(kv, idx, t(k), t(v), t(ik), t(slot), dev_err=err)
    torch.cuda.synchronize()
    check("K/V cache", kvg, complete=False)
    check("index cache", idxg, complete=False)
    assert err.item() == 0
    return kv, idx, kvg, idxg


def queries(w, bsp):
    """The attention and index queries as the calls take them (e4m3 casts into
    guarded buffers where the workload uses e4m3)."""
    q, iq = w.queries()
    out = []
    for x, dt in ((q, w.q_dtype), (iq, w.idx_q_dtype)):
        xb = t(x)
        if dt == W.FP8:
            c = Guarded(tuple(xb.shape), torch.uint8, E4M3_NAN)
            bsp.cast_e4m3(xb, out=c.t)
            torch.cuda.synchronize()
            check("e4m3 cast", c)
            xb = c.t
        out.append(xb)
    return out


@pytest.mark.parametrize("name", ["fp8", "fp8_q4_h2", "mx", "mx_h2", "bf16", "mixed"])
def test_every_call_writes_inside_its_buffers_and_all_of_them(name):
    from block_sparse_paged_score_gb300 import bsp
    w = W.Workload(MINI[name])
    kv, idx, kvg, idxg = guarded_caches(w, bsp)
    q, iq = queries(w, bsp)
    bt = t(w.block_table)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows, nd, ndt = w.num_rows, w.num_decode_tokens * w.hkv, w.num_decode_tokens

    rs, rl = Guarded((rows,), torch.int32, ID_SENTINEL), Guarded((rows,), torch.int32, ID_SENTINEL)
    bsp.row_lengths_decode(t(w.decode_lens), w.q_len, w.hkv, row_seq=rs.t[:nd], row_len=rl.t[:nd])
    if rows > nd:
        bsp.row_lengths_prefill(t(w.query_req_id), t(w.query_abs_pos), w.hkv, row_seq=rs.t[nd:], row_len=rl.t[nd:])
    torch.cuda.synchronize()
    check("row_seq", rs)
    check("row_len", rl)

    sc = Guarded((rows, w.max_pages), torch.float32, NAN32)
    bsp.index_score(idx, iq[:ndt], w.idx_q_dtype, bt, rs.t[:nd], rl.t[:nd], w.q_len, w.max_pages,
                    scores=sc.t[:nd], dev_err=err)
    if rows > nd:
        if w.idx_q_dtype == W.FP8:  # the prefill rows on the tcgen05 prefill scorer
            cu = t(w.cu_prefill)
            bsp.index_score_prefill(idx, iq[ndt:], w.idx_q_dtype, bt, rs.t[nd:], rl.t[nd:], cu, len(w.cu_prefill) - 1,
                                    bsp.prefill_tiles(w.cu_prefill), w.max_pages, scores=sc.t[nd:], dev_err=err)
        else:
            bsp.index_score(idx, iq[ndt:], w.idx_q_dtype, bt, rs.t[nd:], rl.t[nd:], 1, w.max_pages,
                            scores=sc.t[nd:], dev_err=err)
    torch.cuda.synchronize()
    check("scores", sc)

    ti, sb = Guarded((rows, w.k_pages), torch.int32, ID_SENTINEL), Guarded((rows, w.k_pages), torch.int32, ID_SENTINEL)
    ctx = Guarded((rows,), torch.int32, ID_SENTINEL)
    bsp.topk_select(sc.t, rs.t, rl.t, bt, w.kv_dtype, w.k_pages, topk_idx=ti.t, sparse_bt=sb.t, sparse_ctx=ctx.t)
    torch.cuda.synchronize()
    for nm, g in (("topk_idx", ti), ("sparse_bt", sb), ("sparse_ctx", ctx)):
        check(nm, g)

    out = Guarded(tuple(q.shape), torch.bfloat16, NAN16)
    bsp.sparse_pa_decode(kv, q[:ndt], w.q_dtype, w.hq, sb.t[:nd], ctx.t[:nd], w.k_pages, SM_SCALE,
                         out=out.t[:ndt], dev_err=err)
    if rows > nd:
        bsp.sparse_pa_prefill(kv, q[ndt:], w.q_dtype, w.hq, sb.t[nd:], ctx.t[nd:], w.k_pages, SM_SCALE,
                              out=out.t[ndt:], dev_err=err)
    torch.cuda.synchronize()
    check("attention output", out)
    check("K/V cache", kvg, complete=False)
    check("index cache", idxg, complete=False)
    assert err.item() == 0, err.item()


@pytest.mark.parametrize("name", ["fp8", "fp8_q4_h2", "mx"])
def test_decode_step_writes_inside_its_buffers_and_all_of_them(name):
    """bsp_sparse_decode_step with every caller buffer it writes guarded."""
    from block_sparse_paged_score_gb300 import bsp, step
    w = W.Workload(MINI[name])
    kv, idx, kvg, idxg = guarded_caches(w, bsp)
    bt = t(w.block_table)
    st = step.DecodeStep(w, kv, idx, bt)
    a = st.args
    g = {}
    for nm, tensor, sentinel in (("row_seq", st.row_seq, ID_SENTINEL), ("row_len", st.row_len, ID_SENTINEL),
                                 ("scores", st.scores, NAN32), ("topk_idx", st.topk_idx, ID_SENTINEL),
                                 ("sparse_bt", st.sparse_bt, ID_SENTINEL), ("sparse_ctx", st.sparse_ctx, ID_SENTINEL),
                                 ("out", st.out, NAN16), ("q_cast", st.q_cast, E4M3_NAN),
                                 ("idx_q_cast", st.idx_q_cast, E4M3_NAN)):
        g[nm] = Guarded(tuple(tensor.shape), tensor.dtype, sentinel)
        setattr(st, nm, g[nm].t)
        setattr(a, nm, g[nm].t.data_ptr())
    k, v, ik, slot = w.step_tokens()
    q, iq = w.queries()
    st.run(t(k), t(v), t(ik), t(slot), t(q), t(iq), t(w.decode_lens))
    torch.cuda.synchronize()
    for nm, gb in g.items():
        # the casts are written only where the step attends or scores in e4m3
        used = not ((nm == "q_cast" and w.q_dtype != W.FP8) or (nm == "idx_q_cast" and w.idx_q_dtype != W.FP8))
        check(nm, gb, complete=used)
    check("K/V cache", kvg, complete=False)
    check("index cache", idxg, complete=False)
    assert st.dev_err.item() == 0
