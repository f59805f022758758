"""Parity of the CUDA path with the CPU oracle on small seeded workloads that
span several tiles, pages and blocks with ragged tails (GPU required).

Stage by stage, each GPU stage gets inputs that both sides computed
identically or that the oracle computed (never the other way round):
  write      byte-exact cache bytes;
  scores     |gpu - oracle| <= 2e-5 * sum_d |q_d k_d| (fp32 accumulation of
             128 exact products, at most (128 + 1) * 2^-23 of sum |qk|),
             -inf pattern identical;
  top-k      bit-exact when the GPU selector is fed the oracle's scores;
  attention  max-abs 1e-2 and relative-L2 5e-3 (bf16 out) when the GPU
             attention is fed the oracle's sparse table.
End to end, the GPU pipeline and the oracle pipeline run independently and
their selections agree up to near-ties (gap-aware comparison).
"""
import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_paged_score_gb300 import workloads as W

from harness import MINI, SM_SCALE, GpuSide, OracleSide, attention_close, bf16_f32, mini, selection_agrees

pytestmark = pytest.mark.gpu

SCORE_REL = 2e-5


@pytest.fixture(scope="module")
def bsp():
    from block_sparse_paged_score_gb300 import bsp as b
    b.lib()
    return b


_cache = {}


def sides(name):
    if name not in _cache:
        w = mini(name)
        _cache[name] = (w, OracleSide(w), GpuSide(w))
    return _cache[name]


def test_cast_e4m3_byte_exact(bsp):
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(5000) * s for s in (1e-4, 1, 100, 1000)] + [[0.0, -0.0, 448, 464, 1e9]])
    xb = W.to_bf16_bits(x.astype(np.float32))
    xb = np.concatenate([xb, np.zeros((-len(xb)) % 8 + 3, np.uint16)])  # ragged tail
    got = bsp.cast_e4m3(torch.from_numpy(xb.view(np.int16)).cuda()).cpu().numpy()
    assert np.array_equal(got, O.cast_e4m3(xb))


@pytest.mark.parametrize("name", list(MINI))
def test_write_byte_exact(bsp, name):
    w, o, g = sides(name)
    torch.cuda.synchronize()
    assert g.err.item() == 0
    kv = g.kv.buffer.cpu().numpy()
    idx = g.idx.buffer.cpu().numpy()
    bad = np.nonzero(kv != o.kv)[0]
    assert bad.size == 0, f"{bad.size} K/V bytes differ, first at {bad[:8]}"
    bad = np.nonzero(idx != o.idx)[0]
    assert bad.size == 0, f"{bad.size} index bytes differ, first at {bad[:8]}"


@pytest.mark.parametrize("name", list(MINI))
def test_step_write_is_idempotent_and_queries_cast(bsp, name):
    w, o, g = sides(name)
    k, v, ik, slot = w.step_tokens()
    before = g.kv.buffer.clone()
    if len(slot):
        bsp.kv_page_write(g.kv, g.idx, g.t(k), g.t(v), g.t(ik), g.t(slot))
    assert torch.equal(before, g.kv.buffer)
    assert np.array_equal(g.q.cpu().numpy().view(o.q.dtype).reshape(o.q.shape), o.q)
    assert np.array_equal(g.idx_q.cpu().numpy().view(o.idx_q.dtype).reshape(o.idx_q.shape), o.idx_q)


@pytest.mark.parametrize("name", list(MINI))
def test_row_lengths(bsp, name):
    w, o, g = sides(name)
    rs, rl = g.row_lengths()
    assert np.array_equal(rs.cpu().numpy(), o.row_seq)
    assert np.array_equal(rl.cpu().numpy(), o.row_len)


@pytest.mark.parametrize("name", list(MINI))
def test_index_score_within_bound(bsp, name):
    w, o, g = sides(name)
    ref, mag = o.scores(want_absdot=True)
    rs, rl = g.row_lengths()
    # decode rows share sequences in groups of q_len; the prefill part runs with q_group 1
    nd = w.num_decode_rows
    sc = torch.empty((w.num_rows, w.max_pages), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hidx = w.hidx
    if nd:
        bsp.index_score(g.idx, g.idx_q[:w.num_decode_tokens], w.idx_q_dtype, g.block_table, rs[:nd], rl[:nd],
                        w.q_len, w.max_pages, scores=sc[:nd], dev_err=err)
    if w.num_rows > nd:
        bsp.index_score(g.idx, g.idx_q[w.num_decode_tokens:], w.idx_q_dtype, g.block_table, rs[nd:], rl[nd:],
                        1, w.max_pages, scores=sc[nd:], dev_err=err)
    got = sc.cpu().numpy()
    assert err.item() == 0
    inf_ref, inf_got = np.isneginf(ref), np.isneginf(got)
    assert np.array_equal(inf_ref, inf_got)
    fin = ~inf_ref
    diff = np.abs(got[fin] - ref[fin])
    bound = SCORE_REL * mag[fin] + 1e-30
    ratio = float((diff / np.maximum(mag[fin], 1e-30)).max()) if diff.size else 0.0
    assert (diff <= bound).all(), f"max |err|/sum|qk| = {ratio:.3g}"
    print(f"{name}: max |err|/sum|qk| = {ratio:.3g} over {diff.size} pages")
    _cache[name + ":scores"] = (ref, mag)


@pytest.mark.parametrize("name", list(MINI))
def test_topk_bit_exact_on_oracle_scores(bsp, name):
    w, o, g = sides(name)
    ref = o.scores()
    ti, sb, ctx = o.topk(ref)
    rs, rl = g.row_lengths()
    gti, gsb, gctx = bsp.topk_select(torch.from_numpy(ref).cuda(), rs, rl, g.block_table, w.kv_dtype, w.k_pages)
    assert np.array_equal(gti.cpu().numpy(), ti)
    assert np.array_equal(gsb.cpu().numpy(), sb)
    assert np.array_equal(gctx.cpu().numpy(), ctx)


# (width in pages, row count): "many" rows (at least twice the SMs) take the
# 256-thread CTA selector, "few" the 512/1024-thread one, "long" rows past
# 32768 pages the long-row kernel
TIE_CASES = [(100, "many"), (256, "many"), (500, "many"), (1000, "many"), (2047, "many"), (2048, "many"),
             (3000, "many"), (6000, "many"), (12000, "many"), (300, "few"), (700, "few"), (701, "few"),
             (4000, "few"), (8000, "few"), (9000, "few"), (20000, "few"), (40000, "long"), (65536, "long")]


@pytest.mark.parametrize("max_pages,regime", TIE_CASES)
@pytest.mark.parametrize("force_tail", [True, False])
@pytest.mark.parametrize("kv_dtype", [W.FP8, W.MXFP4])
def test_topk_bit_exact_with_ties(bsp, force_tail, kv_dtype, max_pages, regime):
    """Every selector shape: one warp per row up to 128 pages; with many rows
    one 256-thread CTA with 1 to 32 keys per thread in registers up to 8192
    pages (256 ... 6000), then the long-row kernel with the keys in shared
    memory (12000); with fewer rows than twice the SMs one 512- or
    1024-thread CTA up to 32768 pages (300 ... 20000); rows past that read
    their keys from global memory (40000, and 65536, the largest width).
    Widths that are not a multiple of 4 pages (701, 2047) take the CTA
    kernel's one-key-at-a-time score loads instead of its 16-byte ones.  k
    runs up to 2048 pages, the largest the call takes."""
    rng = np.random.default_rng(3)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = {"many": 2 * sms + 16, "few": 60, "long": 20}[regime]
    sc = rng.integers(-4, 5, (rows, max_pages)).astype(np.float32)  # heavy ties
    sc[::5] = rng.standard_normal((len(sc[::5]), max_pages)).astype(np.float32)
    sc[7, ::3] = -0.0
    sc[8] = 0.0
    L = rng.integers(0, max_pages * 16 + 1, rows).astype(np.int32)
    L[:6] = [0, 1, 16, 17, max_pages * 16, max_pages * 16 - 1]
    nblk = (max_pages + 7) // 8
    bt = np.stack([rng.permutation(4 * nblk)[:nblk] for _ in range(rows)]).astype(np.int32)
    rs = np.arange(rows, dtype=np.int32)
    for k in (1, 2, 37, 128, 2048):
        ti, sb, ctx = O.topk_select(sc, rs, L, bt, 1 if kv_dtype == W.MXFP4 else 0, k, force_tail)
        gti, gsb, gctx = bsp.topk_select(torch.from_numpy(sc).cuda(), torch.from_numpy(rs).cuda(),
                                         torch.from_numpy(L).cuda(), torch.from_numpy(bt).cuda(), kv_dtype, k,
                                         flags=bsp.FORCE_TAIL if force_tail else 0)
        assert np.array_equal(gti.cpu().numpy(), ti), k
        assert np.array_equal(gsb.cpu().numpy(), sb), k
        assert np.array_equal(gctx.cpu().numpy(), ctx), k


@pytest.mark.parametrize("prefill", [False, True])
@pytest.mark.parametrize("name", list(MINI))
def test_attention_on_oracle_table(bsp, name, prefill):
    w, o, g = sides(name)
    ti, sb, ctx = o.topk(o.scores())
    ref = bf16_f32(torch.from_numpy(o.attention(sb, ctx).view(np.int16)))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn = bsp.sparse_pa_prefill if prefill else bsp.sparse_pa_decode
    out = fn(g.kv, g.q, w.q_dtype, w.hq, torch.from_numpy(sb).cuda(), torch.from_numpy(ctx).cuda(), w.k_pages,
             SM_SCALE, dev_err=err)
    got = bf16_f32(out).reshape(ref.shape)
    assert err.item() == 0
    ok, mx, rl2 = attention_close(got, ref)
    print(f"{name} prefill={prefill}: worst err/allowed {mx:.3g} rel-L2 {rl2:.3g}")
    assert ok, (mx, rl2)
    # rows with nothing to attend are exactly zero
    z = np.repeat(ctx == 0, w.group)
    assert (got[z] == 0).all()


@pytest.mark.parametrize("name", ["fp8", "mx", "bf16"])
def test_attention_split_merge_paths(bsp, name):
    """Two ways a split decode row is finished: a cluster of up to 8 split
    CTAs merged through distributed shared memory, and more splits merged
    through the workspace (very few rows, wide selections).  One CTA per
    row, the third way, is the prefill call's path and covered above."""
    for k_pages, rows in ((16, None), (128, None), (128, 2)):
        w = W.Workload(dict(MINI[name], k_pages=k_pages))
        o, g = OracleSide(w), GpuSide(w)
        ti, sb, ctx = o.topk(o.scores())
        n = w.num_rows if rows is None else rows
        sel = np.arange(w.num_rows - n, w.num_rows)  # the longest rows
        ref = bf16_f32(torch.from_numpy(o.attention(sb, ctx).view(np.int16))).reshape(w.num_rows, w.group, 128)[sel]
        q = g.q.reshape(w.num_tokens, w.hq, 128)[w.num_tokens - n // w.hkv:].contiguous()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = bsp.sparse_pa_decode(g.kv, q, w.q_dtype, w.hq, torch.from_numpy(sb[sel]).cuda(),
                                   torch.from_numpy(ctx[sel]).cuda(), w.k_pages, SM_SCALE, dev_err=err)
        got = bf16_f32(out).reshape(n, w.group, 128)
        assert err.item() == 0
        ok, worst, rl2 = attention_close(got, ref)
        print(f"{name} k={k_pages} rows={n} ws={bsp.decode_workspace_bytes(n, k_pages, w.group)}: {worst:.3g} {rl2:.3g}")
        assert ok, (k_pages, n, worst, rl2)


# Larger decode batches: 64 rows x 128 pages (split over clusters of CTAs),
# and 3 rows x 2048 pages (64 splits per row merged through the workspace);
# short contexts, pad rows, ragged tails, deeper per-warp rings.
_short = [0, 1, 17, 300, 2047, 2048, 2049, 3000]
LARGE_BATCHES = {
    "fp8": dict(name="pb-fp8", seed=21, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16, idx_q_dtype=W.FP8,
                hkv=1, group=16, k_pages=128, q_len=2, decode_lens=_short + list(range(2100, 4200, 88))[:24]),
    "fp8_h2": dict(name="pb-fp8-h2", seed=22, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16, idx_q_dtype=W.FP8,
                   hkv=2, group=8, k_pages=128, q_len=1, decode_lens=_short + list(range(2500, 5000, 100))[:24]),
    "mx": dict(name="pb-mx", seed=23, kv_dtype=W.MXFP4, idx_dtype=W.MXFP4, q_dtype=W.FP8, idx_q_dtype=W.FP8,
               hkv=1, group=16, k_pages=128, q_len=1, decode_lens=_short * 2 + list(range(2100, 6900, 100))[:48]),
    "bf16": dict(name="pb-bf16", seed=24, kv_dtype=W.BF16, idx_dtype=W.BF16, q_dtype=W.BF16, idx_q_dtype=W.BF16,
                 hkv=1, group=4, k_pages=128, q_len=4, decode_lens=[5, 2048, 2100, 2600] + [2300] * 12),
    # few rows, the widest selection: one row is cut across ~100 ranges
    "few_long": dict(name="pb-few-long", seed=25, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16,
                     idx_q_dtype=W.FP8, hkv=1, group=16, k_pages=2048, q_len=1, decode_lens=[40000, 33000, 5000]),
}


@pytest.mark.parametrize("name", list(LARGE_BATCHES))
def test_attention_large_batches(bsp, name):
    w = W.Workload(LARGE_BATCHES[name])
    o, g = OracleSide(w), GpuSide(w)
    ti, sb, ctx = o.topk(o.scores())
    ref = bf16_f32(torch.from_numpy(o.attention(sb, ctx).view(np.int16)))
    ws = bsp.decode_workspace(w.num_rows, w.k_pages, w.group)
    for call in range(2):  # the counters are back at zero after a call
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = bsp.sparse_pa_decode(g.kv, g.q, w.q_dtype, w.hq, torch.from_numpy(sb).cuda(),
                                   torch.from_numpy(ctx).cuda(), w.k_pages, SM_SCALE, ws=ws, dev_err=err)
        got = bf16_f32(out).reshape(ref.shape)
        assert err.item() == 0
        ok, worst, rl2 = attention_close(got, ref)
        print(f"{name} call {call}: rows={w.num_rows} ws={ws.numel()} worst {worst:.3g} rel-L2 {rl2:.3g}")
        assert ok, (call, worst, rl2)
        assert (got[np.repeat(ctx == 0, w.group)] == 0).all()
        if ws.numel() >= w.num_rows * 4:
            counters = ws[:w.num_rows * 4].view(torch.int32)
            assert int(counters.abs().sum().item()) == 0


@pytest.mark.parametrize("name", ["bf16", "fp8", "fp8_q4_h2", "mx", "fp8_h4", "mx_h4"])
def test_pipeline_end_to_end(bsp, name):
    """GPU path and oracle path run independently from the same inputs."""
    w, o, g = sides(name)
    ref_sc, mag = o.scores(want_absdot=True)
    ti, sb, ctx = o.topk(ref_sc)
    rs, rl = g.row_lengths()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = bsp.index_score(g.idx, g.idx_q, w.idx_q_dtype, g.block_table, rs, rl, w.q_len, w.max_pages, dev_err=err)
    gti, gsb, gctx = bsp.topk_select(sc, rs, rl, g.block_table, w.kv_dtype, w.k_pages)
    out = bsp.sparse_pa_decode(g.kv, g.q, w.q_dtype, w.hq, gsb, gctx, w.k_pages, SM_SCALE, dev_err=err)
    gti, gctx = gti.cpu().numpy(), gctx.cpu().numpy()
    same = []
    for r in range(w.num_rows):
        ok, swaps = selection_agrees(gti[r], ti[r], ref_sc[r], o.row_len[r], w.k_pages,
                                     SCORE_REL * float(mag[r].max()))
        assert ok, f"row {r}: gpu {gti[r]} oracle {ti[r]}"
        same.append(swaps == 0)
    same = np.array(same)
    assert np.array_equal(gctx[same], ctx[same])
    ref = bf16_f32(torch.from_numpy(o.attention(sb, ctx).view(np.int16))).reshape(w.num_rows, w.group, 128)
    got = bf16_f32(out).reshape(w.num_rows, w.group, 128)
    ok, mx, rl2 = attention_close(got[same], ref[same])
    assert ok, (mx, rl2)
    assert err.item() == 0
    print(f"{name}: {int((~same).sum())} rows with near-tie swaps; worst err/allowed {mx:.3g} rel-L2 {rl2:.3g}")


@pytest.mark.parametrize("name", ["fp8", "fp8_q4_h2", "mx", "bf16", "fp8_h4", "mx_h4"])
def test_decode_step_matches_ops(bsp, name):
    """bsp_sparse_decode_step == the separate calls, bit for bit."""
    from block_sparse_paged_score_gb300 import step
    w, o, g = sides(name)
    st = step.DecodeStep(w, g.kv, g.idx, g.block_table)
    k, v, ik, slot = w.step_tokens()
    st.run(g.t(k), g.t(v), g.t(ik), g.t(slot), g.q_bf16, g.idx_q_bf16, g.t(w.decode_lens))
    rs, rl = g.row_lengths()
    sc = bsp.index_score(g.idx, g.idx_q, w.idx_q_dtype, g.block_table, rs, rl, w.q_len, w.max_pages)
    gti, gsb, gctx = bsp.topk_select(sc, rs, rl, g.block_table, w.kv_dtype, w.k_pages)
    out = bsp.sparse_pa_decode(g.kv, g.q, w.q_dtype, w.hq, gsb, gctx, w.k_pages, SM_SCALE)
    assert torch.equal(st.scores, sc)
    assert torch.equal(st.sparse_bt, gsb) and torch.equal(st.sparse_ctx, gctx)
    assert torch.equal(st.out, out)
    assert st.dev_err.item() == 0


@pytest.mark.parametrize("name", ["fp8", "fp8_q4_h2"])
def test_decode_step_with_tokens_written_into_older_blocks(bsp, name):
    """New tokens need not be a sequence's last positions: here they also go
    to the first position of each sequence's first block.  The step must
    score and attend over the freshly written keys, exactly as the separate
    calls made after the write do, and the oracle agrees on page 0."""
    from block_sparse_paged_score_gb300 import step
    w = W.Workload(dict(MINI[name], seed=MINI[name]["seed"] + 900))
    g = GpuSide(w)
    k, v, ik, slot = w.step_tokens()
    rng = np.random.default_rng(7)
    seqs = [s for s in range(w.num_decode) if w.decode_lens[s] > w.q_len]  # position 0 is not a step token
    extra = np.array([w.block_table[s, 0] * W.BLOCK for s in seqs], np.int64)
    shape = (len(seqs),) + k.shape[1:]
    k2 = W.to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * 3)
    v2 = W.to_bf16_bits(rng.standard_normal(shape).astype(np.float32))
    ik2 = W.to_bf16_bits(rng.standard_normal((len(seqs),) + ik.shape[1:]).astype(np.float32) * 3)
    k, v, ik, slot = (np.concatenate([a, b]) for a, b in ((k, k2), (v, v2), (ik, ik2), (slot, extra)))
    st = step.DecodeStep(w, g.kv, g.idx, g.block_table)
    st.run(g.t(k), g.t(v), g.t(ik), g.t(slot), g.q_bf16, g.idx_q_bf16, g.t(w.decode_lens))
    rs, rl = g.row_lengths()
    sc = bsp.index_score(g.idx, g.idx_q, w.idx_q_dtype, g.block_table, rs, rl, w.q_len, w.max_pages)
    gti, gsb, gctx = bsp.topk_select(sc, rs, rl, g.block_table, w.kv_dtype, w.k_pages)
    out = bsp.sparse_pa_decode(g.kv, g.q, w.q_dtype, w.hq, gsb, gctx, w.k_pages, SM_SCALE)
    torch.cuda.synchronize()
    assert st.dev_err.item() == 0
    assert torch.equal(st.scores, sc)
    assert torch.equal(st.sparse_bt, gsb) and torch.equal(st.sparse_ctx, gctx)
    assert torch.equal(st.out, out)
    # and the oracle, written the same way, agrees on the scores of page 0
    o = OracleSide(w)
    O.kv_page_write(w.kv_dtype, w.hkv, o.kv, w.k_scale, w.v_scale, w.idx_dtype, w.hidx, o.idx, k, v, ik, slot)
    ref, mag = o.scores(want_absdot=True)
    got = sc.cpu().numpy()
    for r in range(w.num_rows):
        if o.row_len[r] > 0:
            assert abs(got[r, 0] - ref[r, 0]) <= SCORE_REL * mag[r, 0] + 1e-30, r


@pytest.mark.parametrize("name", ["fp8", "fp8_q4_h2", "mx"])
def test_decode_step_reuses_another_layers_selection(bsp, name):
    """BSP_REUSE_SELECTION: a second layer's step (its own K/V cache, no
    index cache) attends with the first layer's sparse table and writes the
    layer's new tokens.  The table is the oracle's selection for layer 1;
    layer 2's output must match the oracle's attention over layer 2's cache
    with that table (the attention tolerance), equal the attention call on
    the same table bit for bit, leave the index cache untouched, and leave
    the K/V bytes the writer's own call gives."""
    import ctypes as C
    from block_sparse_paged_score_gb300 import step
    w, o, g = sides(name)
    _, sb1, ctx1 = o.topk(o.scores())  # layer 1's selection
    sb1_d, ctx1_d = torch.from_numpy(sb1).cuda(), torch.from_numpy(ctx1).cuda()
    # layer 2: the same shapes and tokens, other values
    w2 = W.Workload(dict(MINI[name], seed=MINI[name]["seed"] + 500))
    g2, o2 = GpuSide(w2), OracleSide(w2)
    k2, v2, _, slot2 = w2.step_tokens()
    st2 = step.DecodeStep(w2, g2.kv, g2.idx, g2.block_table)
    a = st2.args
    a.idx = C.cast(None, C.POINTER(bsp.IndexCacheDesc))
    a.flags = bsp.REUSE_SELECTION
    a.sparse_bt, a.sparse_ctx = sb1_d.data_ptr(), ctx1_d.data_ptr()
    a.row_seq = a.row_len = a.scores = a.topk_idx = None
    idx_before = g2.idx.buffer.clone()
    st2.run(g2.t(k2), g2.t(v2), g2.t(k2), g2.t(slot2), g2.q_bf16, g2.q_bf16, g2.t(w2.decode_lens))
    torch.cuda.synchronize()
    assert st2.dev_err.item() == 0
    ref = bf16_f32(torch.from_numpy(o2.attention(sb1, ctx1).view(np.int16)))
    got = bf16_f32(st2.out).reshape(ref.shape)
    ok, worst, rl2 = attention_close(got, ref, label=f"{name} reuse")
    print(f"{name} reuse: worst err/1e-2 {worst:.3g} rel-L2 {rl2:.3g}")
    assert ok, (worst, rl2)
    assert (got[np.repeat(ctx1 == 0, w.group)] == 0).all()
    same = bsp.sparse_pa_decode(g2.kv, g2.q, w2.q_dtype, w2.hq, sb1_d, ctx1_d, w2.k_pages, SM_SCALE)
    torch.cuda.synchronize()
    assert torch.equal(st2.out, same)
    assert torch.equal(g2.idx.buffer, idx_before)  # no index-key write
    # the new tokens were written into layer 2's cache: the writer's own call gives the same bytes
    kv_copy = g2.kv.buffer.clone()
    bsp.kv_page_write(g2.kv, g2.idx, g2.t(k2), g2.t(v2), g2.t(k2), g2.t(slot2))
    torch.cuda.synchronize()
    assert torch.equal(g2.kv.buffer, kv_copy)
    # and they are the oracle's bytes
    assert np.array_equal(g2.kv.buffer.cpu().numpy(), o2.kv)


def test_device_errors_are_flagged_not_faulted(bsp):
    w, o, g = sides("fp8")
    rows = 4
    sb = torch.full((rows, w.k_pages), 0, dtype=torch.int32, device="cuda")
    sb[1, 0] = int(g.kv.desc.num_ids)  # out of range
    sb[2, 0] = -5
    ctx = torch.full((rows,), 16, dtype=torch.int32, device="cuda")
    q = g.q[:rows]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsp.sparse_pa_decode(g.kv, q, w.q_dtype, w.hq, sb, ctx, w.k_pages, SM_SCALE, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & 1  # BSP_DEVERR_PAGE_ID
    # a block table entry beyond the index cache
    bt = g.block_table.clone()
    bt[0, 0] = w.num_blocks + 3
    err.zero_()
    rs, rl = g.row_lengths()
    bsp.index_score(g.idx, g.idx_q, w.idx_q_dtype, bt, rs, rl, 1, w.max_pages, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & 2
    # a slot beyond the cache
    err.zero_()
    k = torch.zeros((1, w.hkv, 128), dtype=torch.int16, device="cuda")
    slot = torch.tensor([w.num_blocks * 128 + 5], dtype=torch.int64, device="cuda")
    bsp.kv_page_write(g.kv, g.idx, k, k, k[:, :w.hidx], slot, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & 16


def test_host_argument_errors(bsp):
    w, o, g = sides("fp8")
    rs, rl = g.row_lengths()
    with pytest.raises(bsp.BspError) as e:
        bsp.index_score(g.idx, g.idx_q, w.idx_q_dtype, g.block_table, rs, rl, 9, w.max_pages)  # q_group > 8
    assert e.value.status == 2
    ti, sb, ctx = o.topk(o.scores())
    with pytest.raises(bsp.BspError) as e:  # 12 query heads per KV head
        bsp.sparse_pa_decode(g.kv, g.q[:, :12].contiguous(), w.q_dtype, 12, torch.from_numpy(sb).cuda(),
                             torch.from_numpy(ctx).cuda(), w.k_pages)
    assert e.value.status == 2
    # a wide selection over few rows merges through the workspace: too small a one is refused
    sb128 = np.full((sb.shape[0], 128), -1, np.int32)
    sb128[:, :sb.shape[1]] = sb
    assert bsp.decode_workspace_bytes(sb.shape[0], 128, w.group) > 16
    with pytest.raises(bsp.BspError) as e:
        bsp.sparse_pa_decode(g.kv, g.q, w.q_dtype, w.hq, torch.from_numpy(sb128).cuda(), torch.from_numpy(ctx).cuda(),
                             128, ws=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 3
    # pinned host memory is refused, before any call, where the kernels need
    # device memory (selections, score rows); it is taken only for per-token
    # inputs and outputs
    with pytest.raises(ValueError):
        bsp.sparse_pa_decode(g.kv, g.q, w.q_dtype, w.hq, torch.from_numpy(sb).pin_memory(),
                             torch.from_numpy(ctx).cuda(), w.k_pages)
    with pytest.raises(ValueError):
        bsp.topk_select(torch.from_numpy(np.ascontiguousarray(o.scores(), np.float32)).pin_memory(), rs, rl,
                        g.block_table, w.kv_dtype, w.k_pages)


@pytest.mark.parametrize("name", ["fp8", "fp8_q4_h2", "mx"])
def test_host_step_zero_copy_matches_device_step(bsp, name):
    """The decode step fed straight from pinned host memory (its kernels load
    the inputs and store the output in place) equals the step on device
    copies, bit for bit, and so does the copy-engine host step."""
    from block_sparse_paged_score_gb300 import step
    w, o, g = sides(name)
    st = step.DecodeStep(w, g.kv, g.idx, g.block_table)
    k, v, ik, slot = w.step_tokens()
    dev = {"k": g.t(k), "v": g.t(v), "idx_k": g.t(ik), "slot": g.t(slot), "q": g.q_bf16, "idx_q": g.idx_q_bf16,
           "seq_lens": g.t(w.decode_lens)}
    st.run(dev["k"], dev["v"], dev["idx_k"], dev["slot"], dev["q"], dev["idx_q"], dev["seq_lens"])
    ref = st.out.clone()
    host = {kk: vv.cpu() for kk, vv in dev.items()}
    for inputs in ("zero", "copy"):
        for output in ("zero", "copy"):
            hs = step.HostDecodeStep(st, host, inputs=inputs, output=output)
            out = hs.run()
            torch.cuda.synchronize()
            assert st.dev_err.item() == 0
            assert torch.equal(out, ref.cpu()), (inputs, output)


def test_mixed_step_zero_copy_matches_device_step(bsp):
    """The chunked-prefill step (decode rows, prefill chunks, a pad sequence)
    fed straight from pinned host memory, and storing its output there,
    equals the step on device copies bit for bit; so does the copy-engine
    host step."""
    from block_sparse_paged_score_gb300 import step
    w, o, g = sides("mixed")
    st = step.MixedStep(w, g.kv, g.idx, g.block_table)
    k, v, ik, slot = w.step_tokens()
    dev = {"k": g.t(k), "v": g.t(v), "idx_k": g.t(ik), "slot": g.t(slot), "q": g.q_bf16, "idx_q": g.idx_q_bf16,
           "seq_lens": g.t(w.decode_lens)}
    st.run(dev["k"], dev["v"], dev["idx_k"], dev["slot"], dev["q"], dev["idx_q"], dev["seq_lens"])
    ref = st.out.clone()
    torch.cuda.synchronize()
    assert st.dev_err.item() == 0
    host = {kk: vv.cpu() for kk, vv in dev.items()}
    for inputs in ("zero", "copy"):
        for output in ("zero", "copy"):
            hs = step.HostDecodeStep(st, host, inputs=inputs, output=output)
            out = hs.run()
            torch.cuda.synchronize()
            assert st.dev_err.item() == 0
            assert torch.equal(out, ref.cpu()), (inputs, output)


@pytest.mark.parametrize("name", ["fp8", "fp8_q4_h2", "fp8_long8", "fp8_long16", "fp8_long32"])
def test_decode_step_selection_in_scorer(bsp, name):
    """With sel_counters the scorer's last CTA of each sequence selects its
    rows, with 4, 8, 16 or 32 keys per thread by the width of the rows (the
    two short workloads, then rows of 1000, 1875 and 4096 pages).  On two steps in a row (the counters are left at zero): its tables
    equal, bit for bit, the oracle's top-k run on the step's own score rows;
    the score rows are within the score bound of the oracle's; the output is
    within the attention tolerance of the oracle's attention on the step's
    tables; and everything equals the step with a separate selector."""
    from block_sparse_paged_score_gb300 import step
    w, o, g = sides(name)
    ref_sc, mag = o.scores(want_absdot=True)
    k, v, ik, slot = w.step_tokens()
    args = (g.t(k), g.t(v), g.t(ik), g.t(slot), g.q_bf16, g.idx_q_bf16, g.t(w.decode_lens))
    a = step.DecodeStep(w, g.kv, g.idx, g.block_table, select_in_scorer=False)
    b = step.DecodeStep(w, g.kv, g.idx, g.block_table, select_in_scorer=True)
    launches = []
    for _ in range(2):
        a.run(*args)
        n0 = bsp.launch_count()
        b.run(*args)
        launches.append(bsp.launch_count() - n0)
        torch.cuda.synchronize()
        assert a.dev_err.item() == 0 and b.dev_err.item() == 0
        sc = b.scores.cpu().numpy()
        ti, sb, ctx = o.topk(sc)
        assert np.array_equal(b.topk_idx.cpu().numpy(), ti)
        assert np.array_equal(b.sparse_bt.cpu().numpy(), sb)
        assert np.array_equal(b.sparse_ctx.cpu().numpy(), ctx)
        fin = ~np.isneginf(ref_sc)
        assert np.array_equal(np.isneginf(sc), ~fin)
        assert (np.abs(sc[fin] - ref_sc[fin]) <= SCORE_REL * mag[fin] + 1e-30).all()
        ref = bf16_f32(torch.from_numpy(o.attention(sb, ctx).view(np.int16)))
        ok, worst, rl2 = attention_close(bf16_f32(b.out).reshape(ref.shape), ref, label=f"{name} fused")
        assert ok, (worst, rl2)
        for x in ("scores", "topk_idx", "sparse_bt", "sparse_ctx", "out"):
            assert torch.equal(getattr(a, x), getattr(b, x)), x
        assert int(b.sel_counters.abs().sum().item()) == 0
    assert launches == [3, 3]  # prep, scorer with selection, attention


@pytest.mark.parametrize("name", ["fp8", "mx"])
def test_decode_step_in_a_cuda_graph(bsp, name):
    """The library allocates nothing and never synchronises, so a decode step
    captures into a CUDA graph (its kernels' programmatic launches included);
    replaying the graph gives the direct call's result bit for bit."""
    from block_sparse_paged_score_gb300 import step
    w, o, g = sides(name)
    st = step.DecodeStep(w, g.kv, g.idx, g.block_table)
    k, v, ik, slot = w.step_tokens()
    args = (g.t(k), g.t(v), g.t(ik), g.t(slot), g.q_bf16, g.idx_q_bf16, g.t(w.decode_lens))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        st.run(*args, stream=s)
    torch.cuda.synchronize()
    ref = st.out.clone()
    st.out.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        st.run(*args, stream=s)
    for _ in range(2):
        st.out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert st.dev_err.item() == 0
        assert torch.equal(st.out, ref)
