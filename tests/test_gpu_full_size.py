"""Parity at the benchmark's full sizes (GPU required): each workload's step
runs exactly as bench.py runs it -- the CUDA writer fills every sequence's
caches, then one DecodeStep (workloads 2-4) or MixedStep (workloads 5-6).
Every row's length, and every row's selection (top-k pages, page ids and
context length) is checked bit for bit against the oracle's top-k run on the
GPU's own score rows.  A sample of rows is then checked against the oracle,
which writes and scores only the sampled sequences:
  cache bytes of the sampled sequences' blocks equal, byte for byte;
  page scores within 2e-5 * sum_d |q_d k_d|, the same -inf pattern;
  selections equal up to near-ties (gap-aware);
  attention outputs within max-abs 1e-2 and relative-L2 5e-3 of the oracle
  fed the GPU's sparse table.
"""
import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_paged_score_gb300 import workloads as W

from harness import SM_SCALE, attention_close, bf16_f32, selection_agrees

pytestmark = pytest.mark.gpu

SCORE_REL = 2e-5


def _sample_rows(w, rng):
    nd = w.num_decode_rows
    rows = {0, nd - 1, nd // 2} | set(int(x) for x in rng.integers(0, nd, 3))
    if w.q_len > 1:  # every query token of one sequence
        s = int(rng.integers(0, w.num_decode))
        rows |= {(s * w.q_len + j) * w.hkv for j in range(w.q_len)}
    if w.num_rows > nd:  # prefill rows of several chunks, and the last (pad) row
        rows |= set(int(x) for x in rng.integers(nd, w.num_rows, 4)) | {w.num_rows - 1}
    return np.array(sorted(rows), np.int32)


@pytest.mark.parametrize("config", [2, 3, 4, 5, 6])
def test_full_size_step_on_sampled_rows(config):
    from block_sparse_paged_score_gb300 import bsp, step
    w = W.workload(config)
    dev = "cuda"

    def t(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    # the GPU side, as bench.py runs it
    kv = bsp.KvCache(w.kv_dtype, w.hkv, w.num_blocks, w.k_scale, w.v_scale, device=dev)
    idx = bsp.IndexCache(w.idx_dtype, w.hidx, w.num_blocks, device=dev)
    for k, v, ik, slot in w.context_batches():
        bsp.kv_page_write(kv, idx, t(k), t(v), t(ik), t(slot))
    bt = t(w.block_table)
    k, v, ik, slot = w.step_tokens()
    q, iq = w.queries()
    st = (step.MixedStep if w.prefill_chunks else step.DecodeStep)(w, kv, idx, bt, device=dev)
    st.run(t(k), t(v), t(ik), t(slot), t(q), t(iq), t(w.decode_lens))
    torch.cuda.synchronize()
    assert st.dev_err.item() == 0

    # every row: the row lengths, and the selection the oracle's top-k makes
    # from the GPU's own score rows, bit for bit (table ids and lengths too)
    rs_all, rl_all = O.row_lengths_decode(w.decode_lens, w.q_len, w.hkv)
    if w.num_rows > w.num_decode_rows:
        rs_p, rl_p = O.row_lengths_prefill(w.query_req_id, w.query_abs_pos, w.hkv)
        rs_all, rl_all = np.concatenate([rs_all, rs_p]), np.concatenate([rl_all, rl_p])
    assert np.array_equal(st.row_seq.cpu().numpy(), rs_all)
    assert np.array_equal(st.row_len.cpu().numpy(), rl_all)
    got = st.scores.cpu().numpy()
    ti_all, sb_all, ctx_all = O.topk_select(got, rs_all, rl_all, w.block_table, 1 if w.kv_dtype == W.MXFP4 else 0,
                                            w.k_pages, True)
    for name, ref_t, gpu_t in (("topk_idx", ti_all, st.topk_idx), ("sparse_bt", sb_all, st.sparse_bt),
                               ("sparse_ctx", ctx_all, st.sparse_ctx)):
        g_np = gpu_t.cpu().numpy()
        bad = np.flatnonzero((g_np != ref_t).reshape(len(g_np), -1).any(axis=1))
        assert bad.size == 0, f"{name}: {bad.size} of {len(g_np)} rows differ, first {bad[:8].tolist()}"
    print(f"workload {config}: selections of all {w.num_rows} rows bit-exact against the oracle's top-k")

    # the oracle side on the sampled rows' sequences
    rows = _sample_rows(w, np.random.default_rng(config))
    seqs = sorted(set(int(rs_all[r]) for r in rows))
    okv = np.zeros(w.num_blocks * O.kv_block_bytes(w.kv_dtype, w.hkv), np.uint8)
    oidx = np.zeros(w.num_blocks * w.hidx * O.index_field_bytes(w.idx_dtype), np.uint8)
    for kk, vv, ikk, sl in w.context_batches(seqs=seqs):
        O.kv_page_write(w.kv_dtype, w.hkv, okv, w.k_scale, w.v_scale, w.idx_dtype, w.hidx, oidx, kk, vv, ikk, sl)
    keep = np.array([i for i, (s, _) in enumerate(w.step_token_positions()) if s in seqs], np.int64)
    if len(keep):
        O.kv_page_write(w.kv_dtype, w.hkv, okv, w.k_scale, w.v_scale, w.idx_dtype, w.hidx, oidx, k[keep], v[keep],
                        ik[keep], slot[keep])

    # cache bytes of the sampled sequences' blocks
    kb, ib = O.kv_block_bytes(w.kv_dtype, w.hkv), w.hidx * O.index_field_bytes(w.idx_dtype)
    blocks = np.concatenate([w.block_table[s, :(int(w.seq_ctx[s]) + W.BLOCK - 1) // W.BLOCK] for s in seqs])
    blocks = blocks.astype(np.int64)
    if len(blocks):
        bi = torch.from_numpy(blocks).to(dev)
        kv_gpu = kv.buffer.view(w.num_blocks, kb)[bi].cpu().numpy()
        idx_gpu = idx.buffer.view(w.num_blocks, ib)[bi].cpu().numpy()
        assert np.array_equal(kv_gpu, okv.reshape(w.num_blocks, kb)[blocks])
        assert np.array_equal(idx_gpu, oidx.reshape(w.num_blocks, ib)[blocks])

    # scores and selections
    iq_o = iq if w.idx_q_dtype == W.BF16 else O.cast_e4m3(iq)
    ref, mag = O.index_score(w.idx_dtype, w.hidx, oidx, iq_o, w.idx_q_dtype, w.block_table, rs_all, rl_all,
                             w.max_pages, rows=rows, want_absdot=True)
    ti, _, _ = O.topk_select(ref, rs_all, rl_all, w.block_table, 1 if w.kv_dtype == W.MXFP4 else 0, w.k_pages, True,
                             rows=rows)
    gti = st.topk_idx.cpu().numpy()
    for r in rows:
        fin = ~np.isneginf(ref[r])
        assert np.array_equal(np.isneginf(got[r]), ~fin), r
        assert (np.abs(got[r][fin] - ref[r][fin]) <= SCORE_REL * mag[r][fin] + 1e-30).all(), r
        ok, _ = selection_agrees(gti[r], ti[r], ref[r], rl_all[r], w.k_pages, SCORE_REL * float(mag[r].max()))
        assert ok, (r, gti[r], ti[r])

    # attention of the sampled rows on the GPU's own table
    q_o = q if w.q_dtype == W.BF16 else O.cast_e4m3(q)
    sb_gpu, ctx_gpu = st.sparse_bt.cpu().numpy(), st.sparse_ctx.cpu().numpy()
    out_ref = O.sparse_attention(w.kv_dtype, w.hkv, okv, w.k_scale, w.v_scale, q_o, w.q_dtype, w.group, sb_gpu,
                                 ctx_gpu, SM_SCALE, rows=rows)
    ref_o = O.bf16_to_f32(out_ref).reshape(-1, w.group, 128)[rows]
    got_o = bf16_f32(st.out).reshape(-1, w.group, 128)[rows]
    ok, worst, rl2 = attention_close(got_o, ref_o, label=f"workload {config}")
    print(f"workload {config}: {len(rows)} rows, attention worst err/1e-2 {worst:.3g}, rel-L2 {rl2:.3g}")
    assert ok, (worst, rl2)
