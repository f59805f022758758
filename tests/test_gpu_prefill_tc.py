"""Parity of the tcgen05 prefill index scorers with the oracle (GPU required):
fp8 and MXFP4 index caches, e4m3 index queries, chunks of consecutive query
tokens with causal lengths, partial 128-row tiles, several 8192-key ranges and
pad rows."""
import numpy as np
import pytest
import torch

from block_sparse_paged_score_gb300 import workloads as W

from harness import GpuSide, OracleSide

pytestmark = pytest.mark.gpu

SCORE_REL = 2e-5

CASES = {
    "small": dict(name="pre-small", seed=21, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16, idx_q_dtype=W.FP8,
                  hkv=1, group=16, k_pages=16, q_len=1, decode_lens=[40],
                  prefill_chunks=[(384, 200), (700, 300)], pad_seqs=1, pad_q_len=4),
    "ranges": dict(name="pre-ranges", seed=22, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16, idx_q_dtype=W.FP8,
                   hkv=1, group=16, k_pages=32, q_len=1, decode_lens=[5000],
                   prefill_chunks=[(3000, 700), (5200, 1100), (128, 128)], pad_seqs=2, pad_q_len=4),
    # contexts past 8192 keys: several key ranges per query tile
    "wide": dict(name="pre-wide", seed=23, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16, idx_q_dtype=W.FP8,
                 hkv=1, group=16, k_pages=32, q_len=1, decode_lens=[100],
                 prefill_chunks=[(9100, 300), (17000, 260)], pad_seqs=1, pad_q_len=4),
    # MXFP4 index cache (e2m1 keys, e8m0 per 32 dims): the same shapes
    "mx_small": dict(name="pre-mx-small", seed=24, kv_dtype=W.MXFP4, idx_dtype=W.MXFP4, q_dtype=W.FP8,
                     idx_q_dtype=W.FP8, hkv=1, group=16, k_pages=16, q_len=1, decode_lens=[40],
                     prefill_chunks=[(384, 200), (700, 300)], pad_seqs=1, pad_q_len=4),
    "mx_ranges": dict(name="pre-mx-ranges", seed=25, kv_dtype=W.MXFP4, idx_dtype=W.MXFP4, q_dtype=W.FP8,
                      idx_q_dtype=W.FP8, hkv=1, group=16, k_pages=32, q_len=1, decode_lens=[5000],
                      prefill_chunks=[(3000, 700), (5200, 1100), (128, 128)], pad_seqs=2, pad_q_len=4),
    "mx_wide": dict(name="pre-mx-wide", seed=26, kv_dtype=W.MXFP4, idx_dtype=W.MXFP4, q_dtype=W.FP8,
                    idx_q_dtype=W.FP8, hkv=1, group=16, k_pages=32, q_len=1, decode_lens=[100],
                    prefill_chunks=[(9100, 300), (17000, 260)], pad_seqs=1, pad_q_len=4),
}


@pytest.mark.parametrize("case", list(CASES))
def test_prefill_scores_match_oracle(case):
    from block_sparse_paged_score_gb300 import bsp
    w = W.Workload(CASES[case])
    o, g = OracleSide(w), GpuSide(w)
    nd = w.num_decode_tokens
    rows = np.arange(nd, w.num_rows, dtype=np.int32)
    ref, mag = o.scores(rows=rows, want_absdot=True)
    ref, mag = ref[nd:], mag[nd:]
    rs, rl = g.row_lengths()
    cu = g.t(w.cu_prefill)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = bsp.index_score_prefill(g.idx, g.idx_q[nd:], w.idx_q_dtype, g.block_table, rs[nd:], rl[nd:], cu,
                                 len(w.cu_prefill) - 1, bsp.prefill_tiles(w.cu_prefill), w.max_pages, dev_err=err)
    got = sc.cpu().numpy()
    assert err.item() == 0, err.item()
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = ~np.isneginf(ref)
    diff = np.abs(got[fin] - ref[fin])
    ratio = float((diff / np.maximum(mag[fin], 1e-30)).max())
    print(f"{case}: max |err|/sum|qk| = {ratio:.3g} over {int(fin.sum())} pages")
    assert (diff <= SCORE_REL * mag[fin] + 1e-30).all(), ratio
