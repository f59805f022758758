"""Decode attention for any number of rows from 1 to 700.

The split-K plan of the decode attention depends on the row count: past one
wave of resident CTAs each row gets one CTA, below it a row is split over 2
to 8 CTAs of a thread-block cluster (merged on chip) or, for very few rows,
over more CTAs merged through the workspace.  The sweep below crosses every
boundary of that plan on GB300 (152 SMs).

All rows share one small cache (one sequence of 64 blocks written by the
oracle): each row's table is a seeded draw of distinct page ids of that
cache, with full, ragged and empty contexts, so the oracle's attention over
700 rows stays cheap.  Each call is compared with the oracle's attention on
the same cache bytes, queries and tables, within the attention tolerance.
One workspace serves every call, so each call must leave its arrival
counters at zero for the next.  Where the plan gives each row one CTA, the
decode call must equal the plan-free prefill call bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_paged_score_gb300 import workloads as W
from harness import SM_SCALE, OracleSide, attention_close, bf16_f32

pytestmark = pytest.mark.gpu

N_MAX = 700
K_PAGES = 128
ROWS = [1, 2, 3, 5, 8, 9, 13, 19, 20, 37, 38, 64, 75, 76, 77, 100, 151, 152, 153, 256, 303, 304, 305, 456, 457,
        607, 608, 609, 700]

CACHES = {
    "fp8": dict(name="rows-fp8", seed=31, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16, idx_q_dtype=W.FP8,
                hkv=1, group=16, k_pages=K_PAGES, q_len=1, decode_lens=[8192]),
    "mx": dict(name="rows-mx", seed=32, kv_dtype=W.MXFP4, idx_dtype=W.MXFP4, q_dtype=W.FP8, idx_q_dtype=W.FP8,
               hkv=1, group=16, k_pages=K_PAGES, q_len=1, decode_lens=[8192]),
    "bf16": dict(name="rows-bf16", seed=33, kv_dtype=W.BF16, idx_dtype=W.BF16, q_dtype=W.BF16, idx_q_dtype=W.BF16,
                 hkv=1, group=8, k_pages=K_PAGES, q_len=1, decode_lens=[8192]),
}


def _tables(w, rng):
    """N_MAX rows of distinct page ids of the cache's one sequence: most rows
    full (K_PAGES pages), some ragged, two empty (pad rows)."""
    mul = 8 if w.kv_dtype == W.MXFP4 else 16
    blocks = w.block_table[0][w.block_table[0] >= 0].astype(np.int64)
    ids = (blocks[:, None] * mul + np.arange(8)[None, :]).ravel()
    ctx = np.full(N_MAX, K_PAGES * 16, np.int32)
    short = rng.choice(N_MAX, N_MAX // 4, replace=False)
    ctx[short] = rng.integers(1, K_PAGES * 16, len(short))
    ctx[[3, N_MAX - 2]] = 0
    sb = np.full((N_MAX, K_PAGES), -1, np.int32)
    for r in range(N_MAX):
        n = (int(ctx[r]) + 15) // 16
        sb[r, :n] = rng.choice(ids, n, replace=False)
    return sb, ctx


@pytest.mark.parametrize("name", list(CACHES))
def test_attention_for_any_row_count(name):
    from block_sparse_paged_score_gb300 import bsp
    w = W.Workload(CACHES[name])
    o = OracleSide(w)
    rng = np.random.default_rng(CACHES[name]["seed"] + 100)
    sb, ctx = _tables(w, rng)
    hq = w.hkv * w.group
    q_bf16 = W.to_bf16_bits(rng.standard_normal((N_MAX, hq, 128)).astype(np.float32))
    q = q_bf16 if w.q_dtype == W.BF16 else O.cast_e4m3(q_bf16)
    ref = O.sparse_attention(w.kv_dtype, w.hkv, o.kv, w.k_scale, w.v_scale, q, w.q_dtype, w.group, sb, ctx,
                             SM_SCALE)
    ref = bf16_f32(torch.from_numpy(ref.view(np.int16))).reshape(N_MAX, w.group, 128)

    kv = bsp.KvCache(w.kv_dtype, w.hkv, w.num_blocks, w.k_scale, w.v_scale, buffer=torch.from_numpy(o.kv).cuda())
    q_dev = torch.from_numpy(q.view(np.int16) if q.dtype == np.uint16 else q).cuda()
    sb_dev, ctx_dev = torch.from_numpy(sb).cuda(), torch.from_numpy(ctx).cuda()
    ws = torch.zeros(max(16, max(bsp.decode_workspace_bytes(n, K_PAGES, w.group) for n in ROWS)),
                     dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    splits = set()
    for n in ROWS:
        out = bsp.sparse_pa_decode(kv, q_dev[:n], w.q_dtype, hq, sb_dev[:n], ctx_dev[:n], K_PAGES, SM_SCALE, ws=ws,
                                   dev_err=err)
        torch.cuda.synchronize()
        assert err.item() == 0, n
        ok, worst, rl2 = attention_close(bf16_f32(out).reshape(n, w.group, 128), ref[:n], label=f"{name} rows={n}")
        assert ok, (n, worst, rl2)
        ns = bsp.decode_splits(w.kv_dtype, n, K_PAGES)
        splits.add(ns)
        if ns == 1:
            # one CTA a row: the planned decode call equals the plan-free
            # prefill call bit for bit
            pre = bsp.sparse_pa_prefill(kv, q_dev[:n], w.q_dtype, hq, sb_dev[:n], ctx_dev[:n], K_PAGES, SM_SCALE,
                                        dev_err=err)
            torch.cuda.synchronize()
            assert err.item() == 0 and torch.equal(pre, out), n
    # the sweep reached all three ways of finishing a row
    assert 1 in splits and any(2 <= s <= 8 for s in splits) and any(s > 8 for s in splits), sorted(splits)
