"""bsp_sparse_pa_decode_noalloc, the decode attention for callers that cannot
allocate device memory (for example code inside a host application that
reserves all device memory up front), against bsp_sparse_pa_decode with a
caller-owned workspace.  It runs two calls in a row on different inputs, so
the second also shows that the shared scratch carries nothing over from the
first.  Collected last so that a stop at the first failure has already run
every other test; it needs no state from them."""
import ctypes as C

import numpy as np
import pytest
import torch

from block_sparse_paged_score_gb300 import workloads as W

from harness import MINI, SM_SCALE, GpuSide, OracleSide, attention_close, bf16_f32

pytestmark = pytest.mark.gpu


def _call_noalloc(bsp, kv, q, q_dtype, hq, sbt, ctx, k_pages, out, err):
    return bsp.lib().bsp_sparse_pa_decode_noalloc(
        C.byref(kv.desc), q.data_ptr(), q_dtype, hq, sbt.data_ptr(), ctx.data_ptr(), ctx.numel(), k_pages,
        SM_SCALE, out.data_ptr(), err.data_ptr(), C.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    from block_sparse_paged_score_gb300 import bsp
    for name in ("fp8", "mx"):
        # few rows and a wide selection: the plan splits rows over more CTAs
        # than one cluster holds, so the partials go through the scratch
        w = W.Workload(dict(MINI[name], k_pages=128))
        o, g = OracleSide(w), GpuSide(w)
        ti, sb, ctx = o.topk(o.scores())
        assert bsp.decode_workspace_bytes(w.num_rows, w.k_pages, w.group) > 0  # the scratch is used
        calls = [(sb, ctx), (sb[::-1].copy(), np.minimum(ctx[::-1], 40).astype(np.int32))]
        for sbt_np, ctx_np in calls:
            sbt, c = torch.from_numpy(sbt_np).cuda(), torch.from_numpy(ctx_np).cuda()
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            ref = bsp.sparse_pa_decode(g.kv, g.q, w.q_dtype, w.hq, sbt, c, w.k_pages, SM_SCALE, dev_err=err)
            out = torch.full(ref.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
            assert _call_noalloc(bsp, g.kv, g.q, w.q_dtype, w.hq, sbt, c, w.k_pages, out, err) == 0
            torch.cuda.synchronize()
            assert err.item() == 0
            ok, worst, rl2 = attention_close(bf16_f32(out), bf16_f32(ref))
            assert ok, (name, worst, rl2)

