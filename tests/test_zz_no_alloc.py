"""bsp_sparse_pa_decode_noalloc, the decode attention for callers that cannot
allocate device memory (for example code inside a host application that
reserves all device memory up front), checked two ways on two calls in a row:
bit for bit against bsp_sparse_pa_decode with a caller-owned workspace (the
same kernel and plan, so the outputs must be identical), and against the CPU
oracle's attention on the same sparse table within the attention tolerance.
The second call runs on other tables and shorter contexts, so it also shows
that the shared scratch carries nothing over from the first.  Collected last
so that a stop at the first failure has already run every other test; it
needs no state from them."""
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


@pytest.mark.parametrize("name", ["fp8", "mx"])
def test_noalloc_matches_the_workspace_entry_point_and_the_oracle_on_two_calls(name):
    from block_sparse_paged_score_gb300 import bsp
    # few rows and a wide selection: this format's plan splits each row over
    # more CTAs than one cluster holds, so the partials go through the scratch
    w = W.Workload(dict(MINI[name], k_pages=128))
    o, g = OracleSide(w), GpuSide(w)
    assert bsp.decode_splits(w.kv_dtype, w.num_rows, w.k_pages) > 8
    ti, sb, ctx = o.topk(o.scores())
    calls = [(sb, ctx), (sb[::-1].copy(), np.minimum(ctx[::-1], 40).astype(np.int32))]
    for i, (sbt_np, ctx_np) in enumerate(calls):
        sbt, c = torch.from_numpy(sbt_np).cuda(), torch.from_numpy(ctx_np).cuda()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = bsp.sparse_pa_decode(g.kv, g.q, w.q_dtype, w.hq, sbt, c, w.k_pages, SM_SCALE, dev_err=err)
        out = torch.full(ref.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(bsp, g.kv, g.q, w.q_dtype, w.hq, sbt, c, w.k_pages, out, err) == 0
        torch.cuda.synchronize()
        assert err.item() == 0
        assert torch.equal(out, ref), (name, i)
        orc = bf16_f32(torch.from_numpy(o.attention(sbt_np, ctx_np).view(np.int16))).reshape(out.shape)
        ok, worst, rl2 = attention_close(bf16_f32(out), orc, label=f"{name} call {i}")
        print(f"{name} call {i}: worst err/1e-2 {worst:.3g} rel-L2 {rl2:.3g}")
        assert ok, (name, i, worst, rl2)
