"""Parity of the 128-token-block selection (BSP_SELECT_BLOCKS) with the
oracle (GPU required): bit-exact tables on tie-heavy rows for every
blocks-per-thread variant, on the oracle's scores of the small workloads, and
the decode step with the flag against the separate calls and the oracle's
attention on the emitted table."""
import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_paged_score_gb300 import workloads as W

from harness import MINI, SM_SCALE, GpuSide, OracleSide, attention_close, bf16_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsp():
    from block_sparse_paged_score_gb300 import bsp as b
    b.lib()
    return b


def run_gpu(bsp, sc, rs, L, bt, kv_dtype, k, force_tail):
    flags = bsp.SELECT_BLOCKS | (bsp.FORCE_TAIL if force_tail else 0)
    t = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    gti, gsb, gctx = bsp.topk_select(t(sc), t(rs), t(L), t(bt), kv_dtype, k, flags=flags)
    return gti.cpu().numpy(), gsb.cpu().numpy(), gctx.cpu().numpy()


# blocks per row 13 .. 8192: every blocks-per-thread variant (1, 2, 4, 8, 16
# and 32 blocks a thread at 256 threads: 13-256, 500, 1000, 2000, 3750, 5000
# and 8192 blocks)
@pytest.mark.parametrize("max_pages", [100, 2048, 4000, 8000, 16000, 30000, 40000, 65536])
@pytest.mark.parametrize("force_tail", [True, False])
@pytest.mark.parametrize("kv_dtype", [W.FP8, W.MXFP4])
def test_block_select_bit_exact_with_ties(bsp, force_tail, kv_dtype, max_pages):
    rng = np.random.default_rng(max_pages + 7 * force_tail)
    rows = 200 if max_pages <= 8192 else 24
    sc = rng.integers(-4, 5, (rows, max_pages)).astype(np.float32)  # heavy ties between block maxima
    sc[::5] = rng.standard_normal((len(sc[::5]), max_pages)).astype(np.float32)
    sc[7, ::3] = -0.0
    sc[8] = 0.0
    L = rng.integers(0, max_pages * 16 + 1, rows).astype(np.int32)
    L[:7] = [0, 1, 16, 129, 1025, max_pages * 16, max_pages * 16 - 1]
    nblk = (max_pages + 7) // 8
    bt = np.stack([rng.permutation(4 * nblk)[:nblk] for _ in range(rows)]).astype(np.int32)
    rs = np.arange(rows, dtype=np.int32)
    for k in (8, 15, 40, 128, 2048):
        ref = O.topk_select_blocks(sc, rs, L, bt, 1 if kv_dtype == W.MXFP4 else 0, k, force_tail)
        got = run_gpu(bsp, sc, rs, L, bt, kv_dtype, k, force_tail)
        for a, b, what in zip(got, ref, ("topk_idx", "sparse_bt", "sparse_ctx")):
            assert np.array_equal(a, b), (k, what)


@pytest.mark.parametrize("name", [n for n in MINI if MINI[n]["k_pages"] >= 8])
def test_block_select_on_oracle_scores(bsp, name):
    w = W.Workload(MINI[name])
    o, g = OracleSide(w), GpuSide(w)
    ref = o.scores()
    ti, sb, ctx = O.topk_select_blocks(ref, o.row_seq, o.row_len, w.block_table, o.id_rule, w.k_pages, True)
    rs, rl = g.row_lengths()
    gti, gsb, gctx = bsp.topk_select(torch.from_numpy(ref).cuda(), rs, rl, g.block_table, w.kv_dtype, w.k_pages,
                                     flags=bsp.FORCE_TAIL | bsp.SELECT_BLOCKS)
    assert np.array_equal(gti.cpu().numpy(), ti)
    assert np.array_equal(gsb.cpu().numpy(), sb)
    assert np.array_equal(gctx.cpu().numpy(), ctx)


@pytest.mark.parametrize("name", ["fp8", "fp8_q4_h2", "mx"])
def test_decode_step_with_block_selection(bsp, name):
    """The decode step with BSP_SELECT_BLOCKS equals the separate calls bit for
    bit, and its attention over the block table is within the attention
    tolerance of the oracle fed the same table."""
    from block_sparse_paged_score_gb300 import step
    w = W.Workload(dict(MINI[name], seed=MINI[name]["seed"] + 300))
    o, g = OracleSide(w), GpuSide(w)
    st = step.DecodeStep(w, g.kv, g.idx, g.block_table)
    st.args.flags = bsp.FORCE_TAIL | bsp.SELECT_BLOCKS
    k, v, ik, slot = w.step_tokens()
    st.run(g.t(k), g.t(v), g.t(ik), g.t(slot), g.q_bf16, g.idx_q_bf16, g.t(w.decode_lens))
    rs, rl = g.row_lengths()
    sc = bsp.index_score(g.idx, g.idx_q, w.idx_q_dtype, g.block_table, rs, rl, w.q_len, w.max_pages)
    gti, gsb, gctx = bsp.topk_select(sc, rs, rl, g.block_table, w.kv_dtype, w.k_pages,
                                     flags=bsp.FORCE_TAIL | bsp.SELECT_BLOCKS)
    out = bsp.sparse_pa_decode(g.kv, g.q, w.q_dtype, w.hq, gsb, gctx, w.k_pages, SM_SCALE)
    torch.cuda.synchronize()
    assert st.dev_err.item() == 0
    assert torch.equal(st.sparse_bt, gsb) and torch.equal(st.sparse_ctx, gctx) and torch.equal(st.topk_idx, gti)
    assert torch.equal(st.out, out)
    # the table itself is the oracle's block selection of the GPU's scores
    ti, sb, ctx = O.topk_select_blocks(sc.cpu().numpy(), o.row_seq, o.row_len, w.block_table, o.id_rule,
                                       w.k_pages, True)
    assert np.array_equal(gsb.cpu().numpy(), sb) and np.array_equal(gctx.cpu().numpy(), ctx)
    ref = bf16_f32(torch.from_numpy(o.attention(sb, ctx).view(np.int16))).reshape(w.num_rows, w.group, 128)
    ok, worst, rl2 = attention_close(bf16_f32(out).reshape(w.num_rows, w.group, 128), ref)
    assert ok, (worst, rl2)


def test_block_select_needs_eight_pages(bsp):
    sc = torch.zeros((2, 16), dtype=torch.float32, device="cuda")
    z = torch.zeros(2, dtype=torch.int32, device="cuda")
    bt = torch.zeros((2, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError):
        bsp.topk_select(sc, z, z, bt, W.FP8, 7, flags=bsp.SELECT_BLOCKS)
