"""Pins of the oracle's row lengths, index scores, top-k and attention:
a hand-worked example, brute force with numpy/torch on tiny inputs (an
independent formulation of each step), and the invariants the pages state
(pad rows compute nothing, the tail page is always selected, the largest
page id at 128 blocks is 2039, sparse attention equals dense attention when
the selection covers every page)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
E2M1 = {int(c): float(v) for c, v in (l.split() for l in open(os.path.join(GOLD, "e2m1_codes.txt"))
                                      if l.strip() and not l.startswith("#"))}


def bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def e4m3_vals(b):
    return torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


# ---- independent dequantisation (numpy / torch, not the oracle) ------------
def deq_index(idx_dtype, idx, blk, h, hidx):
    fb = {O.BF16: 32768, O.FP8: 16896, O.MXFP4: 8704}[idx_dtype]
    f = idx[(blk * hidx + h) * fb:(blk * hidx + h + 1) * fb]
    if idx_dtype == O.BF16:
        return O.bf16_to_f32(f.view(np.uint16).reshape(128, 128)).astype(np.float64)
    if idx_dtype == O.FP8:
        s = f[16384:].view(np.float32)
        return (e4m3_vals(f[:16384]).reshape(128, 128).astype(np.float32) * s[:, None]).astype(np.float64)
    return deq_mx(f)


def deq_mx(f):
    data = f[:8192].reshape(128, 64)
    lo, hi = data & 15, data >> 4
    nib = np.stack([lo, hi], -1).reshape(128, 128)
    vals = np.vectorize(E2M1.get)(nib)
    sc = 2.0 ** (f[8192:].reshape(128, 4).astype(np.float64) - 127)
    return vals * np.repeat(sc, 32, axis=1)


def make_index(idx_dtype, hidx, nblk, T, rng):
    idx = np.zeros(nblk * hidx * O.index_field_bytes(idx_dtype), np.uint8)
    kv = np.zeros(nblk * O.kv_block_bytes(O.FP8, 1), np.uint8)
    slots = np.arange(T, dtype=np.int64)
    x = rng.standard_normal((T, hidx, 128))
    if idx_dtype == O.MXFP4:
        x = x * np.exp(rng.normal(0, 0.5, (T, hidx, 4, 1))).repeat(32, -1).reshape(T, hidx, 128)
    z = np.zeros((T, 1, 128), np.uint16)
    O.kv_page_write(O.FP8, 1, kv, 1.0, 1.0, idx_dtype, hidx, idx, z, z, bf16(x), slots)
    return idx


# ---- row lengths ----------------------------------------------------------
def test_row_lengths_decode_clamps_pad_rows():
    # ATOM 2962 B12: a pad row (length 0, q > 1) computes nothing
    rs, rl = O.row_lengths_decode(np.array([10, 0, 2], np.int32), 4, 2)
    assert rl.reshape(3, 4, 2)[0, :, 0].tolist() == [7, 8, 9, 10]
    assert rl.reshape(3, 4, 2)[1].tolist() == [[0, 0]] * 4
    assert rl.reshape(3, 4, 2)[2, :, 1].tolist() == [0, 0, 1, 2]
    assert rs.reshape(3, 4, 2)[2].tolist() == [[2, 2]] * 4


def test_row_lengths_prefill():
    rs, rl = O.row_lengths_prefill(np.array([3, 3, 5], np.int32), np.array([0, 17, -2], np.int32), 1)
    assert rs.tolist() == [3, 3, 5] and rl.tolist() == [1, 18, 0]


# ---- index score ----------------------------------------------------------
def test_score_hand_example():
    rows = [l.split() for l in open(os.path.join(GOLD, "score_hand_example.txt"))
            if l.strip() and not l.startswith("#")]
    for ex, L, page, expect in rows:
        L, page, expect = int(L), int(page), float(expect)
        k = np.zeros((2, 1, 128), np.float32)
        q = np.zeros((1, 1, 128), np.float32)
        q[0, 0, :2] = [1, 2]
        if ex == "A":
            k[0, 0, :2] = [3, -1]
            k[1, 0, :2] = [2, 1.5]
            dt, qb, qd = O.BF16, bf16(q), O.BF16
        else:
            k[0, 0, :2] = [7, 3.5]
            dt, qb, qd = O.FP8, O.cast_e4m3(bf16(q)), O.FP8
        idx = np.zeros(O.index_field_bytes(dt), np.uint8)
        kv = np.zeros(O.kv_block_bytes(O.FP8, 1), np.uint8)
        O.kv_page_write(O.FP8, 1, kv, 1.0, 1.0, dt, 1, idx, bf16(k), bf16(k), bf16(k), np.array([0, 1], np.int64))
        sc = O.index_score(dt, 1, idx, qb, qd, np.zeros((1, 1), np.int32), np.zeros(1, np.int32),
                           np.array([L], np.int32), 2)
        assert sc[0, page] == expect


@pytest.mark.parametrize("idx_dtype,q_dtype", [(O.BF16, O.BF16), (O.FP8, O.FP8), (O.FP8, O.BF16),
                                               (O.MXFP4, O.FP8), (O.MXFP4, O.BF16)])
def test_score_brute_force(idx_dtype, q_dtype):
    rng = np.random.default_rng(5)
    hidx, nblk = 2, 5
    idx = make_index(idx_dtype, hidx, nblk, nblk * 128, rng)
    # two sequences over a permuted block table
    perm = rng.permutation(nblk).astype(np.int32)
    bt = np.array([perm[:3], np.r_[perm[3:], -1]], np.int32)
    tokens = 3
    q = bf16(rng.standard_normal((tokens, hidx, 128)))
    qb = q if q_dtype == O.BF16 else O.cast_e4m3(q)
    qv = O.bf16_to_f32(q).astype(np.float64) if q_dtype == O.BF16 else e4m3_vals(qb)
    row_seq = np.repeat(np.array([0, 1, 0], np.int32), hidx)
    row_len = np.repeat(np.array([300, 200, 17], np.int32), hidx)
    max_pages = 24
    sc, ad = O.index_score(idx_dtype, hidx, idx, qb, q_dtype, bt, row_seq, row_len, max_pages, want_absdot=True)
    for r in range(tokens * hidx):
        h, s, L = r % hidx, row_seq[r], row_len[r]
        keys = np.concatenate([deq_index(idx_dtype, idx, bt[s, b], h, hidx) for b in range((L + 127) // 128)])[:L]
        tok = (keys @ qv.reshape(-1, 128)[r]).astype(np.float32)
        n = (L + 15) // 16
        for p in range(max_pages):
            if p < n:
                ref = tok[16 * p:16 * p + 16].max()
                assert sc[r, p] == pytest.approx(ref, rel=1e-6, abs=1e-30)
                mag = np.abs(keys[16 * p:16 * p + 16] * qv.reshape(-1, 128)[r]).sum(1).max()
                assert ad[r, p] == pytest.approx(mag, rel=1e-6)
            else:
                assert sc[r, p] == -np.inf


# ---- top-k ----------------------------------------------------------------
def brute_topk(s, L, k, force_tail=True):
    n = min((L + 15) // 16, len(s))
    kk = min(k, n)
    if kk == 0:
        return []
    cand = n - 1 if force_tail else n
    order = np.lexsort((np.arange(cand), -s[:cand].astype(np.float64)))
    take = list(order[:kk - 1 if force_tail else kk])
    if force_tail:
        take.append(n - 1)
    return sorted(int(p) for p in take)


@pytest.mark.parametrize("force_tail", [True, False])
def test_topk_brute_force_with_ties(force_tail):
    rng = np.random.default_rng(6)
    rows, max_pages, k = 60, 40, 7
    sc = rng.integers(-3, 4, (rows, max_pages)).astype(np.float32)  # many exact ties
    sc[::7] = 0.0
    sc[3, ::2] = -0.0
    L = rng.integers(0, max_pages * 16 + 1, rows).astype(np.int32)
    L[:4] = [0, 1, 16, 17]
    bt = rng.permutation(100).astype(np.int32).reshape(-1, 5)[:rows] if False else \
        np.tile(np.arange(5, dtype=np.int32) * 3 + 1, (rows, 1))
    rs = np.arange(rows, dtype=np.int32)
    ti, sb, ctx = O.topk_select(sc, rs, L, bt, 0, k, force_tail)
    for r in range(rows):
        sel = brute_topk(sc[r], L[r], k, force_tail)
        assert ti[r, :len(sel)].tolist() == sel and (ti[r, len(sel):] == -1).all()
        n = (L[r] + 15) // 16
        exp_ctx = sum(16 if p != n - 1 else L[r] - 16 * (n - 1) for p in sel)
        assert ctx[r] == exp_ctx
        assert sb[r, :len(sel)].tolist() == [int(bt[r, p // 8]) * 16 + p % 8 for p in sel]


def test_topk_invariants_and_mx_id_rule():
    rng = np.random.default_rng(7)
    rows, max_pages = 30, 64
    sc = rng.standard_normal((rows, max_pages)).astype(np.float32)
    L = rng.integers(1, max_pages * 16 + 1, rows).astype(np.int32)
    bt = rng.permutation(8 * rows).astype(np.int32).reshape(rows, 8)
    ti, sb, ctx = O.topk_select(sc, np.arange(rows, dtype=np.int32), L, bt, 1, 16, True)
    for r in range(rows):
        n = (L[r] + 15) // 16
        sel = ti[r][ti[r] >= 0]
        assert len(sel) == min(16, n) and len(set(sel)) == len(sel)
        assert (np.diff(sel) > 0).all() and sel[-1] == n - 1 and sel.max() < n
        assert sb[r, :len(sel)].tolist() == [int(bt[r, p // 8]) * 8 + p % 8 for p in sel]
        # every unselected candidate scores no higher than every selected non-tail page
        cand = set(range(n - 1)) - set(sel.tolist())
        if cand and len(sel) > 1:
            assert max(sc[r, list(cand)]) <= min(sc[r, sel[:-1]])


def test_max_page_id_at_128_blocks_is_2039():
    g = {l.split()[0]: l.split()[1] for l in open(os.path.join(GOLD, "page_geometry.txt"))
         if l.strip() and not l.startswith("#")}
    L = 128 * 128
    bt = np.arange(128, dtype=np.int32)[None, :]
    sc = np.zeros((1, 1024), np.float32)
    ti, sb, ctx = O.topk_select(sc, np.zeros(1, np.int32), np.array([L], np.int32), bt, 0, 1024, True)
    assert sb.max() == int(g["max_page_id_128_blocks"]) == 127 * 16 + 7
    assert sb.max() < int(g["blocks_128_v_view"].split(",")[0])
    assert ctx[0] == L and (ti[0] == np.arange(1024)).all()


# ---- attention ------------------------------------------------------------
def make_cache(kv_dtype, hkv, nblk, rng, kfun=None):
    kv = np.zeros(nblk * O.kv_block_bytes(kv_dtype, hkv), np.uint8)
    T = nblk * 128
    k = rng.standard_normal((T, hkv, 128)) if kfun is None else kfun(T)
    v = rng.standard_normal((T, hkv, 128))
    ks, vs = (0.0095, 0.0105) if kv_dtype == O.FP8 else (1.0, 1.0)
    idx = np.zeros(nblk * hkv * 16896, np.uint8)
    O.kv_page_write(kv_dtype, hkv, kv, ks, vs, O.FP8, hkv, idx, bf16(k), bf16(v), None,
                    np.arange(T, dtype=np.int64))
    return kv, ks, vs


def deq_kv(kv_dtype, hkv, kv, ks, vs, side, pid, h):
    """[16, 128] dequantised K (side 0) or V (side 1) of page id pid, head h."""
    if kv_dtype == O.MXFP4:
        blk, u = divmod(pid, 8)
        f = kv[O.mx_field_offset(hkv, blk, side, h):][:8704]
        return deq_mx(f)[16 * u:16 * u + 16]
    if kv_dtype == O.BF16:
        w = kv.view(np.uint16)
        base = (side * 8 * hkv + pid * hkv + h) * 2048
        pg = O.bf16_to_f32(w[base:base + 2048]).astype(np.float64)
        return pg.reshape(16, 16, 8).transpose(1, 0, 2).reshape(16, 128) if side == 0 else \
            pg.reshape(2, 128, 8).transpose(0, 2, 1).reshape(16, 128)
    base = (side * 8 * hkv + pid * hkv + h) * 2048
    pg = e4m3_vals(kv[base:base + 2048]).astype(np.float32) * np.float32(vs if side else ks)
    pg = pg.astype(np.float64)
    return pg.reshape(8, 16, 16).transpose(1, 0, 2).reshape(16, 128) if side == 0 else \
        pg.reshape(128, 16).T


@pytest.mark.parametrize("kv_dtype,q_dtype", [(O.BF16, O.BF16), (O.FP8, O.BF16), (O.MXFP4, O.FP8)])
def test_sparse_attention_brute_force(kv_dtype, q_dtype):
    rng = np.random.default_rng(8)
    hkv, G, nblk = 2, 4, 3
    kv, ks, vs = make_cache(kv_dtype, hkv, nblk, rng)
    rows, kp = 4 * hkv, 5
    pages_total = nblk * 8
    sbt = np.full((rows, kp), -1, np.int32)
    ctx = np.array([0, 1, 37, 80, 16, 5, 70, 33], np.int32)
    for r in range(rows):
        n = (ctx[r] + 15) // 16
        lp = np.sort(rng.choice(pages_total, n, replace=False))
        sbt[r, :n] = [(p // 8) * (16 if kv_dtype != O.MXFP4 else 8) + p % 8 for p in lp]
    q = bf16(rng.standard_normal((rows // hkv, hkv * G, 128)))
    qb = q if q_dtype == O.BF16 else O.cast_e4m3(q)
    qv = (O.bf16_to_f32(q).astype(np.float64) if q_dtype == O.BF16 else e4m3_vals(qb)).reshape(rows * G, 128)
    sm = np.float32(1 / math.sqrt(128))
    out = O.bf16_to_f32(O.sparse_attention(kv_dtype, hkv, kv, ks, vs, qb, q_dtype, G, sbt, ctx, float(sm)))
    for r in range(rows):
        h = r % hkv
        n = ctx[r]
        if n == 0:
            assert (out[r * G:(r + 1) * G] == 0).all()
            continue
        K = np.concatenate([deq_kv(kv_dtype, hkv, kv, ks, vs, 0, sbt[r, m], h) for m in range((n + 15) // 16)])[:n]
        V = np.concatenate([deq_kv(kv_dtype, hkv, kv, ks, vs, 1, sbt[r, m], h) for m in range((n + 15) // 16)])[:n]
        for i in range(G):
            z = float(sm) * (K @ qv[r * G + i])
            p = np.exp(z - z.max())
            o = (p @ V) / p.sum()
            ref = O.bf16_to_f32(bf16(o.astype(np.float32)))
            got = out[r * G + i]
            ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
            assert (np.abs(got - ref) <= ulp).all()


def test_attention_one_token_and_identical_keys():
    rng = np.random.default_rng(9)
    kv, _, _ = make_cache(O.BF16, 1, 1, rng, kfun=lambda T: np.ones((T, 1, 128)))
    q = bf16(rng.standard_normal((1, 4, 128)))
    sm = float(np.float32(1 / math.sqrt(128)))
    # L = 1: the output is that token's V
    out1 = O.sparse_attention(O.BF16, 1, kv, 1.0, 1.0, q, O.BF16, 4, np.array([[3]], np.int32),
                              np.array([1], np.int32), sm)
    w = kv.view(np.uint16)
    v_tok0 = np.array([w[(8 + 3) * 2048 + (0 // 8) * 1024 + d * 8 + 0] for d in range(128)], np.uint16)
    assert (out1 == v_tok0[None]).all()
    # identical keys: softmax is uniform, output = mean of the selected V
    out2 = O.bf16_to_f32(O.sparse_attention(O.BF16, 1, kv, 1.0, 1.0, q, O.BF16, 4, np.array([[0, 5]], np.int32),
                                            np.array([32], np.int32), sm))
    V = np.concatenate([deq_kv(O.BF16, 1, kv, 1, 1, 1, pid, 0) for pid in (0, 5)])
    mean = O.bf16_to_f32(bf16(V.mean(0).astype(np.float32)))
    assert (np.abs(out2 - mean[None]) <= np.abs(mean) * 2 ** -8 + 1e-6).all()


@pytest.mark.parametrize("kv_dtype", [O.BF16, O.FP8, O.MXFP4])
def test_sparse_equals_dense_when_every_page_is_selected(kv_dtype):
    """Top-k covering every page (k*16 >= L) emits every page in order, so the
    sparse attention reads exactly the dense context."""
    rng = np.random.default_rng(10)
    nblk, hkv, G = 4, 1, 4
    kv, ks, vs = make_cache(kv_dtype, hkv, nblk, rng)
    bt = rng.permutation(nblk).astype(np.int32)[None, :]
    L = np.array([1, 100, 300, 512], np.int32)
    rs = np.zeros(4, np.int32)
    sc = rng.standard_normal((4, 32)).astype(np.float32)
    ti, sb, ctx = O.topk_select(sc, rs, L, bt, 1 if kv_dtype == O.MXFP4 else 0, 32, True)
    assert (ctx == L).all()
    q = bf16(rng.standard_normal((4, G, 128)))
    qd = O.BF16
    sm = float(np.float32(1 / math.sqrt(128)))
    sp = O.sparse_attention(kv_dtype, hkv, kv, ks, vs, q, qd, G, sb, ctx, sm)
    dn = O.dense_attention(kv_dtype, hkv, kv, ks, vs, q, qd, G, bt, rs, L, sm)
    assert np.array_equal(sp, dn)


def test_pad_rows_compute_nothing():
    rng = np.random.default_rng(11)
    kv, ks, vs = make_cache(O.FP8, 1, 1, rng)
    rs, rl = O.row_lengths_decode(np.array([0], np.int32), 4, 1)
    sc = O.index_score(O.FP8, 1, np.zeros(16896, np.uint8), O.cast_e4m3(bf16(np.ones((4, 1, 128)))), O.FP8,
                       np.zeros((1, 1), np.int32), rs, rl, 8)
    assert (sc == -np.inf).all()
    ti, sb, ctx = O.topk_select(sc, rs, rl, np.zeros((1, 1), np.int32), 0, 4, True)
    assert (ctx == 0).all() and (ti == -1).all() and (sb == -1).all()
    out = O.sparse_attention(O.FP8, 1, kv, ks, vs, bf16(np.ones((4, 16, 128))), O.BF16, 16, sb, ctx, 0.1)
    assert (out == 0).all()
