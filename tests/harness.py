"""Shared set-up of the parity tests: the same seeded workload written into
the CUDA path's caches (by the CUDA writer) and into the oracle's caches (by
the oracle's writer).  Nothing here feeds a CUDA result to the oracle."""
import math

import numpy as np
import torch

import oracle as O
from block_sparse_paged_score_gb300 import workloads as W

SM_SCALE = float(np.float32(1.0 / math.sqrt(128)))

# small workloads that span several tiles, pages and blocks with ragged tails
MINI = {
    "bf16": dict(name="mini-bf16", seed=11, kv_dtype=W.BF16, idx_dtype=W.BF16, q_dtype=W.BF16, idx_q_dtype=W.BF16,
                 hkv=1, group=4, k_pages=16, q_len=1, decode_lens=[1, 15, 16, 17, 200, 333, 1024]),
    "fp8": dict(name="mini-fp8", seed=12, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16, idx_q_dtype=W.FP8,
                hkv=1, group=16, k_pages=16, q_len=1, decode_lens=[1, 15, 16, 17, 130, 300, 511, 700, 1500]),
    "fp8_q4_h2": dict(name="mini-fp8-q4-h2", seed=13, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16,
                      idx_q_dtype=W.FP8, hkv=2, group=8, k_pages=8, q_len=4, decode_lens=[0, 2, 4, 37, 129, 260, 999]),
    "fp8_bf16q": dict(name="mini-fp8-bf16q", seed=14, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16,
                      idx_q_dtype=W.BF16, hkv=1, group=2, k_pages=12, q_len=2, decode_lens=[3, 190, 640]),
    "mx": dict(name="mini-mx", seed=15, kv_dtype=W.MXFP4, idx_dtype=W.MXFP4, q_dtype=W.FP8, idx_q_dtype=W.FP8,
               hkv=1, group=16, k_pages=16, q_len=1, decode_lens=[1, 16, 33, 260, 700, 1300]),
    "mx_bf16q": dict(name="mini-mx-bf16q", seed=16, kv_dtype=W.MXFP4, idx_dtype=W.MXFP4, q_dtype=W.BF16,
                     idx_q_dtype=W.BF16, hkv=2, group=4, k_pages=8, q_len=2, decode_lens=[5, 300, 777]),
    # the longest decode query (q_len 8): full 8-row groups in every scorer
    "fp8_q8": dict(name="mini-fp8-q8", seed=18, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16, idx_q_dtype=W.FP8,
                   hkv=1, group=16, k_pages=16, q_len=8, decode_lens=[3, 8, 9, 200, 1100]),
    "mx_q8": dict(name="mini-mx-q8", seed=19, kv_dtype=W.MXFP4, idx_dtype=W.MXFP4, q_dtype=W.FP8, idx_q_dtype=W.FP8,
                  hkv=1, group=16, k_pages=16, q_len=8, decode_lens=[5, 8, 130, 1300]),
    # two KV / index heads with the tcgen05 MXFP4 scorer (e4m3 index queries)
    "mx_h2": dict(name="mini-mx-h2", seed=20, kv_dtype=W.MXFP4, idx_dtype=W.MXFP4, q_dtype=W.FP8, idx_q_dtype=W.FP8,
                  hkv=2, group=8, k_pages=16, q_len=2, decode_lens=[7, 129, 900, 2000]),
    # four KV / index heads per GPU (the deployment without tensor parallelism)
    "fp8_h4": dict(name="mini-fp8-h4", seed=40, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16, idx_q_dtype=W.FP8,
                   hkv=4, group=16, k_pages=16, q_len=2, decode_lens=[3, 200, 1300]),
    "mx_h4": dict(name="mini-mx-h4", seed=41, kv_dtype=W.MXFP4, idx_dtype=W.MXFP4, q_dtype=W.FP8, idx_q_dtype=W.FP8,
                  hkv=4, group=16, k_pages=16, q_len=2, decode_lens=[5, 260, 1100]),
    "mixed": dict(name="mini-mixed", seed=17, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16, idx_q_dtype=W.FP8,
                  hkv=1, group=16, k_pages=16, q_len=1, decode_lens=[40, 900],
                  prefill_chunks=[(384, 200), (700, 300)], pad_seqs=1, pad_q_len=4),
}

# longer decode contexts, one per width of the scorer's fused selection
# (rows up to 128 * w pages for w = 8, 16 and 32 keys per thread)
LONG = {
    "fp8_long8": dict(name="long-fp8-1000p", seed=21, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16,
                      idx_q_dtype=W.FP8, hkv=1, group=16, k_pages=128, q_len=2, decode_lens=[9000, 16000]),
    "fp8_long16": dict(name="long-fp8-1875p", seed=22, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16,
                       idx_q_dtype=W.FP8, hkv=1, group=16, k_pages=128, q_len=2, decode_lens=[2100, 30000]),
    "fp8_long32": dict(name="long-fp8-4096p", seed=23, kv_dtype=W.FP8, idx_dtype=W.FP8, q_dtype=W.BF16,
                       idx_q_dtype=W.FP8, hkv=1, group=16, k_pages=128, q_len=2, decode_lens=[40000, 65536]),
}


def mini(name):
    return W.Workload(MINI[name] if name in MINI else LONG[name])


class OracleSide:
    """The oracle's caches and queries for a workload."""

    def __init__(self, w, seqs=None):
        self.w = w
        self.kv = np.zeros(w.num_blocks * O.kv_block_bytes(w.kv_dtype, w.hkv), np.uint8)
        self.idx = np.zeros(w.num_blocks * w.hidx * O.index_field_bytes(w.idx_dtype), np.uint8)
        for k, v, ik, slot in w.context_batches(seqs=seqs):
            O.kv_page_write(w.kv_dtype, w.hkv, self.kv, w.k_scale, w.v_scale, w.idx_dtype, w.hidx, self.idx,
                            k, v, ik, slot)
        q, iq = w.queries()
        self.q_bf16, self.idx_q_bf16 = q, iq
        self.q = q if w.q_dtype == W.BF16 else O.cast_e4m3(q)
        self.idx_q = iq if w.idx_q_dtype == W.BF16 else O.cast_e4m3(iq)
        rs_d, rl_d = O.row_lengths_decode(w.decode_lens, w.q_len, w.hkv)
        if w.num_prefill_tokens + w.num_pad_tokens:
            rs_p, rl_p = O.row_lengths_prefill(w.query_req_id, w.query_abs_pos, w.hkv)
            self.row_seq, self.row_len = np.concatenate([rs_d, rs_p]), np.concatenate([rl_d, rl_p])
        else:
            self.row_seq, self.row_len = rs_d, rl_d
        self.id_rule = 1 if w.kv_dtype == W.MXFP4 else 0

    def scores(self, rows=None, want_absdot=False):
        w = self.w
        return O.index_score(w.idx_dtype, w.hidx, self.idx, self.idx_q, w.idx_q_dtype, w.block_table,
                             self.row_seq, self.row_len, w.max_pages, rows=rows, want_absdot=want_absdot)

    def topk(self, scores, rows=None):
        w = self.w
        return O.topk_select(scores, self.row_seq, self.row_len, w.block_table, self.id_rule, w.k_pages, True,
                             rows=rows)

    def attention(self, sparse_bt, sparse_ctx, rows=None):
        w = self.w
        return O.sparse_attention(w.kv_dtype, w.hkv, self.kv, w.k_scale, w.v_scale, self.q, w.q_dtype, w.group,
                                  sparse_bt, sparse_ctx, SM_SCALE, rows=rows)


class GpuSide:
    """The CUDA path's caches for a workload, written by bsp_kv_page_write."""

    def __init__(self, w, seqs=None, device="cuda"):
        from block_sparse_paged_score_gb300 import bsp
        self.bsp = bsp
        self.w = w
        self.dev = device
        self.kv = bsp.KvCache(w.kv_dtype, w.hkv, w.num_blocks, w.k_scale, w.v_scale, device=device)
        self.idx = bsp.IndexCache(w.idx_dtype, w.hidx, w.num_blocks, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        for k, v, ik, slot in w.context_batches(seqs=seqs):
            bsp.kv_page_write(self.kv, self.idx, self.t(k), self.t(v), self.t(ik), self.t(slot), dev_err=self.err)
        q, iq = w.queries()
        self.q_bf16 = self.t(q)
        self.idx_q_bf16 = self.t(iq)
        self.q = self.q_bf16 if w.q_dtype == W.BF16 else bsp.cast_e4m3(self.q_bf16)
        self.idx_q = self.idx_q_bf16 if w.idx_q_dtype == W.BF16 else bsp.cast_e4m3(self.idx_q_bf16)
        self.block_table = self.t(w.block_table)

    def t(self, a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(self.dev)
        return torch.from_numpy(a).to(self.dev)

    def row_lengths(self):
        w, bsp = self.w, self.bsp
        rs, rl = bsp.row_lengths_decode(self.t(w.decode_lens), w.q_len, w.hkv)
        if w.num_prefill_tokens + w.num_pad_tokens:
            rs2, rl2 = bsp.row_lengths_prefill(self.t(w.query_req_id), self.t(w.query_abs_pos), w.hkv)
            rs, rl = torch.cat([rs, rs2]), torch.cat([rl, rl2])
        return rs, rl


def bf16_f32(t):
    """bf16 CUDA tensor (or int16 bits) -> float32 numpy"""
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return O.bf16_to_f32(t.cpu().numpy().view(np.uint16))


def _bf16_bits(x):
    return (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.int64)


def attention_close(got, ref, max_abs=1e-2, rel_l2=5e-3, label=""):
    """The attention tolerance on bf16 outputs after identical dequantisation:
    max-abs 1e-2 and relative L2 5e-3, as stated for the path.

    Both sides round their result to bf16 at the end.  At |x| >= 2 one bf16
    spacing (2^-6) is wider than 1e-2, so two correct results that straddle
    a rounding boundary there differ by more than 1e-2.  Such elements are
    not absorbed into a wider bound: an element over 1e-2 passes only if got
    and ref are adjacent bf16 numbers of the same sign (one spacing apart,
    which exceeds 1e-2 only at |x| >= 2), and every such exception is printed
    by its flat index.  Returns (ok, worst |err| / 1e-2 over the other
    elements, rel-L2)."""
    got = np.asarray(got, np.float32)
    ref = np.asarray(ref, np.float32)
    d = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    rl2 = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    adjacent = (np.abs(_bf16_bits(got) - _bf16_bits(ref)) == 1) & (np.signbit(got) == np.signbit(ref))
    exc = (d > max_abs) & adjacent
    if exc.any():
        idx = np.flatnonzero(exc)
        print(f"attention {label}: {idx.size} one-spacing exception(s) at |x| >= 2, flat index "
              f"{idx[:20].tolist()}{' ...' if idx.size > 20 else ''}: got {got.ravel()[idx[:5]].tolist()} "
              f"ref {ref.ravel()[idx[:5]].tolist()}")
    rest = d[~exc]
    worst = float(rest.max() / max_abs) if rest.size else 0.0
    return worst <= 1.0 and rl2 <= rel_l2, worst, rl2


def selection_agrees(gpu_sel, orc_sel, orc_scores, row_len, k, bound, rel=1e-6):
    """Gap-aware comparison of one row's selections: equal sets, or every page
    in the symmetric difference scores within max(rel*|tau|, bound) of the
    oracle's threshold tau (the lowest oracle score it selected)."""
    a = set(int(p) for p in gpu_sel if p >= 0)
    b = set(int(p) for p in orc_sel if p >= 0)
    if a == b:
        return True, 0
    if len(a) != len(b):
        return False, -1
    n = (int(row_len) + 15) // 16
    cand = [p for p in b if p != n - 1]
    if not cand:
        return False, -1
    tau = min(orc_scores[p] for p in cand)
    tol = max(rel * abs(tau), bound)
    for p in a ^ b:
        if abs(orc_scores[p] - tau) > tol:
            return False, -1
    return True, len(a ^ b) // 2
