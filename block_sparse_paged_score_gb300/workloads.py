"""Seeded synthetic workloads of the sparse-decode path.

This module only draws inputs: context lengths, block tables (a seeded
random permutation of the physical blocks), slot mappings, and bf16 values
of the keys, values, index keys and queries.  It holds none of the method's
arithmetic (no quantisation, scoring, selection or attention), so the CUDA
path and the CPU oracle can both be fed from it.

Values are N(0, 1) drawn with numpy's PCG64 and rounded to bf16 (torch's
round-to-nearest-even cast).  MXFP4 workloads draw z * exp(u) with z ~ N(0,1)
per element and u ~ N(0, 0.5) per 32-element group, so that the groups span
a range of shared exponents.  Every (kind, sequence, 128-token block) has a
generator of its own, so any block can be regenerated alone.

The named workloads restate the shapes of the pages' deployments
(MiniMax-M3 sparse decode with 128-token blocks and 16-token pages, one KV
head and one index head per rank, 16 query heads per KV head, top-k of 2048
tokens) as concrete seeded inputs; no dataset is involved.
"""
import math

import numpy as np
import torch

BF16, FP8, MXFP4 = 0, 1, 2
BLOCK, PAGE, DIM = 128, 16, 128

KIND_K, KIND_V, KIND_IDX, KIND_Q, KIND_IDXQ, KIND_LEN, KIND_PERM, KIND_GROUP = range(8)

FP8_K_SCALE = 0.0095
FP8_V_SCALE = 0.0105

WORKLOADS = {
    1: dict(name="tiny-bf16-L1024", seed=1001, kv_dtype=BF16, idx_dtype=BF16, q_dtype=BF16, idx_q_dtype=BF16,
            hkv=1, group=4, k_pages=16, q_len=1, decode_lens=[1024]),
    2: dict(name="fp8-32seq-L4k-8k", seed=1002, kv_dtype=FP8, idx_dtype=FP8, q_dtype=BF16, idx_q_dtype=FP8,
            hkv=1, group=16, k_pages=128, q_len=1, decode_lens=("uniform", 32, 4096, 8192)),
    3: dict(name="fp8-128seq-L32k-q4", seed=1003, kv_dtype=FP8, idx_dtype=FP8, q_dtype=BF16, idx_q_dtype=FP8,
            hkv=1, group=16, k_pages=128, q_len=4, decode_lens=[32768] * 128),
    4: dict(name="mxfp4-64seq-L128k", seed=1004, kv_dtype=MXFP4, idx_dtype=MXFP4, q_dtype=FP8, idx_q_dtype=FP8,
            hkv=1, group=16, k_pages=128, q_len=1, decode_lens=[131072] * 64),
    5: dict(name="fp8-mixed-64dec-4x4096pre-8pad", seed=1005, kv_dtype=FP8, idx_dtype=FP8, q_dtype=BF16,
            idx_q_dtype=FP8, hkv=1, group=16, k_pages=128, q_len=1, decode_lens=("uniform", 64, 1024, 65536),
            prefill_chunks=[(16384, 4096), (32768, 4096), (49152, 4096), (65536, 4096)],
            pad_seqs=2, pad_q_len=4),
    # the chunked-prefill batch above with an MXFP4 index cache (the MXFP4
    # prefill scorer's workload)
    6: dict(name="fp8kv-mxfp4idx-mixed-64dec-4x4096pre-8pad", seed=1006, kv_dtype=FP8, idx_dtype=MXFP4,
            q_dtype=BF16, idx_q_dtype=FP8, hkv=1, group=16, k_pages=128, q_len=1,
            decode_lens=("uniform", 64, 1024, 65536),
            prefill_chunks=[(16384, 4096), (32768, 4096), (49152, 4096), (65536, 4096)],
            pad_seqs=2, pad_q_len=4),
}


def to_bf16_bits(x):
    """float32 array -> bf16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rng(*key):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


class Workload:
    """One batch of the path: sequences, their caches' contents and the step's queries.

    Token order of the step (and therefore of rows, token-major): decode
    tokens first (sequence s, query j -> token s*q_len + j), then the prefill
    chunks in order, then the pad rows.
    """

    def __init__(self, spec):
        self.spec = dict(spec)
        s = self.spec
        self.name = s.get("name", "custom")
        self.seed = s["seed"]
        self.kv_dtype, self.idx_dtype = s["kv_dtype"], s["idx_dtype"]
        self.q_dtype, self.idx_q_dtype = s["q_dtype"], s["idx_q_dtype"]
        self.hkv = s["hkv"]
        self.hidx = s.get("hidx", s["hkv"])
        self.group = s["group"]
        self.hq = self.hkv * self.group
        self.k_pages = s["k_pages"]
        self.q_len = s["q_len"]
        self.mx_values = self.kv_dtype == MXFP4 or self.idx_dtype == MXFP4
        self.k_scale = FP8_K_SCALE if self.kv_dtype == FP8 else 1.0
        self.v_scale = FP8_V_SCALE if self.kv_dtype == FP8 else 1.0
        self.sm_scale = float(np.float32(1.0 / math.sqrt(DIM)))

        dl = s["decode_lens"]
        if isinstance(dl, tuple) and dl[0] == "uniform":
            _, n, lo, hi = dl
            self.decode_lens = _rng(self.seed, KIND_LEN).integers(lo, hi, size=n, endpoint=True).astype(np.int32)
        else:
            self.decode_lens = np.asarray(dl, dtype=np.int32)
        self.num_decode = len(self.decode_lens)
        # prefill chunks: (context end position, tokens in the chunk)
        self.prefill_chunks = list(s.get("prefill_chunks", []))
        self.pad_seqs = s.get("pad_seqs", 0)
        self.pad_q_len = s.get("pad_q_len", 0)

        # sequences: decode, prefill, pad; seq_ctx = tokens cached once the step's tokens are written
        ctx = list(self.decode_lens) + [end for end, _ in self.prefill_chunks] + [0] * self.pad_seqs
        self.seq_ctx = np.asarray(ctx, dtype=np.int64)
        self.num_seqs = len(ctx)
        nblk = [(c + BLOCK - 1) // BLOCK for c in ctx]
        self.num_blocks = int(sum(nblk))
        self.bt_stride = max(1, max(nblk))
        perm = _rng(self.seed, KIND_PERM).permutation(self.num_blocks).astype(np.int32)
        self.block_table = np.full((self.num_seqs, self.bt_stride), -1, dtype=np.int32)
        off = 0
        for i, n in enumerate(nblk):
            self.block_table[i, :n] = perm[off:off + n]
            off += n
        self.max_pages = int(max(1, (int(self.seq_ctx.max()) + PAGE - 1) // PAGE))

        # step tokens
        self.num_decode_tokens = self.num_decode * self.q_len
        self.num_prefill_tokens = int(sum(n for _, n in self.prefill_chunks))
        self.num_pad_tokens = self.pad_seqs * self.pad_q_len
        self.num_tokens = self.num_decode_tokens + self.num_prefill_tokens + self.num_pad_tokens
        # prefill metadata (absolute sequence index into the block table, absolute position)
        req, pos = [], []
        for c, (end, n) in enumerate(self.prefill_chunks):
            req += [self.num_decode + c] * n
            pos += list(range(end - n, end))
        for p in range(self.pad_seqs):
            req += [self.num_decode + len(self.prefill_chunks) + p] * self.pad_q_len
            pos += list(range(-self.pad_q_len, 0))
        self.query_req_id = np.asarray(req, dtype=np.int32)
        self.query_abs_pos = np.asarray(pos, dtype=np.int32)
        # prefill chunk token offsets (pad sequences form chunks of their own)
        sizes = [n for _, n in self.prefill_chunks] + [self.pad_q_len] * self.pad_seqs
        self.cu_prefill = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32) if sizes else np.zeros(1, np.int32)

    # ---- values ------------------------------------------------------------
    def _heads(self, kind):
        return self.hidx if kind == KIND_IDX else self.hkv

    def block_values(self, kind, seq, b):
        """bf16 bits [128, H, 128] of block b of sequence seq (kind K, V or IDX)."""
        h = self._heads(kind)
        g = _rng(self.seed, kind, seq, b)
        x = g.standard_normal((BLOCK, h, DIM), dtype=np.float32)
        if self.mx_values:
            u = g.normal(0.0, 0.5, size=(BLOCK, h, DIM // 32)).astype(np.float32)
            x = (x.reshape(BLOCK, h, DIM // 32, 32) * np.exp(u)[..., None]).reshape(BLOCK, h, DIM)
        return to_bf16_bits(x)

    def token_values(self, kind, seq, positions):
        positions = np.asarray(positions, dtype=np.int64)
        out = np.empty((len(positions), self._heads(kind), DIM), dtype=np.uint16)
        cache = {}
        for i, p in enumerate(positions):
            b = int(p // BLOCK)
            if b not in cache:
                cache[b] = self.block_values(kind, seq, b)
            out[i] = cache[b][p % BLOCK]
        return out

    def slot(self, seq, positions):
        positions = np.asarray(positions, dtype=np.int64)
        blocks = self.block_table[seq][positions // BLOCK].astype(np.int64)
        return blocks * BLOCK + positions % BLOCK

    def context_batches(self, max_tokens=1 << 18, seqs=None):
        """Yield (k, v, idx_k, slot) covering every cached token of `seqs`
        (default all sequences), in batches of whole blocks."""
        seqs = range(self.num_seqs) if seqs is None else seqs
        ks, vs, iks, sl, n = [], [], [], [], 0
        for s in seqs:
            L = int(self.seq_ctx[s])
            for b in range((L + BLOCK - 1) // BLOCK):
                m = min(BLOCK, L - b * BLOCK)
                ks.append(self.block_values(KIND_K, s, b)[:m])
                vs.append(self.block_values(KIND_V, s, b)[:m])
                iks.append(self.block_values(KIND_IDX, s, b)[:m])
                sl.append(self.slot(s, np.arange(b * BLOCK, b * BLOCK + m)))
                n += m
                if n >= max_tokens:
                    yield np.concatenate(ks), np.concatenate(vs), np.concatenate(iks), np.concatenate(sl)
                    ks, vs, iks, sl, n = [], [], [], [], 0
        if n:
            yield np.concatenate(ks), np.concatenate(vs), np.concatenate(iks), np.concatenate(sl)

    def step_token_positions(self):
        """(seq, position) of every token the step writes, in step token order
        (pad rows write nothing and are excluded)."""
        out = []
        for s in range(self.num_decode):
            L = int(self.decode_lens[s])
            for j in range(self.q_len):
                if L - self.q_len + j >= 0:
                    out.append((s, L - self.q_len + j))
        for c, (end, n) in enumerate(self.prefill_chunks):
            for p in range(end - n, end):
                out.append((self.num_decode + c, p))
        return out

    def step_tokens(self):
        """(k, v, idx_k, slot) of the tokens the step writes."""
        pos = self.step_token_positions()
        k = np.empty((len(pos), self.hkv, DIM), np.uint16)
        v = np.empty_like(k)
        ik = np.empty((len(pos), self.hidx, DIM), np.uint16)
        slot = np.empty(len(pos), np.int64)
        by_seq = {}
        for i, (s, p) in enumerate(pos):
            by_seq.setdefault(s, []).append((i, p))
        for s, items in by_seq.items():
            idxs = [i for i, _ in items]
            ps = [p for _, p in items]
            k[idxs] = self.token_values(KIND_K, s, ps)
            v[idxs] = self.token_values(KIND_V, s, ps)
            ik[idxs] = self.token_values(KIND_IDX, s, ps)
            slot[idxs] = self.slot(s, ps)
        return k, v, ik, slot

    def queries(self):
        """bf16 bits: q [tokens, Hq, 128] and idx_q [tokens, Hidx, 128]."""
        q = _rng(self.seed, KIND_Q).standard_normal((self.num_tokens, self.hq, DIM), dtype=np.float32)
        iq = _rng(self.seed, KIND_IDXQ).standard_normal((self.num_tokens, self.hidx, DIM), dtype=np.float32)
        return to_bf16_bits(q), to_bf16_bits(iq)

    # ---- sizes -----------------------------------------------------------
    @property
    def num_rows(self):
        return self.num_tokens * self.hkv

    @property
    def num_decode_rows(self):
        return self.num_decode_tokens * self.hkv


def workload(config_id):
    return Workload(WORKLOADS[config_id])
