"""The benchmark workloads have the shapes they are named for (CPU only): the
sequence counts and context lengths, heads, top-k, cache and query formats,
the chunked-prefill batch with its pad rows, the decode-first token order,
block tables that are a permutation of the physical blocks, and the value
recipe (N(0, 1); MXFP4 workloads scaled per 32-element group)."""
import numpy as np
import pytest

from block_sparse_paged_score_gb300 import workloads as W


def test_tiny_bf16():
    w = W.workload(1)
    assert (w.num_decode, w.q_len, w.hkv, w.group, w.k_pages) == (1, 1, 1, 4, 16)
    assert list(w.decode_lens) == [1024] and w.max_pages == 64
    assert (w.kv_dtype, w.idx_dtype, w.q_dtype, w.idx_q_dtype) == (W.BF16,) * 4


def test_fp8_32_sequences_of_4k_to_8k():
    w = W.workload(2)
    assert (w.num_decode, w.q_len, w.hkv, w.group, w.k_pages) == (32, 1, 1, 16, 128)
    assert w.k_pages * W.PAGE == 2048
    assert ((w.decode_lens >= 4096) & (w.decode_lens <= 8192)).all() and len(set(w.decode_lens)) > 16
    assert (w.kv_dtype, w.idx_dtype, w.q_dtype, w.idx_q_dtype) == (W.FP8, W.FP8, W.BF16, W.FP8)


def test_fp8_128_sequences_of_32k_with_four_query_tokens():
    w = W.workload(3)
    assert (w.num_decode, w.q_len, w.hkv, w.group, w.k_pages) == (128, 4, 1, 16, 128)
    assert (w.decode_lens == 32768).all() and w.num_rows == 512
    assert (w.kv_dtype, w.idx_dtype) == (W.FP8, W.FP8)


def test_mxfp4_64_sequences_of_128k():
    w = W.workload(4)
    assert (w.num_decode, w.q_len, w.hkv, w.group, w.k_pages) == (64, 1, 1, 16, 128)
    assert (w.decode_lens == 131072).all() and w.max_pages == 8192
    assert (w.kv_dtype, w.idx_dtype, w.q_dtype, w.idx_q_dtype) == (W.MXFP4, W.MXFP4, W.FP8, W.FP8)


@pytest.mark.parametrize("config", [5, 6])
def test_chunked_prefill_batch(config):
    w = W.workload(config)
    assert w.num_decode == 64 and ((w.decode_lens >= 1024) & (w.decode_lens <= 65536)).all()
    assert [n for _, n in w.prefill_chunks] == [4096] * 4
    assert max(end for end, _ in w.prefill_chunks) <= 65536
    assert w.num_pad_tokens == 8 and w.pad_q_len > 1
    # decode tokens first, then the chunks in order, then the pad rows (negative positions: length 0)
    assert w.num_tokens == 64 + 4 * 4096 + 8
    pos = w.query_abs_pos
    assert (pos[:4 * 4096] >= 0).all() and (pos[4 * 4096:] < 0).all()
    for c, (end, n) in enumerate(w.prefill_chunks):
        assert list(pos[c * 4096:(c + 1) * 4096]) == list(range(end - n, end))
        assert (w.query_req_id[c * 4096:(c + 1) * 4096] == 64 + c).all()
    assert list(w.cu_prefill) == [0, 4096, 8192, 12288, 16384, 16388, 16392]
    assert w.idx_dtype == (W.FP8 if config == 5 else W.MXFP4)


@pytest.mark.parametrize("config", [1, 2, 3, 4, 5, 6])
def test_block_tables_are_a_permutation_of_the_physical_blocks(config):
    w = W.workload(config)
    used = w.block_table[w.block_table >= 0]
    assert sorted(used.tolist()) == list(range(w.num_blocks))
    for s, L in enumerate(w.seq_ctx):
        n = (int(L) + W.BLOCK - 1) // W.BLOCK
        assert (w.block_table[s, :n] >= 0).all() and (w.block_table[s, n:] == -1).all()
    # a seeded shuffle, not the identity
    assert not np.array_equal(used, np.sort(used)) or w.num_blocks < 4


def _f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_value_recipe():
    x = _f32(W.workload(2).block_values(W.KIND_K, 0, 0)).reshape(128, 1, 4, 32)
    assert abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1.0) < 0.05
    m = W.workload(4)
    y = _f32(m.block_values(W.KIND_K, 0, 0)).reshape(128, 1, 4, 32)
    # per 32-element group a scale exp(u), u ~ N(0, 0.5): the log-spread of the groups varies about 4x more
    # than N(0, 1) values alone give (sd 0.52 against 0.13)
    assert 0.35 < float(np.log(y.std(axis=-1)).std()) < 0.7
    assert float(np.log(x.std(axis=-1)).std()) < 0.2
    # the same (kind, sequence, block) always draws the same values
    assert np.array_equal(m.block_values(W.KIND_K, 3, 7), W.workload(4).block_values(W.KIND_K, 3, 7))
