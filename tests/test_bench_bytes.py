"""The roofline's numerator (CPU only): the algorithmic bytes bench.py charges
a scorer or attention launch follow from the cache layouts -- one 128-token
index field or one block of K and V pages, divided by its 128 tokens -- and
from the workload's contexts, queries, score rows and outputs."""
import numpy as np
import pytest

import bench
import oracle as O
from block_sparse_paged_score_gb300 import workloads as W


@pytest.mark.parametrize("dtype", [W.BF16, W.FP8, W.MXFP4])
def test_bytes_per_token_are_the_layouts(dtype):
    w = W.Workload(dict(W.WORKLOADS[1], idx_dtype=dtype, kv_dtype=dtype, name="probe"))
    q_idx = w.num_decode_tokens * w.hidx * 128 * (2 if w.idx_q_dtype == W.BF16 else 1)
    scores = w.num_decode_tokens * w.hkv * w.max_pages * 4
    keys = int(w.decode_lens.sum()) * O.index_field_bytes(dtype) // 128 * w.hidx
    assert bench.index_algorithmic_bytes(w) == keys + q_idx + scores
    per_tok_kv = bench.attention_algorithmic_bytes(w, 1) - bench.attention_algorithmic_bytes(w, 0)
    assert per_tok_kv * 128 == O.kv_block_bytes(dtype, 1)


def test_index_and_attention_bytes_of_a_batch():
    w = W.workload(2)
    keys = int(w.decode_lens.astype(np.int64).sum()) * 132  # fp8 index: 128 B of e4m3 + a 4 B scale per token
    q_idx = 32 * 128  # e4m3 index queries, one index head
    scores = 32 * w.max_pages * 4
    assert bench.index_algorithmic_bytes(w) == keys + q_idx + scores
    ctx = 32 * 2048
    kv = ctx * 256  # fp8 K and V: 128 B each per token
    q = out = 32 * 16 * 128 * 2  # bf16 queries and output, 16 heads
    assert bench.attention_algorithmic_bytes(w, ctx) == kv + q + out


def test_smaller_decode_batch_for_captures():
    """--decode-seqs keeps the first N sequences of a decode-only workload
    under a name that says so, and refuses a chunked-prefill one."""
    full = bench.rank_workload_spec(3, 0)
    spec = bench.rank_workload_spec(3, 0, 80)
    assert spec["name"] == "fp8-80seq-L32k-q4" and full["name"] == "fp8-128seq-L32k-q4"
    assert list(spec["decode_lens"]) == list(full["decode_lens"])[:80]
    w = W.Workload(spec)
    assert w.num_decode_rows == 80 * 4
    assert bench.rank_workload_spec(3, 1, 80)["seed"] == full["seed"] + 1000
    with pytest.raises(SystemExit):
        bench.rank_workload_spec(5, 0, 8)
