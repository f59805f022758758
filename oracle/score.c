/*
 * score.c -- steps 2 and 3: row lengths and index scores (test
 * infrastructure; see bsp_oracle.h).
 *
 * Row lengths.  [ATOM-2962] "Other behaviour changes", pad-row fix (B12): the
 * causal length of a row is clamped where it enters, so that a pad row
 * (length 0, q_len > 1) computes nothing from a negative length.  Rows are
 * (token, head) pairs in token-major order ([MSA-API] forward: the emitted
 * tables hold rows token*kvh + h).  Decode token j (0-based) of a sequence of
 * length seq_len with q_len query tokens sees L = seq_len - (q_len - 1 - j);
 * a prefill token at absolute position a sees L = a + 1.  Both are clamped
 * at 0.
 *
 * Index score.  [ATOM-2962] commit "... page-128 block table": the scorers
 * produce an fp32 score per row over the row's context, read through the
 * block table, into a workspace that holds -inf where nothing is scored
 * ("the persistent score buffer equals a fresh -inf buffer").  The pages give
 * neither the formula nor the pooling, so this oracle takes the plainest
 * reading: the score of token t is the dot product of the row's index query
 * with the dequantised index key of t (no ReLU, weight or scale); the score
 * of a 16-token page is the max over its valid tokens t < L; pages at or
 * beyond ceil(L/16) score -inf.  The dequantised key is the cached value as a
 * reader sees it: bf16 exactly; fp8 as the fp32 product float(e4m3) * s_t;
 * MXFP4 as e2m1 * 2^(scale-127) (exact).  The dot product is accumulated in
 * fp64 and rounded once to fp32.
 */
#include "bsp_oracle.h"

#include <math.h>
#include <string.h>

void orc_row_lengths_decode(const int32_t* seq_lens, int num_seqs, int q_len, int num_heads,
                            int32_t* row_seq, int32_t* row_len) {
  for (int s = 0; s < num_seqs; ++s)
    for (int j = 0; j < q_len; ++j) {
      int64_t L = (int64_t)seq_lens[s] - (q_len - 1 - j);
      if (L < 0) L = 0;
      for (int h = 0; h < num_heads; ++h) {
        int64_t r = ((int64_t)s * q_len + j) * num_heads + h;
        row_seq[r] = s;
        row_len[r] = (int32_t)L;
      }
    }
}

void orc_row_lengths_prefill(const int32_t* query_req_id, const int32_t* query_abs_pos, int T,
                             int num_heads, int32_t* row_seq, int32_t* row_len) {
  for (int i = 0; i < T; ++i) {
    int64_t L = (int64_t)query_abs_pos[i] + 1;
    if (L < 0) L = 0;
    for (int h = 0; h < num_heads; ++h) {
      row_seq[(int64_t)i * num_heads + h] = query_req_id[i];
      row_len[(int64_t)i * num_heads + h] = (int32_t)L;
    }
  }
}

/* one dequantised index key (token o of the field) */
static void index_key(int idx_dtype, const uint8_t* field, int o, double* k) {
  if (idx_dtype == ORC_BF16) {
    const uint8_t* p = field + (int64_t)o * 256;
    for (int d = 0; d < ORC_DIM; ++d) {
      uint16_t b;
      memcpy(&b, p + 2 * d, 2);
      k[d] = (double)orc_bf16_decode(b);
    }
  } else if (idx_dtype == ORC_FP8) {
    float s;
    memcpy(&s, field + 16384 + o * 4, 4);
    for (int d = 0; d < ORC_DIM; ++d) {
      float kd = (float)orc_e4m3_decode(field[o * 128 + d]) * s; /* fp32 product */
      k[d] = (double)kd;
    }
  } else {
    for (int d = 0; d < ORC_DIM; ++d) {
      uint8_t byte = field[o * 64 + d / 2];
      uint8_t nib = (d & 1) ? (byte >> 4) : (byte & 15);
      k[d] = orc_e2m1_decode(nib) * orc_e8m0_decode(field[8192 + o * 4 + d / 32]);
    }
  }
}

static void query_row(const void* q, int q_dtype, int64_t row, double* out) {
  if (q_dtype == ORC_BF16) {
    const uint16_t* p = (const uint16_t*)q + row * ORC_DIM;
    for (int d = 0; d < ORC_DIM; ++d) out[d] = (double)orc_bf16_decode(p[d]);
  } else {
    const uint8_t* p = (const uint8_t*)q + row * ORC_DIM;
    for (int d = 0; d < ORC_DIM; ++d) out[d] = orc_e4m3_decode(p[d]);
  }
}

void orc_index_score(int idx_dtype, int Hidx, const uint8_t* idx, int64_t block_stride,
                     const void* q, int q_dtype,
                     const int32_t* block_table, int bt_stride,
                     const int32_t* row_seq, const int32_t* row_len, int rows, int max_pages,
                     float* scores, float* absdot, const int32_t* row_subset, int n_subset) {
  int n_work = row_subset ? n_subset : rows;
  int64_t fb = orc_index_field_bytes(idx_dtype);
#pragma omp parallel for schedule(dynamic, 1)
  for (int w = 0; w < n_work; ++w) {
    int r = row_subset ? row_subset[w] : w;
    int h = r % Hidx;
    int s = row_seq[r];
    int64_t L = row_len[r] < 0 ? 0 : row_len[r];
    double qv[ORC_DIM], kv[ORC_DIM];
    query_row(q, q_dtype, r, qv);
    float* out = scores + (int64_t)r * max_pages;
    float* mag = absdot ? absdot + (int64_t)r * max_pages : 0;
    for (int p = 0; p < max_pages; ++p) {
      out[p] = -INFINITY;
      if (mag) mag[p] = 0.0f;
    }
    for (int64_t t = 0; t < L; ++t) {
      int64_t block = block_table[(int64_t)s * bt_stride + t / ORC_BLOCK];
      const uint8_t* field = idx + block * block_stride + (int64_t)h * fb;
      index_key(idx_dtype, field, (int)(t % ORC_BLOCK), kv);
      double dot = 0.0, adot = 0.0;
      for (int d = 0; d < ORC_DIM; ++d) {
        dot += qv[d] * kv[d];
        adot += fabs(qv[d] * kv[d]);
      }
      float sc = (float)dot;
      int64_t p = t / ORC_PAGE;
      if (p >= max_pages) continue;
      if (sc > out[p]) out[p] = sc;
      if (mag && (float)adot > mag[p]) mag[p] = (float)adot;
    }
  }
}
