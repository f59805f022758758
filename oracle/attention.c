/*
 * attention.c -- step 5: attention over the selected pages, and the dense
 * attention it must equal when the selection covers every page (test
 * infrastructure; see bsp_oracle.h).
 *
 * [MSA-API] forward: decode and prefill both attend q against the K/V caches
 * through the emitted sparse block table and context lengths, with the
 * layer's softmax scale and, for an fp8 cache, the per-tensor k/v scales.
 * [vLLM-61889] Details: the kernel "carries one page id and applies it to both
 * caches", so entry m/16 of a row's table names the page of its sparse token
 * m for K and for V alike, at offset m%16.  [ATOM-2962] commit "...
 * ATOM_M3_INDEX_Q_FP8": with MXFP4 K/V the query is e4m3 and rows are
 * (token, KV head).  A row covers the G query heads h*G .. h*G+G-1 that share
 * KV head h (grouped-query attention).
 *
 * Per head: z_m = sm_scale * sum_d q_d k_{m,d}; p = softmax(z) with the max
 * subtracted; o_d = sum_m p_m v_{m,d}; all in fp64, then rounded to fp32 and
 * to bf16 (RNE).  Dequantised K/V are the values a reader of the cache sees:
 * bf16 exactly, fp8 as the fp32 product float(e4m3) * scale, MXFP4 as
 * e2m1 * 2^(scale-127).  A row with nothing to attend (context 0, the pad rows
 * of [ATOM-2962] B12 that "compute nothing") is written as zeros (reading: the
 * pages leave its output open; zeros make it defined).
 */
#include "bsp_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static double kv_elem(int kv_dtype, int Hkv, const uint8_t* kv, float k_scale, float v_scale,
                      int side, int64_t page_id, int h, int t, int d) {
  if (kv_dtype == ORC_MXFP4) {
    int64_t block = page_id / ORC_PAGES_PER_SIDE;
    int o = (int)(page_id % ORC_PAGES_PER_SIDE) * ORC_PAGE + t;
    const uint8_t* field = kv + orc_mx_field_offset(Hkv, block, side, h);
    uint8_t byte = field[o * 64 + d / 2];
    uint8_t nib = (d & 1) ? (byte >> 4) : (byte & 15);
    return orc_e2m1_decode(nib) * orc_e8m0_decode(field[8192 + o * 4 + d / 32]);
  }
  int64_t off = orc_l1_offset(kv_dtype, Hkv, side, page_id, h, t, d);
  if (kv_dtype == ORC_BF16) {
    uint16_t b;
    memcpy(&b, kv + off, 2);
    return (double)orc_bf16_decode(b);
  }
  float deq = (float)orc_e4m3_decode(kv[off]) * (side ? v_scale : k_scale); /* fp32 product */
  return (double)deq;
}

static double q_elem(const void* q, int q_dtype, int64_t head_row, int d) {
  if (q_dtype == ORC_BF16) return (double)orc_bf16_decode(((const uint16_t*)q)[head_row * ORC_DIM + d]);
  return orc_e4m3_decode(((const uint8_t*)q)[head_row * ORC_DIM + d]);
}

/* softmax attention of the G heads of row r over n tokens whose K and V are
 * given as dequantised [n][128] arrays */
static void attend(const double* K, const double* V, int64_t n, const void* q, int q_dtype, int64_t r,
                   int G, float sm_scale, uint16_t* out) {
  double* z = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int i = 0; i < G; ++i) {
    int64_t hr = r * G + i;
    uint16_t* o = out + hr * ORC_DIM;
    if (n <= 0) {
      for (int d = 0; d < ORC_DIM; ++d) o[d] = orc_bf16_encode(0.0f);
      continue;
    }
    double qv[ORC_DIM];
    for (int d = 0; d < ORC_DIM; ++d) qv[d] = q_elem(q, q_dtype, hr, d);
    double zmax = -INFINITY;
    for (int64_t m = 0; m < n; ++m) {
      double dot = 0.0;
      for (int d = 0; d < ORC_DIM; ++d) dot += qv[d] * K[m * ORC_DIM + d];
      z[m] = (double)sm_scale * dot;
      if (z[m] > zmax) zmax = z[m];
    }
    double denom = 0.0, acc[ORC_DIM];
    for (int d = 0; d < ORC_DIM; ++d) acc[d] = 0.0;
    for (int64_t m = 0; m < n; ++m) {
      double p = exp(z[m] - zmax);
      denom += p;
      for (int d = 0; d < ORC_DIM; ++d) acc[d] += p * V[m * ORC_DIM + d];
    }
    for (int d = 0; d < ORC_DIM; ++d) o[d] = orc_bf16_encode((float)(acc[d] / denom));
  }
  free(z);
}

void orc_sparse_attention(int kv_dtype, int Hkv, const uint8_t* kv, float k_scale, float v_scale,
                          const void* q, int q_dtype, int G,
                          const int32_t* sparse_bt, const int32_t* sparse_ctx, int rows, int k_pages,
                          float sm_scale, uint16_t* out, const int32_t* row_subset, int n_subset) {
  int n_work = row_subset ? n_subset : rows;
#pragma omp parallel for schedule(dynamic, 1)
  for (int w = 0; w < n_work; ++w) {
    int r = row_subset ? row_subset[w] : w;
    int h = r % Hkv;
    int64_t n = sparse_ctx[r] < 0 ? 0 : sparse_ctx[r];
    if (n > (int64_t)k_pages * ORC_PAGE) n = (int64_t)k_pages * ORC_PAGE;
    double* K = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * ORC_DIM);
    double* V = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * ORC_DIM);
    for (int64_t m = 0; m < n; ++m) {
      int64_t id = sparse_bt[(int64_t)r * k_pages + m / ORC_PAGE];
      int t = (int)(m % ORC_PAGE);
      for (int d = 0; d < ORC_DIM; ++d) {
        K[m * ORC_DIM + d] = kv_elem(kv_dtype, Hkv, kv, k_scale, v_scale, 0, id, h, t, d);
        V[m * ORC_DIM + d] = kv_elem(kv_dtype, Hkv, kv, k_scale, v_scale, 1, id, h, t, d);
      }
    }
    attend(K, V, n, q, q_dtype, r, G, sm_scale, out);
    free(K);
    free(V);
  }
}

void orc_dense_attention(int kv_dtype, int Hkv, const uint8_t* kv, float k_scale, float v_scale,
                         const void* q, int q_dtype, int G,
                         const int32_t* block_table, int bt_stride,
                         const int32_t* row_seq, const int32_t* row_len, int rows,
                         float sm_scale, uint16_t* out, const int32_t* row_subset, int n_subset) {
  int n_work = row_subset ? n_subset : rows;
#pragma omp parallel for schedule(dynamic, 1)
  for (int w = 0; w < n_work; ++w) {
    int r = row_subset ? row_subset[w] : w;
    int h = r % Hkv;
    int64_t n = row_len[r] < 0 ? 0 : row_len[r];
    double* K = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * ORC_DIM);
    double* V = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * ORC_DIM);
    for (int64_t t = 0; t < n; ++t) {
      int64_t block = block_table[(int64_t)row_seq[r] * bt_stride + t / ORC_BLOCK];
      int p = (int)((t % ORC_BLOCK) / ORC_PAGE);
      int64_t id = kv_dtype == ORC_MXFP4 ? block * ORC_PAGES_PER_SIDE + p : block * 16 + p;
      for (int d = 0; d < ORC_DIM; ++d) {
        K[t * ORC_DIM + d] = kv_elem(kv_dtype, Hkv, kv, k_scale, v_scale, 0, id, h, (int)(t % ORC_PAGE), d);
        V[t * ORC_DIM + d] = kv_elem(kv_dtype, Hkv, kv, k_scale, v_scale, 1, id, h, (int)(t % ORC_PAGE), d);
      }
    }
    attend(K, V, n, q, q_dtype, r, G, sm_scale, out);
    free(K);
    free(V);
  }
}
