/*
 * bsp_oracle.h -- plain, slow CPU oracle for indexer-selected block-sparse
 * paged-attention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This library exists so that the test-suite, the
 * package smoke check and the benchmark's CPU-baseline leg can check the CUDA
 * path against an independent statement of what the path computes.  Nothing
 * in the product (the CUDA library and its Python binding) includes, links or
 * calls it, and it includes nothing of theirs.
 *
 * Every routine is written from the pages' statement of the method, in the
 * pages' order, with no blocking, fusion or reordering:
 *   [vLLM-61889]  vLLM pull request 61889, "MiniMax-M3 LBHNC sparse decode"
 *                 (sections Overview, Claims, Validation, Details);
 *   [ATOM-2962]   ROCm/ATOM pull request 2962, "[MiniMax-M3.1] MXFP4 index
 *                 cache and MXFP4 KV cache" (PR description, "Other behaviour
 *                 changes", "Known limits", "Follow-ups", commit messages);
 *   [MSA-API]     vLLM API docs, vllm.models.minimax_m3.amd.sparse_attention_msa
 *                 (MiniMaxM3SparseAiterPAImpl.forward and
 *                 MiniMaxM3SparseAiterPAMetadataBuilder).
 * Where the pages leave a step open, the reading taken is stated at the
 * routine.  Floating point is carried in fp64 except where the pages' data
 * formats fix a narrower type (the stored e4m3 / e2m1 / e8m0 / bf16 bytes,
 * the fp32 per-token index scale, the fp32 page score).
 *
 * Parity status per routine (see the test-suite for each pin):
 *   codecs, layouts, write, row lengths, index score, top-k and emission
 *   (page- and block-granular), sparse and dense attention: pinned.
 *   The following readings are fixed by this oracle and the GPU path is only
 *   checked for consistency with them ("parity unpinned" in the sense that the
 *   pages print no worked example for them): max-pooling of token scores into
 *   a 16-token page score, the MXFP4 shared-exponent rule, the nibble order
 *   inside an MXFP4 byte, the fp8 index-key scale granularity (one fp32 scale
 *   per token), forcing the tail page into every selection, and the
 *   page-id rule for MXFP4 caches.
 *
 * All pointers are host pointers.  Buffers are caller-owned.
 */
#ifndef BSP_ORACLE_H
#define BSP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cache / operand formats */
enum { ORC_BF16 = 0, ORC_FP8 = 1, ORC_MXFP4 = 2 };

/* sizes fixed by the pages: 128-token blocks ([vLLM-61889] server command
 * "--block-size 128"), 16-token pages ([MSA-API] "page-16"), 8 pages per block
 * side, head_dim 128 (K view [.., 8, 16, 16] in [vLLM-61889] Validation). */
#define ORC_BLOCK 128
#define ORC_PAGE 16
#define ORC_PAGES_PER_SIDE 8
#define ORC_DIM 128
#define ORC_MX_FIELD_BYTES 8704   /* [ATOM-2962] Follow-ups: 128x64 B + 128x4 B */
#define ORC_FP8_INDEX_FIELD_BYTES 16896 /* reading: 128x128 B e4m3 + 128x4 B fp32 */
#define ORC_BF16_INDEX_FIELD_BYTES 32768

/* ---- codecs ---------------------------------------------------------- */
uint8_t orc_e4m3_encode(float x);          /* RNE, saturating to +-448 */
double orc_e4m3_decode(uint8_t b);
uint8_t orc_e2m1_encode(double x);         /* 4-bit code, RNE, saturating to +-6 */
double orc_e2m1_decode(uint8_t nibble);
double orc_e8m0_decode(uint8_t b);         /* 2^(b-127) */
uint16_t orc_bf16_encode(float x);         /* RNE */
float orc_bf16_decode(uint16_t b);
/* shared exponent of one 32-element MXFP4 group: the e8m0 byte */
uint8_t orc_mx_scale_byte(const float* x, int n);

/* e4m3 unit-scale saturating cast of n bf16 values (the writer's q output) */
void orc_cast_e4m3(const uint16_t* x_bf16, uint8_t* out, int64_t n);

/* ---- layouts --------------------------------------------------------- */
int64_t orc_kv_block_bytes(int kv_dtype, int num_kv_heads);
int64_t orc_index_field_bytes(int idx_dtype);
/* byte offset of K (side 0) / V (side 1) element (token t of page id P,
 * head h, dim d) in a bf16/fp8 interleaved cache; for bf16 the offset of the
 * 2-byte element. */
int64_t orc_l1_offset(int kv_dtype, int num_kv_heads, int side, int64_t page_id, int h, int t, int d);
/* MXFP4: offset of the field of (block, side, head) */
int64_t orc_mx_field_offset(int num_kv_heads, int64_t block, int side, int h);

/* ---- step 1: write ----------------------------------------------------- */
/* Quantise and scatter T tokens.  k, v: bf16 [T, Hkv, 128]; idx_k: bf16
 * [T, Hidx, 128] or NULL; slot: [T], slot = block*128 + offset, -1 skips. */
void orc_kv_page_write(int kv_dtype, int num_kv_heads, uint8_t* kv_cache, float k_scale, float v_scale,
                       int idx_dtype, int num_idx_heads, uint8_t* idx_cache,
                       const uint16_t* k, const uint16_t* v, const uint16_t* idx_k,
                       const int64_t* slot, int T);

/* ---- step 2: row lengths ---------------------------------------------- */
void orc_row_lengths_decode(const int32_t* seq_lens, int num_seqs, int q_len, int num_heads,
                            int32_t* row_seq, int32_t* row_len);
void orc_row_lengths_prefill(const int32_t* query_req_id, const int32_t* query_abs_pos, int T,
                             int num_heads, int32_t* row_seq, int32_t* row_len);

/* ---- step 3: index score ---------------------------------------------- */
/* scores[r, p] for rows r = token*Hidx + h; q: [tokens, Hidx, 128] (bf16 bits
 * or e4m3 bytes).  If absdot != NULL it receives, per (row, page), the largest
 * sum_d |q_d k_d| over the page's valid tokens (0 where the page is empty).
 * row_subset (nullable): compute only these rows. */
void orc_index_score(int idx_dtype, int num_idx_heads, const uint8_t* idx_cache, int64_t block_stride,
                     const void* q, int q_dtype,
                     const int32_t* block_table, int bt_stride,
                     const int32_t* row_seq, const int32_t* row_len, int rows, int max_pages,
                     float* scores, float* absdot, const int32_t* row_subset, int n_subset);

/* ---- step 4: top-k and block-table emission ---------------------------- */
/* id_rule: 0 = interleaved page-16 cache (block*16 + p%8), 1 = MXFP4 page-128
 * cache (block*8 + p%8). */
void orc_topk_select(const float* scores, int rows, int max_pages,
                     const int32_t* row_seq, const int32_t* row_len,
                     const int32_t* block_table, int bt_stride, int id_rule, int k_pages, int force_tail,
                     int32_t* topk_idx, int32_t* sparse_bt, int32_t* sparse_ctx,
                     const int32_t* row_subset, int n_subset);

/* The same with 128-token blocks as the unit of selection: k_pages / 8
 * blocks per row, each emitting its pages (see topk.c). */
void orc_topk_select_blocks(const float* scores, int rows, int max_pages,
                            const int32_t* row_seq, const int32_t* row_len,
                            const int32_t* block_table, int bt_stride, int id_rule, int k_pages, int force_tail,
                            int32_t* topk_idx, int32_t* sparse_bt, int32_t* sparse_ctx,
                            const int32_t* row_subset, int n_subset);

/* ---- step 5: attention ------------------------------------------------- */
/* q: [tokens, Hkv*G, 128] (bf16 bits or e4m3 bytes); out: bf16 bits, same
 * shape.  Row r = token*Hkv + h covers q heads h*G .. h*G+G-1. */
void orc_sparse_attention(int kv_dtype, int num_kv_heads, const uint8_t* kv_cache, float k_scale, float v_scale,
                          const void* q, int q_dtype, int group,
                          const int32_t* sparse_bt, const int32_t* sparse_ctx, int rows, int k_pages,
                          float sm_scale, uint16_t* out, const int32_t* row_subset, int n_subset);
/* the same softmax over logical tokens 0..L-1 read through the block table */
void orc_dense_attention(int kv_dtype, int num_kv_heads, const uint8_t* kv_cache, float k_scale, float v_scale,
                         const void* q, int q_dtype, int group,
                         const int32_t* block_table, int bt_stride,
                         const int32_t* row_seq, const int32_t* row_len, int rows,
                         float sm_scale, uint16_t* out, const int32_t* row_subset, int n_subset);

/* threads the oracle's OpenMP loops use (1 when built without OpenMP) */
int orc_num_threads(void);
/* sets the threads of the oracle's later OpenMP loops (n > 0; no-op without
   OpenMP); for timing the oracle on one core */
void orc_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
