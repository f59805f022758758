/*
 * layout.c -- where each cached element lives (test infrastructure; see
 * bsp_oracle.h).
 *
 * Interleaved bf16 / fp8 K/V cache ([vLLM-61889] Overview, Claims, Validation
 * and Details): a 128-token block holds 16 page slots, slots 0..7 are the K
 * pages of its 16-token pages and slots 8..15 the V pages, so the page stride
 * of a block is 16 and "a token's V pages [sit] a fixed half-block after its
 * K pages".  A page id P = block*16 + j addresses the K page at K-base + P and
 * the V page at V-base + P with V-base = K-base + 8 page slots.  The views
 * printed there, K [2048, 1, 8, 16, 16] and V [2040, 1, 1, 128, 16] per 128
 * blocks of fp8, fix the inner order of a page for one head:
 *   K: [128/x][16 tokens][x],   V: [16/x][128 dims][x],   x = 16 B / element.
 * The bf16 shapes ([16,16,8] and [2,128,8]) follow from the same x rule
 * (reading: the pages only print the fp8 views).
 *
 * MXFP4 fields ([ATOM-2962] Follow-ups): one 8704 B field per (block, KV
 * head) for K and one for V, "128 x 64 B e2m1 data, 128 x 4 B e8m0 scales".
 * Readings: data byte of (token t, dim d) at t*64 + d/2 with even d in the low
 * nibble; scale byte of (t, group g = d/32) at 8192 + t*4 + g; per block the
 * Hkv K fields come first, then the Hkv V fields.
 *
 * Index-key fields per (block, index head), token-major: bf16 128 x 256 B;
 * MXFP4 as above; fp8 (reading, the pages give no fp8 index layout):
 * 128 x 128 B e4m3 followed by 128 x 4 B fp32 per-token scales.
 */
#include "bsp_oracle.h"

static int elem_size(int kv_dtype) { return kv_dtype == ORC_BF16 ? 2 : 1; }

static int64_t page_bytes_per_head(int kv_dtype) {
  return (int64_t)ORC_PAGE * ORC_DIM * elem_size(kv_dtype);
}

int64_t orc_kv_block_bytes(int kv_dtype, int num_kv_heads) {
  if (kv_dtype == ORC_MXFP4) return (int64_t)2 * num_kv_heads * ORC_MX_FIELD_BYTES;
  return (int64_t)2 * ORC_PAGES_PER_SIDE * num_kv_heads * page_bytes_per_head(kv_dtype);
}

int64_t orc_index_field_bytes(int idx_dtype) {
  if (idx_dtype == ORC_BF16) return ORC_BF16_INDEX_FIELD_BYTES;
  if (idx_dtype == ORC_FP8) return ORC_FP8_INDEX_FIELD_BYTES;
  return ORC_MX_FIELD_BYTES;
}

int64_t orc_l1_offset(int kv_dtype, int num_kv_heads, int side, int64_t page_id, int h, int t, int d) {
  int esz = elem_size(kv_dtype);
  int x = 16 / esz;
  int64_t id_stride = (int64_t)num_kv_heads * page_bytes_per_head(kv_dtype);
  int64_t side_base = side ? (int64_t)ORC_PAGES_PER_SIDE * id_stride : 0;
  int64_t elem;
  if (side == 0)
    elem = (int64_t)(d / x) * ORC_PAGE * x + (int64_t)t * x + d % x;
  else
    elem = (int64_t)(t / x) * ORC_DIM * x + (int64_t)d * x + t % x;
  return side_base + page_id * id_stride + (int64_t)h * page_bytes_per_head(kv_dtype) + elem * esz;
}

int64_t orc_mx_field_offset(int num_kv_heads, int64_t block, int side, int h) {
  return block * orc_kv_block_bytes(ORC_MXFP4, num_kv_heads) +
         ((int64_t)side * num_kv_heads + h) * ORC_MX_FIELD_BYTES;
}
