/*
 * topk.c -- step 4: per-row top-k of pages and the emitted sparse block table
 * (test infrastructure; see bsp_oracle.h).
 *
 * [ATOM-2962]: the selection runs per row over the score row and the emit
 * (_emit_sparse_block_table_row) turns the selection into a physical page
 * table plus a context length per row, clamping the causal length where it
 * enters (B12); pages_per_block is 8 for the page-16 interleaved cache and 1
 * for page-128 caches; on decode "the tail page is always selected".
 * [MSA-API] metadata builder: the page-16 rebase turns a 128-token block id B
 * into page ids at page stride 16, B*16 + j for the K side of page j; the
 * largest id at 128 blocks is 127*16 + 7 = 2039 ([vLLM-61889] Claims).
 *
 * Readings:
 *  - the unit of selection is the 16-token page and its score is the pooled
 *    page score of score.c;
 *  - with force_tail, the tail page n-1 (n = ceil(L/16)) is always selected and
 *    the other k'-1 (k' = min(k, n)) are the highest-scoring of pages
 *    0..n-2; without it the k' highest of 0..n-1; equal scores go to the lower
 *    page index;
 *  - selected logical pages are emitted in ascending order, so the tail comes
 *    last; unused table entries are -1;
 *  - physical id: interleaved cache block_table[p/8]*16 + p%8; MXFP4 cache
 *    (128-token fields, one page a block) block_table[p/8]*8 + p%8, i.e. the
 *    16-token unit p%8 of the block's field;
 *  - sparse_ctx = 16 * (number of selected full pages) + (valid tokens of the
 *    tail page if it is selected): the number of tokens the attention reads,
 *    in table order.  A row with L = 0 selects nothing and gets 0.
 */
#include "bsp_oracle.h"

#include <stdlib.h>

typedef struct {
  float score;
  int page;
} cand;

/* higher score first; equal scores: lower page first */
static int cand_cmp(const void* a, const void* b) {
  const cand* x = (const cand*)a;
  const cand* y = (const cand*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->page > y->page) - (x->page < y->page);
}

static int int_cmp(const void* a, const void* b) {
  int x = *(const int*)a, y = *(const int*)b;
  return (x > y) - (x < y);
}

void orc_topk_select(const float* scores, int rows, int max_pages,
                     const int32_t* row_seq, const int32_t* row_len,
                     const int32_t* block_table, int bt_stride, int id_rule, int k_pages, int force_tail,
                     int32_t* topk_idx, int32_t* sparse_bt, int32_t* sparse_ctx,
                     const int32_t* row_subset, int n_subset) {
  int n_work = row_subset ? n_subset : rows;
#pragma omp parallel for schedule(dynamic, 4)
  for (int w = 0; w < n_work; ++w) {
    int r = row_subset ? row_subset[w] : w;
    int64_t L = row_len[r] < 0 ? 0 : row_len[r];
    if (L > (int64_t)max_pages * ORC_PAGE) L = (int64_t)max_pages * ORC_PAGE; /* the score row ends there */
    int n = (int)((L + ORC_PAGE - 1) / ORC_PAGE);
    int kk = n < k_pages ? n : k_pages;
    int32_t* ti = topk_idx + (int64_t)r * k_pages;
    int32_t* bt = sparse_bt + (int64_t)r * k_pages;
    for (int m = 0; m < k_pages; ++m) ti[m] = bt[m] = -1;
    sparse_ctx[r] = 0;
    if (kk == 0) continue;

    const float* sr = scores + (int64_t)r * max_pages;
    int n_cand = force_tail ? n - 1 : n;
    int n_take = force_tail ? kk - 1 : kk;
    cand* c = (cand*)malloc(sizeof(cand) * (size_t)(n_cand > 0 ? n_cand : 1));
    for (int p = 0; p < n_cand; ++p) {
      c[p].score = sr[p];
      c[p].page = p;
    }
    qsort(c, (size_t)n_cand, sizeof(cand), cand_cmp);
    int* sel = (int*)malloc(sizeof(int) * (size_t)kk);
    for (int m = 0; m < n_take; ++m) sel[m] = c[m].page;
    if (force_tail) sel[kk - 1] = n - 1;
    qsort(sel, (size_t)kk, sizeof(int), int_cmp);

    int64_t ctx = 0;
    int tail_len = (int)(L - (int64_t)ORC_PAGE * (n - 1));
    for (int m = 0; m < kk; ++m) {
      int p = sel[m];
      int64_t block = block_table[(int64_t)row_seq[r] * bt_stride + p / ORC_PAGES_PER_SIDE];
      ti[m] = p;
      bt[m] = (int32_t)(id_rule == 0 ? block * 16 + p % ORC_PAGES_PER_SIDE
                                     : block * ORC_PAGES_PER_SIDE + p % ORC_PAGES_PER_SIDE);
      ctx += (p == n - 1) ? tail_len : ORC_PAGE;
    }
    sparse_ctx[r] = (int32_t)ctx;
    free(sel);
    free(c);
  }
}

/*
 * The 128-token-block variant of step 4 ([ATOM-2962], commit "... page-128
 * block table": the MXFP4 scorer keeps one fp32 per 128 tokens and the emit
 * takes pages_per_block as a parameter, so a selected unit can be a whole
 * 128-token block that expands into its pages).
 *
 * Readings:
 *  - a block's score is the largest page score among its pages below n, i.e.
 *    the largest token score in the block (max-pooling, as for pages);
 *  - the row selects kb' = min(k_pages / 8, nb) of its nb = ceil(n / 8)
 *    blocks; with force_tail the tail block nb-1 is always one of them and
 *    the other kb'-1 are the highest-scoring of blocks 0..nb-2, equal scores
 *    to the lower block; without it the kb' highest of 0..nb-1;
 *  - each selected block, in ascending order, emits its pages below n in
 *    ascending order, with the same page ids as the page-granular emit; so
 *    the table holds at most 8 * kb' <= k_pages entries, and only the last
 *    block of the row can contribute fewer than 8;
 *  - sparse_ctx counts the tokens the table covers, as for pages.
 */
void orc_topk_select_blocks(const float* scores, int rows, int max_pages,
                            const int32_t* row_seq, const int32_t* row_len,
                            const int32_t* block_table, int bt_stride, int id_rule, int k_pages, int force_tail,
                            int32_t* topk_idx, int32_t* sparse_bt, int32_t* sparse_ctx,
                            const int32_t* row_subset, int n_subset) {
  int n_work = row_subset ? n_subset : rows;
#pragma omp parallel for schedule(dynamic, 4)
  for (int w = 0; w < n_work; ++w) {
    int r = row_subset ? row_subset[w] : w;
    int64_t L = row_len[r] < 0 ? 0 : row_len[r];
    if (L > (int64_t)max_pages * ORC_PAGE) L = (int64_t)max_pages * ORC_PAGE;
    int n = (int)((L + ORC_PAGE - 1) / ORC_PAGE);
    int nb = (n + ORC_PAGES_PER_SIDE - 1) / ORC_PAGES_PER_SIDE;
    int kb = k_pages / ORC_PAGES_PER_SIDE;
    if (kb > nb) kb = nb;
    int32_t* ti = topk_idx + (int64_t)r * k_pages;
    int32_t* bt = sparse_bt + (int64_t)r * k_pages;
    for (int m = 0; m < k_pages; ++m) ti[m] = bt[m] = -1;
    sparse_ctx[r] = 0;
    if (kb == 0) continue;

    const float* sr = scores + (int64_t)r * max_pages;
    int n_cand = force_tail ? nb - 1 : nb;
    int n_take = force_tail ? kb - 1 : kb;
    cand* c = (cand*)malloc(sizeof(cand) * (size_t)(n_cand > 0 ? n_cand : 1));
    for (int b = 0; b < n_cand; ++b) {
      float best = sr[b * ORC_PAGES_PER_SIDE];
      for (int p = b * ORC_PAGES_PER_SIDE + 1; p < (b + 1) * ORC_PAGES_PER_SIDE && p < n; ++p)
        if (sr[p] > best) best = sr[p];
      c[b].score = best;
      c[b].page = b; /* the block index */
    }
    qsort(c, (size_t)n_cand, sizeof(cand), cand_cmp);
    int* sel = (int*)malloc(sizeof(int) * (size_t)kb);
    for (int m = 0; m < n_take; ++m) sel[m] = c[m].page;
    if (force_tail) sel[kb - 1] = nb - 1;
    qsort(sel, (size_t)kb, sizeof(int), int_cmp);

    int64_t ctx = 0;
    int tail_len = (int)(L - (int64_t)ORC_PAGE * (n - 1));
    int m = 0;
    for (int i = 0; i < kb; ++i) {
      int b = sel[i];
      int64_t block = block_table[(int64_t)row_seq[r] * bt_stride + b];
      for (int p = b * ORC_PAGES_PER_SIDE; p < (b + 1) * ORC_PAGES_PER_SIDE && p < n; ++p, ++m) {
        ti[m] = p;
        bt[m] = (int32_t)(id_rule == 0 ? block * 16 + p % ORC_PAGES_PER_SIDE
                                       : block * ORC_PAGES_PER_SIDE + p % ORC_PAGES_PER_SIDE);
        ctx += (p == n - 1) ? tail_len : ORC_PAGE;
      }
    }
    sparse_ctx[r] = (int32_t)ctx;
    free(sel);
    free(c);
  }
}
