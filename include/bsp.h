/*
 * bsp.h -- C ABI of libbsp: indexer-selected block-sparse paged-attention
 * decode on NVIDIA GB300 (sm_103a).
 *
 * The operation follows three public pages:
 *   [vLLM-61889]  vLLM pull request 61889, "MiniMax-M3 LBHNC sparse decode":
 *                 the interleaved K/V cache, its K and V views, one page id for
 *                 both caches, the largest page id 127*16+7 = 2039 at 128
 *                 blocks (Overview, Claims, Validation, Details);
 *   [ATOM-2962]   ROCm/ATOM pull request 2962, "[MiniMax-M3.1] MXFP4 index
 *                 cache and MXFP4 KV cache": MXFP4 pages (e2m1 + one e8m0 per
 *                 32, 8704 B per 128-token page), the fused writer, the index
 *                 scorers, the selector, the block-table emission and the pad-row
 *                 clamp (PR description, "Other behaviour changes", commit
 *                 messages);
 *   [MSA-API]     vLLM API docs, vllm.models.minimax_m3.amd.sparse_attention_msa:
 *                 MiniMaxM3SparseAiterPAImpl.forward (decode and prefill calls,
 *                 decode-first rows, token-major (token, kv head) rows) and the
 *                 metadata builder's page-16 rebase.
 *
 * One step of the path is
 *     bsp_kv_page_write -> bsp_row_lengths_* -> bsp_index_score(_prefill)
 *       -> bsp_topk_select -> bsp_sparse_pa_decode / bsp_sparse_pa_prefill
 * and bsp_sparse_decode_step runs it as one call.
 *
 * Conventions shared by every call
 *  - Fixed sizes: 128-token blocks, 16-token pages, 8 pages per block side,
 *    head_dim 128 (the index key dim is 128 too).  Query heads per KV head
 *    G in {1, 2, 4, 8, 16}.  Anything else returns BSP_ERR_UNSUPPORTED.
 *  - Rows.  A row is one (query token, KV head) pair, numbered token-major:
 *    row = token * num_heads + head ([MSA-API] forward).  The index cache has
 *    one index head per KV head in the shapes this library is built for, but
 *    the index calls take their own head count.
 *  - Memory.  Every pointer to data is a DEVICE pointer unless stated; the
 *    caller owns every buffer (including workspaces).  The per-token inputs and
 *    the output, which the kernels touch once with plain loads and stores, may
 *    instead point into pinned host memory (page-locked, which unified
 *    addressing maps into the device's address space; the kernels then read
 *    and write it in place over the host link): bsp_kv_page_write's k, v,
 *    idx_k and slot; bsp_cast_e4m3's x and out; bsp_row_lengths_decode's
 *    seq_lens; the attention calls' q and out; the step inputs and out of
 *    bsp_sparse_decode_step.  Caches, block tables, score rows, selections and
 *    workspaces must be device memory (the kernels read them by TMA or more
 *    than once).  The library never allocates, never synchronises the stream
 *    and never reads device memory back to the host inside a call, so every
 *    call may be captured into a CUDA graph.  All work is enqueued on `stream`
 *    (0 = legacy default stream).
 *  - Errors.  Invalid arguments are detected on the host and returned before
 *    anything is enqueued.  A failed launch returns BSP_ERR_CUDA (the CUDA
 *    error stays readable through bsp_last_cuda_error).  Data-dependent
 *    faults the host cannot see (a page or block id out of range, rows of one
 *    query group that disagree on their sequence) are handled on the device:
 *    the access is skipped and a bit is OR-ed into *dev_err when dev_err is
 *    not NULL (see BSP_DEVERR_*).  No kernel traps and no kernel waits on
 *    another kernel; the library's few internal waits (TMA completion) are
 *    bounded and report BSP_DEVERR_TIMEOUT.
 *  - Alignment.  Cache bases, strides and every tensor base must be 16-byte
 *    aligned (TMA bulk copies); checked on the host.
 */
#ifndef BSP_H
#define BSP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* bsp_stream_t; /* the same type as cudaStream_t */
typedef struct CUevent_st* bsp_event_t;   /* the same type as cudaEvent_t */

typedef enum {
  BSP_OK = 0,
  BSP_ERR_INVALID_ARG = 1, /* a NULL pointer, a negative size, misalignment */
  BSP_ERR_UNSUPPORTED = 2, /* a size or dtype outside what is built */
  BSP_ERR_WORKSPACE = 3,   /* the workspace is smaller than the *_workspace_bytes query */
  BSP_ERR_CUDA = 4         /* a CUDA call failed; see bsp_last_cuda_error */
} bsp_status;

typedef enum {
  BSP_BF16 = 0,     /* bfloat16 */
  BSP_FP8_E4M3 = 1, /* OCP e4m3 (e4m3fn), saturating casts */
  BSP_MXFP4 = 2     /* e2m1 data + one e8m0 scale per 32 elements */
} bsp_dtype;

/* device error bits (OR-ed into *dev_err) */
#define BSP_DEVERR_PAGE_ID 1      /* a sparse page id >= num_ids or < 0 */
#define BSP_DEVERR_BLOCK_ID 2     /* a block-table entry >= num_blocks or < 0 */
#define BSP_DEVERR_GROUP_SEQ 4    /* rows of one query group name different sequences */
#define BSP_DEVERR_TIMEOUT 8      /* a bounded wait for a TMA copy gave up */
#define BSP_DEVERR_SLOT 16        /* a slot beyond the cache */

/* top-k flags */
#define BSP_FORCE_TAIL 1 /* the tail page of every row is always selected */
/* decode-step flag: reuse another layer's selection (see bsp_sparse_decode_step) */
#define BSP_REUSE_SELECTION 2
/* top-k flag: 128-token blocks are the unit of selection (see bsp_topk_select) */
#define BSP_SELECT_BLOCKS 4

/* ------------------------------------------------------------------------
 * K/V cache descriptor.
 *
 * bf16 and fp8 caches use the interleaved layout of [vLLM-61889]: a 128-token
 * block holds 16 page slots, slots 0..7 the K pages of its eight 16-token
 * pages, slots 8..15 their V pages.  A page id P = block*16 + j (j < 8)
 * addresses the K page at k_base + P*id_stride_bytes and the V page at
 * v_base + P*id_stride_bytes, with v_base = k_base + 8*id_stride_bytes ("V
 * pages a fixed half-block after").  Inside a page slot the Hkv heads follow
 * each other (page_bytes each: fp8 2048, bf16 4096) and one head's page is
 *   K  [128/x][16 tokens][x],  V  [16/x][128 dims][x],  x = 16 B / element,
 * i.e. the views K [ids, Hkv, 8, 16, 16] and V [ids-8, Hkv, 1, 128, 16] of
 * [vLLM-61889] Validation for fp8.  Valid ids are < num_ids = 16*blocks - 8
 * (the V view's length; the largest id a block table can emit is
 * 16*(blocks-1) + 7).
 *
 * MXFP4 caches ([ATOM-2962] Follow-ups): per block and KV head one 8704 B K
 * field and one V field (128 tokens x 64 B e2m1, even dim in the low nibble,
 * then 128 x 4 B e8m0 scales); per block the Hkv K fields, then the Hkv V
 * fields; id_stride_bytes = bytes per block = 2*Hkv*8704, v_base = k_base +
 * Hkv*8704.  A page id is block*8 + u, u = the 16-token unit of the field;
 * num_ids = 8*blocks.
 *
 * bsp_kv_cache_interleaved() fills the descriptor for a packed cache of
 * `num_blocks` blocks starting at `base`.
 * ---------------------------------------------------------------------- */
typedef struct bsp_kv_cache {
  int32_t dtype;           /* bsp_dtype */
  int32_t num_kv_heads;    /* Hkv >= 1 */
  void* k_base;            /* device */
  void* v_base;            /* device */
  int64_t id_stride_bytes; /* see above */
  int64_t num_ids;         /* page ids must be < num_ids */
  int64_t num_blocks;      /* blocks the cache holds (the writer's slot bound) */
  float k_scale;           /* fp8: dequantised K = e4m3 * k_scale (per tensor) */
  float v_scale;           /* fp8: dequantised V = e4m3 * v_scale */
} bsp_kv_cache;

/* ------------------------------------------------------------------------
 * Index-key cache descriptor.  Per (block, index head) one token-major field:
 *   bf16  128 x 256 B                                         (32768 B)
 *   fp8   128 x 128 B e4m3, then 128 x 4 B fp32 per-token scale (16896 B)
 *   MXFP4 as the K/V fields                                    (8704 B)
 * The field of (block b, head h) is at base + b*block_stride_bytes + h*field.
 * ---------------------------------------------------------------------- */
typedef struct bsp_index_cache {
  int32_t dtype;              /* bsp_dtype */
  int32_t num_heads;          /* index heads */
  void* base;                 /* device */
  int64_t block_stride_bytes; /* >= num_heads * field bytes */
  int64_t num_blocks;
} bsp_index_cache;

bsp_status bsp_kv_cache_interleaved(int32_t dtype, int32_t num_kv_heads, void* base, int64_t num_blocks,
                                    float k_scale, float v_scale, bsp_kv_cache* out);
bsp_status bsp_index_cache_packed(int32_t dtype, int32_t num_heads, void* base, int64_t num_blocks,
                                  bsp_index_cache* out);
/* bytes of one 128-token block of a packed cache */
int64_t bsp_kv_block_bytes(int32_t dtype, int32_t num_kv_heads);
int64_t bsp_index_field_bytes(int32_t dtype);

/* ------------------------------------------------------------------------
 * a1  bsp_kv_page_write -- quantise and scatter new tokens into the pages.
 * [ATOM-2962] commit "... index key" (the fused writer stores K, V and the
 * index key straight onto the pool pages) and PR description (MXFP4 format);
 * [vLLM-61889] Details (per-tensor fp8 scales).  QK-norm and RoPE are model
 * math outside this call: k, v, idx_k are the post-RoPE rows.
 *   k, v        bf16 [T, Hkv, 128]
 *   idx_k       bf16 [T, idx->num_heads, 128], or NULL to skip the index
 *               cache (a layer reusing another layer's top-k)
 *   idx         index cache, or NULL (then idx_k must be NULL)
 *   slot        int64 [T]: block*128 + offset; -1 skips the token
 * Encodings: bf16 stored as is; fp8 K/V byte = e4m3_sat(x / k_scale) with an
 * IEEE fp32 division; MXFP4 per 32-group shared exponent
 * e = clamp(floor(log2(amax)) - 2, -127, 127), byte e+127, nibble =
 * e2m1_rn_sat(x * 2^-e); fp8 index key s = amax/448 (1 if amax = 0) stored as
 * fp32, byte = e4m3_sat(x / s).  Slots beyond the cache set
 * BSP_DEVERR_SLOT and are skipped.
 * ---------------------------------------------------------------------- */
bsp_status bsp_kv_page_write(const bsp_kv_cache* kv, const bsp_index_cache* idx,
                             const void* k, const void* v, const void* idx_k,
                             const int64_t* slot, int32_t num_tokens, int32_t* dev_err, bsp_stream_t stream);

/* The writer's e4m3 query output: out[i] = e4m3_sat(x[i]) with unit scale
 * ([ATOM-2962] commit "... index key": "the unit-scale saturating cast").
 * x bf16 [n], out uint8 [n]. */
bsp_status bsp_cast_e4m3(const void* x, void* out, int64_t n, bsp_stream_t stream);

/* ------------------------------------------------------------------------
 * Row lengths with the pad-row clamp ([ATOM-2962] "Other behaviour changes",
 * B12: "clamps a row's causal length where it enters, so a pad row (length 0,
 * q > 1) computes nothing from a negative length").
 * Decode: token j of sequence s (token index s*q_len + j) sees
 *   L = max(0, seq_lens[s] - (q_len - 1 - j)).
 * Prefill: token i sees L = max(0, query_abs_pos[i] + 1), sequence
 *   query_req_id[i] (an index into the block table the later calls get).
 * Outputs row_seq[rows], row_len[rows], rows = tokens * num_heads.
 * ---------------------------------------------------------------------- */
bsp_status bsp_row_lengths_decode(const int32_t* seq_lens, int32_t num_seqs, int32_t q_len, int32_t num_heads,
                                  int32_t* row_seq, int32_t* row_len, bsp_stream_t stream);
bsp_status bsp_row_lengths_prefill(const int32_t* query_req_id, const int32_t* query_abs_pos, int32_t num_tokens,
                                   int32_t num_heads, int32_t* row_seq, int32_t* row_len, bsp_stream_t stream);

/* ------------------------------------------------------------------------
 * a2  bsp_index_score -- page scores of the index query against the index
 * cache ([ATOM-2962] commit "... page-128 block table" and "Known limits":
 * fp32 scores in a workspace that holds -inf where nothing is scored).
 *   scores[r, p] = max over tokens t of page p with t < L_r of
 *                  sum_d q_{r,d} * k_{t,d}         (fp32; k dequantised)
 *   scores[r, p] = -inf for p >= ceil(L_r / 16),   p < max_pages
 *   idx_q     [tokens, idx->num_heads, 128], bf16 or e4m3 (q_dtype)
 *   block_table int32 [*, bt_stride]: 128-token block ids of each sequence
 *   row_seq, row_len  int32 [rows] (rows = tokens * idx->num_heads)
 *   q_group   1..8: consecutive query tokens that share a sequence (the
 *             decode query length).  The key cache of a sequence is streamed
 *             once per group, not once per row.  Every row of a group must
 *             name the same sequence (else BSP_DEVERR_GROUP_SEQ).
 *   max_pages width of the score rows; L_r is clamped to max_pages*16;
 *             max_pages <= 8 * bt_stride (the table covers every page).
 *   scores    fp32 [rows, max_pages], every element written.
 * Dot products run on tensor cores (mma.sync, fp16/bf16 operands that hold
 * the dequantised values exactly, fp32 accumulation).
 * ---------------------------------------------------------------------- */
bsp_status bsp_index_score(const bsp_index_cache* idx, const void* idx_q, int32_t q_dtype,
                           const int32_t* block_table, int32_t bt_stride,
                           const int32_t* row_seq, const int32_t* row_len, int32_t num_rows,
                           int32_t q_group, int32_t max_pages, float* scores,
                           int32_t* dev_err, bsp_stream_t stream);

/* ------------------------------------------------------------------------
 * a2' bsp_index_score_prefill -- the same scores for prefill chunks, as a
 * dense fp8 contraction on the tcgen05 tensor cores (TMEM accumulator, TMA
 * operand loads; [ATOM-2962] commit "... page-128 block table": the prefill
 * scorer).  Rows of one chunk are consecutive query tokens of one sequence.
 *   cu_tokens int32 [num_chunks+1]: token offsets of the chunks (device)
 *   max_tiles host upper bound on sum_c ceil(tokens_c / 128)
 *   idx->dtype BSP_FP8_E4M3 or BSP_MXFP4 (e2m1 keys read by the tensor core
 *   from 4-bit-unpacking TMA loads, the e8m0 group scales applied to one
 *   accumulator per 32-dim group), q_dtype BSP_FP8_E4M3, one index head
 *   (idx->num_heads == 1); else BSP_ERR_UNSUPPORTED.
 * Other arguments as bsp_index_score (rows = tokens).
 * ---------------------------------------------------------------------- */
bsp_status bsp_index_score_prefill(const bsp_index_cache* idx, const void* idx_q, int32_t q_dtype,
                                   const int32_t* block_table, int32_t bt_stride,
                                   const int32_t* row_seq, const int32_t* row_len, int32_t num_rows,
                                   const int32_t* cu_tokens, int32_t num_chunks, int32_t max_tiles,
                                   int32_t max_pages, float* scores, int32_t* dev_err, bsp_stream_t stream);

/* ------------------------------------------------------------------------
 * a3  bsp_topk_select -- per-row top-k of pages and the emitted sparse block
 * table ([ATOM-2962]: selection, _emit_sparse_block_table_row with
 * pages_per_block 8 or 1, the B12 clamp, "the tail page is always selected";
 * [MSA-API] metadata builder: the page-16 rebase).
 *   n = ceil(L_r/16), k' = min(k_pages, n).  With BSP_FORCE_TAIL the tail
 *   page n-1 is always selected and the other k'-1 are the highest scores of
 *   pages 0..n-2; otherwise the k' highest of 0..n-1.  Equal scores go to the
 *   lower page (-0 and +0 are equal).  Selected pages are emitted ascending.
 *   topk_idx  int32 [rows, k_pages] logical pages, -1 padded
 *   sparse_bt int32 [rows, k_pages] page ids, -1 padded:
 *             kv_dtype bf16/fp8 (interleaved page-16 cache):
 *                 block_table[s][p/8]*16 + p%8
 *             kv_dtype MXFP4 (128-token fields): block_table[s][p/8]*8 + p%8
 *   sparse_ctx int32 [rows]: 16*(selected full pages) + (valid tokens of the
 *             tail page if selected); 0 for L_r = 0.
 * With BSP_SELECT_BLOCKS the unit of selection is the 128-token block
 * ([ATOM-2962] commit "... page-128 block table": one score per 128 tokens,
 * an emit with pages_per_block): a block's score is the largest score of its
 * pages below n; kb' = min(k_pages/8, ceil(n/8)) blocks are selected (with
 * BSP_FORCE_TAIL the tail block always, the rest by score, equal scores to
 * the lower block), and each selected block, ascending, emits its pages below
 * n with the page ids above -- at most 8*kb' entries, -1 padded, sparse_ctx as
 * above.  Needs k_pages >= 8 (else BSP_ERR_INVALID_ARG).
 * k_pages <= 2048, max_pages <= 65536.
 * ---------------------------------------------------------------------- */
bsp_status bsp_topk_select(const float* scores, int32_t num_rows, int32_t max_pages,
                           const int32_t* row_seq, const int32_t* row_len,
                           const int32_t* block_table, int32_t bt_stride, int32_t kv_dtype,
                           int32_t k_pages, int32_t flags,
                           int32_t* topk_idx, int32_t* sparse_bt, int32_t* sparse_ctx, bsp_stream_t stream);

/* ------------------------------------------------------------------------
 * a4  bsp_sparse_pa_decode -- grouped-query attention of each row over the
 * tokens its sparse table selects ([MSA-API] forward: the decode call with
 * sparse_block_table and sparse_context_lens; [vLLM-61889] Details: one page
 * id for K and V; [ATOM-2962]: MXFP4 K/V with an e4m3 query, one row per
 * (token, KV head)).
 *   q        [tokens, Hkv*G, 128]: bf16, or e4m3 (MXFP4 caches need e4m3 or
 *            bf16; fp8 caches need bf16 q)
 *   rows     tokens * Hkv; row r covers q heads (r%Hkv)*G .. +G-1 of token r/Hkv
 *   token m < sparse_ctx[r] of row r is token m%16 of page sparse_bt[r, m/16]
 *   out      bf16 [tokens, Hkv*G, 128] = softmax(sm_scale * q K^T) V; rows
 *            with sparse_ctx 0 get zeros
 * Split-K over pages: a row's pages may be split over several CTAs whose
 * partial results are merged by log-sum-exp -- on chip when the splits form
 * one thread-block cluster (up to 8), else through `ws`, where the last CTA
 * of a row to finish merges the row.  `ws` is a device workspace of at least
 * bsp_sparse_pa_decode_workspace_bytes() (enough for any KV format; 0 when
 * no plan for these sizes needs one, and then `ws` may be NULL).  It holds
 * per-row arrival counters that must be ZERO before the first call (e.g.
 * cudaMemset once after allocation).  Every call leaves them zero again, so
 * a workspace is zeroed once, not per call.  Calls that overlap on the GPU
 * need separate workspaces.
 * ---------------------------------------------------------------------- */
size_t bsp_sparse_pa_decode_workspace_bytes(int32_t num_rows, int32_t k_pages, int32_t group);
/* The number of CTAs (splits) each row of a decode call with these sizes runs
 * on, for KV format kv_dtype on the current device: 1 (one CTA finishes the
 * row), 2..8 (the splits merge on chip in one thread-block cluster) or more
 * (they merge through the workspace).  0 for invalid arguments. */
int32_t bsp_sparse_pa_decode_splits(int32_t kv_dtype, int32_t num_rows, int32_t k_pages);
bsp_status bsp_sparse_pa_decode(const bsp_kv_cache* kv, const void* q, int32_t q_dtype, int32_t num_q_heads,
                                const int32_t* sparse_bt, const int32_t* sparse_ctx, int32_t num_rows,
                                int32_t k_pages, float sm_scale, void* out, void* ws, size_t ws_bytes,
                                int32_t* dev_err, bsp_stream_t stream);

/* ------------------------------------------------------------------------
 * bsp_sparse_pa_decode_noalloc -- the same computation as bsp_sparse_pa_decode
 * for callers that cannot allocate device memory, and so cannot provide the
 * split-K workspace: code embedded in a host application that plans and
 * reserves all device memory up front and forbids allocation afterwards, or
 * a caller reaching this ABI from a runtime with no device allocator at hand.
 * The pages have no counterpart to this call; it exists only for such
 * callers.
 *  - The workspace is a scratch array inside the library, a file-scope
 *    __device__ array of 16 MiB that every GPU loading the library holds
 *    until the process exits.  A call whose split-K plan for this KV format
 *    needs more returns BSP_ERR_WORKSPACE and enqueues nothing (the plan
 *    uses a workspace only for fewer rows than SMs / 8 with more than 8
 *    splits a row, at most 64 splits of 8320 B: about 10 MB on 152 SMs).
 *  - The first call on a device looks up the array's address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.  The address is cached per device and does
 *    not survive cudaDeviceReset: after a reset, do not call this again in
 *    the same process.
 *  - Calls share the array and it keeps the last call's contents.  When the
 *    plan uses the workspace, a call first clears the part that must start at
 *    zero (the split-K arrival counters, an async memset on `stream`); a
 *    plan that merges on chip touches the array not at all.  Calls that
 *    overlap on the GPU (other streams, other host threads) race on it and
 *    must be serialised by the caller.
 *  - It calls no allocator (no cudaMalloc / cudaFree).  Arguments and errors
 *    are those of bsp_sparse_pa_decode.
 * ---------------------------------------------------------------------- */
bsp_status bsp_sparse_pa_decode_noalloc(const bsp_kv_cache* kv, const void* q, int32_t q_dtype, int32_t num_q_heads,
                                        const int32_t* sparse_bt, const int32_t* sparse_ctx, int32_t num_rows,
                                        int32_t k_pages, float sm_scale, void* out, int32_t* dev_err,
                                        bsp_stream_t stream);

/* ------------------------------------------------------------------------
 * a5  bsp_sparse_pa_prefill -- the same attention for prefill rows, one row
 * per (prefill token, KV head), each with its own sparse table and a context
 * length from its absolute position ([MSA-API] forward: the prefill call with
 * query_req_id, query_abs_pos, sparse_bt, sparse_ctx; [ATOM-2962] commit "...
 * ATOM_M3_INDEX_Q_FP8": prefill is plan-free, one task and one direct write
 * per row).  No workspace: each row is finished by one CTA.
 * ---------------------------------------------------------------------- */
bsp_status bsp_sparse_pa_prefill(const bsp_kv_cache* kv, const void* q, int32_t q_dtype, int32_t num_q_heads,
                                 const int32_t* sparse_bt, const int32_t* sparse_ctx, int32_t num_rows,
                                 int32_t k_pages, float sm_scale, void* out, int32_t* dev_err, bsp_stream_t stream);

/* ------------------------------------------------------------------------
 * The whole decode step as one call: write the step's new tokens, cast the
 * queries the writer emits as e4m3, compute the row lengths, score, select
 * and attend.  Buffers are caller-owned.  Pointers are device pointers; the
 * step's inputs (k_new, v_new, idx_k_new, slot, q, idx_q, seq_lens) and `out`
 * may instead point into pinned host memory (cudaHostAlloc / page-locked,
 * which unified addressing maps into the device's address space): the
 * kernels then load and store them in place, with no copy.
 * `events` (nullable) receives 5 cudaEventRecord calls on `stream`: before
 * the write, before scoring, before the selection, before the attention, and
 * at the end.
 *
 * With BSP_REUSE_SELECTION in `flags` the step attends with the sparse_bt /
 * sparse_ctx already in the arguments -- the selection of another layer
 * that shares this layer's tokens (ROCm/ATOM PR 2962: layers without an
 * indexer reuse a previous layer's top-k) -- and skips the index-key write,
 * the row lengths, the scoring and the selection.  idx, idx_k_new, idx_q,
 * idx_q_cast, row_seq, row_len, scores and topk_idx are then unused (NULL is
 * fine); the three middle events mark the same point.
 * ---------------------------------------------------------------------- */
typedef struct bsp_decode_step_args {
  const bsp_kv_cache* kv;
  const bsp_index_cache* idx;   /* idx->num_heads == kv->num_kv_heads */
  /* new tokens: k, v bf16 [T, Hkv, 128], idx_k bf16 [T, Hidx, 128], slot [T] */
  const void* k_new;
  const void* v_new;
  const void* idx_k_new;
  const int64_t* slot;
  int32_t num_new_tokens;
  /* queries of the step (num_seqs * q_len tokens), bf16 as the model emits them */
  const void* q;              /* bf16 [tokens, Hkv*G, 128] */
  int32_t q_dtype;            /* BSP_BF16: attend with q; BSP_FP8_E4M3: cast into q_cast first */
  void* q_cast;               /* uint8 [tokens, Hkv*G, 128] when q_dtype is e4m3, else unused */
  int32_t num_q_heads;
  const void* idx_q;          /* bf16 [tokens, Hidx, 128] */
  int32_t idx_q_dtype;        /* as q_dtype, with idx_q_cast */
  void* idx_q_cast;
  const int32_t* seq_lens;    /* [num_seqs], including the new tokens */
  int32_t num_seqs;
  int32_t q_len;              /* 1..8 */
  const int32_t* block_table; /* [num_seqs, bt_stride] */
  int32_t bt_stride;
  int32_t max_pages;
  int32_t k_pages;
  int32_t flags;              /* BSP_FORCE_TAIL, BSP_REUSE_SELECTION, BSP_SELECT_BLOCKS */
  float sm_scale;
  /* outputs and scratch (caller-owned device memory) */
  int32_t* row_seq;           /* [rows] */
  int32_t* row_len;           /* [rows] */
  float* scores;              /* [rows, max_pages] */
  int32_t* topk_idx;          /* [rows, k_pages] */
  int32_t* sparse_bt;         /* [rows, k_pages] */
  int32_t* sparse_ctx;        /* [rows] */
  void* out;                  /* bf16 [tokens, Hkv*G, 128] */
  void* ws;                   /* bsp_sparse_pa_decode_workspace_bytes(rows, k_pages, G) */
  size_t ws_bytes;
  int32_t* dev_err;
  /* optional (NULL: a separate selector launch): int32 [num_seqs * Hidx],
   * zeroed once by the caller and left zero by every step.  The scorer's
   * last CTA of each (sequence, index head) then selects that sequence's
   * rows itself, one launch fewer -- the same outputs bit for bit, but
   * every scorer CTA then waits for a counter round trip before it retires
   * and one CTA selects all of a sequence's rows, so on large batches the
   * step is slower.  Used for fp8 index caches with e4m3 index queries,
   * max_pages <= 4096 and page-granular selection; otherwise ignored. */
  int32_t* sel_counters;
} bsp_decode_step_args;

bsp_status bsp_sparse_decode_step(const bsp_decode_step_args* a, bsp_event_t* events, bsp_stream_t stream);

/* ---- misc -------------------------------------------------------------- */
const char* bsp_status_str(bsp_status s);
/* the last CUDA error a call saw (cudaError_t as int), 0 if none */
int32_t bsp_last_cuda_error(void);
/* number of kernels this library has launched in this process */
int64_t bsp_launch_count(void);
/* library version, e.g. 100 for 1.0.0 */
int32_t bsp_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BSP_H */
