// api.cu -- the C ABI of libbsp (declared in include/bsp.h): argument
// validation on the host, the split plans, and the kernel launches.  Nothing
// here allocates, synchronises or reads device memory.
#include <algorithm>
#include <atomic>
#include <cstdint>

#include "../../include/bsp.h"
#include "common.cuh"
#include "kernels.h"

using namespace bsp;

namespace {

std::atomic<int32_t> g_last_cuda_error{0};
std::atomic<int64_t> g_launches{0};

std::atomic<int> g_sms[kMaxDevices];

int device_sms() {
  return cached_per_device(g_sms, [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || n <= 0)
      n = 148;
    return n;
  });
}

bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool valid_dtype(int32_t d) { return d == BSP_BF16 || d == BSP_FP8_E4M3 || d == BSP_MXFP4; }
bool valid_group(int32_t g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

bsp_status cuda_status(cudaError_t e) {
  if (e != cudaSuccess) {
    g_last_cuda_error.store(static_cast<int32_t>(e));
    return BSP_ERR_CUDA;
  }
  return BSP_OK;
}

int64_t index_field(int32_t dtype) {
  return dtype == BSP_BF16 ? kBf16IndexField : (dtype == BSP_FP8_E4M3 ? kFp8IndexField : kMxField);
}

bsp_status check_kv(const bsp_kv_cache* kv) {
  if (!kv || !valid_dtype(kv->dtype) || kv->num_kv_heads < 1 || !kv->k_base || !kv->v_base) return BSP_ERR_INVALID_ARG;
  if (!al(kv->k_base, 16) || !al(kv->v_base, 16) || kv->id_stride_bytes <= 0 || kv->id_stride_bytes % 16)
    return BSP_ERR_INVALID_ARG;
  const int64_t page = kv->dtype == BSP_BF16 ? 4096 : 2048;
  if (kv->dtype == BSP_MXFP4 ? kv->id_stride_bytes < 2LL * kv->num_kv_heads * kMxField
                             : kv->id_stride_bytes < kv->num_kv_heads * page)
    return BSP_ERR_INVALID_ARG;
  if (kv->num_ids < 0 || kv->num_blocks < 0) return BSP_ERR_INVALID_ARG;
  return BSP_OK;
}

bsp_status check_idx(const bsp_index_cache* idx) {
  if (!idx || !valid_dtype(idx->dtype) || idx->num_heads < 1 || !idx->base || !al(idx->base, 16))
    return BSP_ERR_INVALID_ARG;
  if (idx->block_stride_bytes < idx->num_heads * index_field(idx->dtype) || idx->block_stride_bytes % 16 ||
      idx->num_blocks < 0)
    return BSP_ERR_INVALID_ARG;
  return BSP_OK;
}

}  // namespace

extern "C" {

int64_t bsp_kv_block_bytes(int32_t dtype, int32_t num_kv_heads) {
  if (!valid_dtype(dtype) || num_kv_heads < 1) return -1;
  if (dtype == BSP_MXFP4) return 2LL * num_kv_heads * kMxField;
  return 16LL * num_kv_heads * (dtype == BSP_BF16 ? 4096 : 2048);
}

int64_t bsp_index_field_bytes(int32_t dtype) { return valid_dtype(dtype) ? index_field(dtype) : -1; }

bsp_status bsp_kv_cache_interleaved(int32_t dtype, int32_t num_kv_heads, void* base, int64_t num_blocks,
                                    float k_scale, float v_scale, bsp_kv_cache* out) {
  if (!out || !valid_dtype(dtype) || num_kv_heads < 1 || !base || !al(base, 16) || num_blocks < 1)
    return BSP_ERR_INVALID_ARG;
  out->dtype = dtype;
  out->num_kv_heads = num_kv_heads;
  out->k_base = base;
  out->num_blocks = num_blocks;
  out->k_scale = k_scale;
  out->v_scale = v_scale;
  if (dtype == BSP_MXFP4) {
    out->id_stride_bytes = 2LL * num_kv_heads * kMxField;
    out->v_base = static_cast<uint8_t*>(base) + static_cast<int64_t>(num_kv_heads) * kMxField;
    out->num_ids = 8 * num_blocks;
  } else {
    out->id_stride_bytes = static_cast<int64_t>(num_kv_heads) * (dtype == BSP_BF16 ? 4096 : 2048);
    out->v_base = static_cast<uint8_t*>(base) + 8 * out->id_stride_bytes;
    out->num_ids = 16 * num_blocks - 8;
  }
  return BSP_OK;
}

bsp_status bsp_index_cache_packed(int32_t dtype, int32_t num_heads, void* base, int64_t num_blocks,
                                  bsp_index_cache* out) {
  if (!out || !valid_dtype(dtype) || num_heads < 1 || !base || !al(base, 16) || num_blocks < 1)
    return BSP_ERR_INVALID_ARG;
  out->dtype = dtype;
  out->num_heads = num_heads;
  out->base = base;
  out->block_stride_bytes = num_heads * index_field(dtype);
  out->num_blocks = num_blocks;
  return BSP_OK;
}

bsp_status bsp_kv_page_write(const bsp_kv_cache* kv, const bsp_index_cache* idx, const void* k, const void* v,
                             const void* idx_k, const int64_t* slot, int32_t num_tokens, int32_t* dev_err,
                             bsp_stream_t stream) {
  bsp_status st = check_kv(kv);
  if (st != BSP_OK) return st;
  if (num_tokens < 0) return BSP_ERR_INVALID_ARG;
  if (num_tokens == 0) return BSP_OK;
  if (!k || !v || !slot || !al(k, 16) || !al(v, 16) || !al(slot, 8)) return BSP_ERR_INVALID_ARG;
  if (idx_k && !idx) return BSP_ERR_INVALID_ARG;
  if (idx_k) {
    if ((st = check_idx(idx)) != BSP_OK) return st;
    if (!al(idx_k, 16)) return BSP_ERR_INVALID_ARG;
  }
  KvWriteParams p{};
  p.kv_dtype = kv->dtype;
  p.hkv = kv->num_kv_heads;
  p.k_base = static_cast<uint8_t*>(kv->k_base);
  p.v_base = static_cast<uint8_t*>(kv->v_base);
  p.id_stride = kv->id_stride_bytes;
  p.num_blocks = kv->num_blocks;
  p.k_scale = kv->k_scale;
  p.v_scale = kv->v_scale;
  if (idx_k) {
    p.idx_dtype = idx->dtype;
    p.hidx = idx->num_heads;
    p.idx_base = static_cast<uint8_t*>(idx->base);
    p.idx_block_stride = idx->block_stride_bytes;
    p.idx_num_blocks = idx->num_blocks;
  }
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.idx_k = static_cast<const uint16_t*>(idx_k);
  p.slot = slot;
  p.num_tokens = num_tokens;
  p.err = dev_err;
  st = cuda_status(launch_kv_page_write(p, reinterpret_cast<cudaStream_t>(stream)));
  if (st == BSP_OK) ++g_launches;
  return st;
}

bsp_status bsp_cast_e4m3(const void* x, void* out, int64_t n, bsp_stream_t stream) {
  if (n < 0) return BSP_ERR_INVALID_ARG;
  if (n == 0) return BSP_OK;
  if (!x || !out || !al(x, 16) || !al(out, 8)) return BSP_ERR_INVALID_ARG;
  bsp_status st = cuda_status(launch_cast_e4m3(static_cast<const uint16_t*>(x), static_cast<uint8_t*>(out), n,
                                               reinterpret_cast<cudaStream_t>(stream)));
  if (st == BSP_OK) ++g_launches;
  return st;
}

bsp_status bsp_row_lengths_decode(const int32_t* seq_lens, int32_t num_seqs, int32_t q_len, int32_t num_heads,
                                  int32_t* row_seq, int32_t* row_len, bsp_stream_t stream) {
  if (num_seqs < 0 || q_len < 1 || num_heads < 1) return BSP_ERR_INVALID_ARG;
  if (num_seqs == 0) return BSP_OK;
  if (!seq_lens || !row_seq || !row_len) return BSP_ERR_INVALID_ARG;
  bsp_status st = cuda_status(launch_row_lengths_decode(seq_lens, num_seqs, q_len, num_heads, row_seq, row_len,
                                                        reinterpret_cast<cudaStream_t>(stream)));
  if (st == BSP_OK) ++g_launches;
  return st;
}

bsp_status bsp_row_lengths_prefill(const int32_t* query_req_id, const int32_t* query_abs_pos, int32_t num_tokens,
                                   int32_t num_heads, int32_t* row_seq, int32_t* row_len, bsp_stream_t stream) {
  if (num_tokens < 0 || num_heads < 1) return BSP_ERR_INVALID_ARG;
  if (num_tokens == 0) return BSP_OK;
  if (!query_req_id || !query_abs_pos || !row_seq || !row_len) return BSP_ERR_INVALID_ARG;
  bsp_status st = cuda_status(launch_row_lengths_prefill(query_req_id, query_abs_pos, num_tokens, num_heads, row_seq,
                                                         row_len, reinterpret_cast<cudaStream_t>(stream)));
  if (st == BSP_OK) ++g_launches;
  return st;
}

// the decode scorer's argument checks (also run by the decode step before its
// first launch)
static bsp_status index_score_check(const bsp_index_cache* idx, const void* idx_q, int32_t q_dtype,
                                    const int32_t* block_table, int32_t bt_stride, const int32_t* row_seq,
                                    const int32_t* row_len, int32_t num_rows, int32_t q_group, int32_t max_pages,
                                    const float* scores) {
  bsp_status st = check_idx(idx);
  if (st != BSP_OK) return st;
  if (num_rows < 0 || max_pages < 1 || bt_stride < 1) return BSP_ERR_INVALID_ARG;
  if (q_dtype != BSP_BF16 && q_dtype != BSP_FP8_E4M3) return BSP_ERR_UNSUPPORTED;
  if (q_group < 1 || q_group > 8) return BSP_ERR_UNSUPPORTED;
  if (num_rows % idx->num_heads) return BSP_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_pages) > static_cast<int64_t>(bt_stride) * 8) return BSP_ERR_INVALID_ARG;
  if (num_rows == 0) return BSP_OK;
  if (!idx_q || !block_table || !row_seq || !row_len || !scores || !al(idx_q, 8)) return BSP_ERR_INVALID_ARG;
  return BSP_OK;
}

// seq_is_group: the decode step's own rows, where query group g is sequence g
static bsp_status index_score_impl(const bsp_index_cache* idx, const void* idx_q, int32_t q_dtype,
                                   const int32_t* block_table, int32_t bt_stride, const int32_t* row_seq,
                                   const int32_t* row_len, int32_t num_rows, int32_t q_group, int32_t max_pages,
                                   float* scores, int32_t* dev_err, bsp_stream_t stream, int32_t seq_is_group,
                                   const TopkParams* sel = nullptr, int32_t* sel_counters = nullptr) {
  bsp_status st = index_score_check(idx, idx_q, q_dtype, block_table, bt_stride, row_seq, row_len, num_rows,
                                    q_group, max_pages, scores);
  if (st != BSP_OK || num_rows == 0) return st;
  IndexScoreParams p{};
  p.idx_dtype = idx->dtype;
  p.hidx = idx->num_heads;
  p.idx_base = static_cast<const uint8_t*>(idx->base);
  p.block_stride = idx->block_stride_bytes;
  p.num_blocks = idx->num_blocks;
  p.q = idx_q;
  p.q_dtype = q_dtype;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.row_seq = row_seq;
  p.row_len = row_len;
  p.num_rows = num_rows;
  p.num_tokens = num_rows / idx->num_heads;
  p.q_group = q_group;
  p.max_pages = max_pages;
  p.scores = scores;
  p.err = dev_err;
  p.seq_is_group = seq_is_group;
  if (sel) {
    p.sel = *sel;
    p.sel_counters = sel_counters;
  }
  st = cuda_status(launch_index_score(p, device_sms(), reinterpret_cast<cudaStream_t>(stream)));
  if (st == BSP_OK) ++g_launches;
  return st;
}

bsp_status bsp_index_score(const bsp_index_cache* idx, const void* idx_q, int32_t q_dtype,
                           const int32_t* block_table, int32_t bt_stride, const int32_t* row_seq,
                           const int32_t* row_len, int32_t num_rows, int32_t q_group, int32_t max_pages,
                           float* scores, int32_t* dev_err, bsp_stream_t stream) {
  return index_score_impl(idx, idx_q, q_dtype, block_table, bt_stride, row_seq, row_len, num_rows, q_group,
                          max_pages, scores, dev_err, stream, 0);
}

bsp_status bsp_index_score_prefill(const bsp_index_cache* idx, const void* idx_q, int32_t q_dtype,
                                   const int32_t* block_table, int32_t bt_stride, const int32_t* row_seq,
                                   const int32_t* row_len, int32_t num_rows, const int32_t* cu_tokens,
                                   int32_t num_chunks, int32_t max_tiles, int32_t max_pages, float* scores,
                                   int32_t* dev_err, bsp_stream_t stream) {
  bsp_status st = check_idx(idx);
  if (st != BSP_OK) return st;
  const bool mx = idx->dtype == BSP_MXFP4;
  if ((idx->dtype != BSP_FP8_E4M3 && !mx) || q_dtype != BSP_FP8_E4M3 || idx->num_heads != 1)
    return BSP_ERR_UNSUPPORTED;
  if (idx->block_stride_bytes % (mx ? 64 : 128)) return BSP_ERR_UNSUPPORTED;
  if (num_rows < 0 || max_pages < 1 || bt_stride < 1 || num_chunks < 0 || max_tiles < 0) return BSP_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_pages) > static_cast<int64_t>(bt_stride) * 8) return BSP_ERR_INVALID_ARG;
  if (num_rows == 0 || num_chunks == 0 || max_tiles == 0) return BSP_OK;
  if (!idx_q || !block_table || !row_seq || !row_len || !scores || !cu_tokens || !al(idx_q, 16))
    return BSP_ERR_INVALID_ARG;
  PrefillScoreParams p{};
  p.idx_base = static_cast<const uint8_t*>(idx->base);
  p.block_stride = idx->block_stride_bytes;
  p.num_blocks = idx->num_blocks;
  p.q = static_cast<const uint8_t*>(idx_q);
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.row_seq = row_seq;
  p.row_len = row_len;
  p.num_rows = num_rows;
  p.cu_tokens = cu_tokens;
  p.num_chunks = num_chunks;
  p.max_tiles = max_tiles;
  p.max_pages = max_pages;
  p.scores = scores;
  p.err = dev_err;
  cudaError_t e = mx ? launch_index_score_prefill_mx(p, reinterpret_cast<cudaStream_t>(stream))
                     : launch_index_score_prefill(p, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return BSP_ERR_UNSUPPORTED;
  st = cuda_status(e);
  if (st == BSP_OK) ++g_launches;
  return st;
}

// The selector's parameters, checked.  rows_per_seq > 0: row r belongs to
// sequence r / rows_per_seq (the decode step's own rows).
static bsp_status topk_params(const float* scores, int32_t num_rows, int32_t max_pages, const int32_t* row_seq,
                              const int32_t* row_len, const int32_t* block_table, int32_t bt_stride, int32_t kv_dtype,
                              int32_t k_pages, int32_t flags, int32_t* topk_idx, int32_t* sparse_bt,
                              int32_t* sparse_ctx, int32_t rows_per_seq, TopkParams& p) {
  if (num_rows < 0 || max_pages < 1 || bt_stride < 1 || k_pages < 1 || !valid_dtype(kv_dtype))
    return BSP_ERR_INVALID_ARG;
  if (k_pages > 2048 || max_pages > 65536) return BSP_ERR_UNSUPPORTED;
  if ((flags & BSP_SELECT_BLOCKS) && k_pages < kPagesPerSide) return BSP_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_pages) > static_cast<int64_t>(bt_stride) * 8) return BSP_ERR_INVALID_ARG;
  if (num_rows > 0 &&
      (!scores || !row_seq || !row_len || !block_table || !topk_idx || !sparse_bt || !sparse_ctx || !al(scores, 16)))
    return BSP_ERR_INVALID_ARG;
  p = TopkParams{};
  p.scores = scores;
  p.num_rows = num_rows;
  p.max_pages = max_pages;
  p.row_seq = row_seq;
  p.row_len = row_len;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.id_mul = kv_dtype == BSP_MXFP4 ? 8 : 16;
  p.k_pages = k_pages;
  p.force_tail = (flags & BSP_FORCE_TAIL) ? 1 : 0;
  p.topk_idx = topk_idx;
  p.sparse_bt = sparse_bt;
  p.sparse_ctx = sparse_ctx;
  p.rows_per_seq = rows_per_seq;
  p.blocks = (flags & BSP_SELECT_BLOCKS) ? 1 : 0;
  return BSP_OK;
}

static bsp_status topk_impl(const float* scores, int32_t num_rows, int32_t max_pages, const int32_t* row_seq,
                            const int32_t* row_len, const int32_t* block_table, int32_t bt_stride, int32_t kv_dtype,
                            int32_t k_pages, int32_t flags, int32_t* topk_idx, int32_t* sparse_bt,
                            int32_t* sparse_ctx, bsp_stream_t stream, int32_t rows_per_seq) {
  TopkParams p;
  bsp_status st = topk_params(scores, num_rows, max_pages, row_seq, row_len, block_table, bt_stride, kv_dtype, k_pages,
                              flags, topk_idx, sparse_bt, sparse_ctx, rows_per_seq, p);
  if (st != BSP_OK || num_rows == 0) return st;
  st = cuda_status(launch_topk_select(p, reinterpret_cast<cudaStream_t>(stream)));
  if (st == BSP_OK) ++g_launches;
  return st;
}

bsp_status bsp_topk_select(const float* scores, int32_t num_rows, int32_t max_pages, const int32_t* row_seq,
                           const int32_t* row_len, const int32_t* block_table, int32_t bt_stride, int32_t kv_dtype,
                           int32_t k_pages, int32_t flags, int32_t* topk_idx, int32_t* sparse_bt, int32_t* sparse_ctx,
                           bsp_stream_t stream) {
  return topk_impl(scores, num_rows, max_pages, row_seq, row_len, block_table, bt_stride, kv_dtype, k_pages, flags,
                   topk_idx, sparse_bt, sparse_ctx, stream, 0);
}

size_t bsp_sparse_pa_decode_workspace_bytes(int32_t num_rows, int32_t k_pages, int32_t group) {
  (void)group;
  if (num_rows <= 0 || k_pages <= 0) return 0;
  // the largest of the three KV formats' plans (the query has no format)
  size_t need = 0;
  for (int32_t kv : {BSP_BF16, BSP_FP8_E4M3, BSP_MXFP4})
    need = std::max(need, sparse_pa_ws_bytes(num_rows, sparse_pa_plan(kv, num_rows, k_pages, device_sms())));
  return need;
}

int32_t bsp_sparse_pa_decode_splits(int32_t kv_dtype, int32_t num_rows, int32_t k_pages) {
  if (!valid_dtype(kv_dtype) || num_rows < 1 || k_pages < 1) return 0;
  return sparse_pa_plan(kv_dtype, num_rows, k_pages, device_sms()).nsplit;
}

}  // extern "C"

namespace bsp {

bsp_status sparse_pa_check_args(const bsp_kv_cache* kv, const void* q, int32_t q_dtype, int32_t num_q_heads,
                                const int32_t* sparse_bt, const int32_t* sparse_ctx, int32_t num_rows,
                                int32_t k_pages, const void* out) {
  bsp_status st = check_kv(kv);
  if (st != BSP_OK) return st;
  if (num_rows < 0 || k_pages < 1 || num_q_heads < 1) return BSP_ERR_INVALID_ARG;
  if (num_q_heads % kv->num_kv_heads || num_rows % kv->num_kv_heads) return BSP_ERR_INVALID_ARG;
  if (!valid_group(num_q_heads / kv->num_kv_heads)) return BSP_ERR_UNSUPPORTED;
  if (q_dtype != BSP_BF16 && q_dtype != BSP_FP8_E4M3) return BSP_ERR_UNSUPPORTED;
  if (num_rows == 0) return BSP_OK;
  if (!q || !sparse_bt || !sparse_ctx || !out || !al(out, 16) || !al(q, 16)) return BSP_ERR_INVALID_ARG;
  return BSP_OK;
}

size_t sparse_pa_decode_ws_need(int32_t kv_dtype, int32_t num_rows, int32_t k_pages) {
  if (num_rows <= 0 || k_pages <= 0) return 0;
  return sparse_pa_ws_bytes(num_rows, sparse_pa_plan(kv_dtype, num_rows, k_pages, device_sms()));
}

}  // namespace bsp

extern "C" {

static bsp_status sparse_pa_common(const bsp_kv_cache* kv, const void* q, int32_t q_dtype, int32_t num_q_heads,
                                   const int32_t* sparse_bt, const int32_t* sparse_ctx, int32_t num_rows,
                                   int32_t k_pages, float sm_scale, void* out, void* ws, size_t ws_bytes,
                                   int32_t* dev_err, bsp_stream_t stream, bool decode, bool q_early = false) {
  bsp_status st = sparse_pa_check_args(kv, q, q_dtype, num_q_heads, sparse_bt, sparse_ctx, num_rows, k_pages, out);
  if (st != BSP_OK || num_rows == 0) return st;
  const int32_t group = num_q_heads / kv->num_kv_heads;
  SparsePaParams p{};
  p.kv_dtype = kv->dtype;
  p.hkv = kv->num_kv_heads;
  p.k_base = static_cast<const uint8_t*>(kv->k_base);
  p.v_base = static_cast<const uint8_t*>(kv->v_base);
  p.id_stride = kv->id_stride_bytes;
  p.num_ids = kv->num_ids;
  p.k_scale = kv->k_scale;
  p.v_scale = kv->v_scale;
  p.q = q;
  p.q_dtype = q_dtype;
  p.group = group;
  p.sparse_bt = sparse_bt;
  p.sparse_ctx = sparse_ctx;
  p.num_rows = num_rows;
  p.k_pages = k_pages;
  p.sm_scale = sm_scale;
  p.out = out;
  p.err = dev_err;
  p.q_early = q_early;
  if (decode) {
    const PaPlan plan = sparse_pa_plan(kv->dtype, num_rows, k_pages, device_sms());
    p.nsplit = plan.nsplit;
    p.pages_per_split = plan.pages_per_split;
    p.cluster = plan.cluster;
    p.ring = plan.ring;
    const size_t need = sparse_pa_ws_bytes(num_rows, plan);
    if (need) {
      if (!ws || ws_bytes < need || !al(ws, 16)) return BSP_ERR_WORKSPACE;
      p.ws = static_cast<float*>(ws);
    }
  } else {
    const PaPlan plan = sparse_pa_prefill_plan(kv->dtype, k_pages);
    p.nsplit = plan.nsplit;
    p.pages_per_split = plan.pages_per_split;
    p.ring = plan.ring;
  }
  int launches = 0;
  st = cuda_status(launch_sparse_pa(p, reinterpret_cast<cudaStream_t>(stream), &launches));
  g_launches += launches;
  return st;
}

// the decode attention's workspace check (also run by the decode step before
// its first launch): a plan that merges through the workspace needs `need`
// bytes of it, 16-byte aligned
static bsp_status sparse_pa_ws_check(int32_t kv_dtype, int32_t num_rows, int32_t k_pages, const void* ws,
                                     size_t ws_bytes) {
  const size_t need = sparse_pa_decode_ws_need(kv_dtype, num_rows, k_pages);
  return need && (!ws || ws_bytes < need || !al(ws, 16)) ? BSP_ERR_WORKSPACE : BSP_OK;
}

bsp_status bsp_sparse_pa_decode(const bsp_kv_cache* kv, const void* q, int32_t q_dtype, int32_t num_q_heads,
                                const int32_t* sparse_bt, const int32_t* sparse_ctx, int32_t num_rows,
                                int32_t k_pages, float sm_scale, void* out, void* ws, size_t ws_bytes,
                                int32_t* dev_err, bsp_stream_t stream) {
  return sparse_pa_common(kv, q, q_dtype, num_q_heads, sparse_bt, sparse_ctx, num_rows, k_pages, sm_scale, out, ws,
                          ws_bytes, dev_err, stream, true);
}

bsp_status bsp_sparse_pa_prefill(const bsp_kv_cache* kv, const void* q, int32_t q_dtype, int32_t num_q_heads,
                                 const int32_t* sparse_bt, const int32_t* sparse_ctx, int32_t num_rows,
                                 int32_t k_pages, float sm_scale, void* out, int32_t* dev_err, bsp_stream_t stream) {
  return sparse_pa_common(kv, q, q_dtype, num_q_heads, sparse_bt, sparse_ctx, num_rows, k_pages, sm_scale, out,
                          nullptr, 0, dev_err, stream, false);
}

bsp_status bsp_sparse_decode_step(const bsp_decode_step_args* a, bsp_event_t* events, bsp_stream_t stream) {
  if (!a || !a->kv) return BSP_ERR_INVALID_ARG;
  const bool reuse = (a->flags & BSP_REUSE_SELECTION) != 0;
  if (!reuse && !a->idx) return BSP_ERR_INVALID_ARG;
  const int32_t hkv = a->kv->num_kv_heads;
  const int32_t hidx = reuse ? 0 : a->idx->num_heads;
  if (!reuse && hidx != hkv) return BSP_ERR_UNSUPPORTED;  // rows are shared by the scorer and the attention
  if (a->num_seqs < 0 || a->q_len < 1 || a->q_len > 8) return BSP_ERR_INVALID_ARG;
  if (static_cast<int64_t>(a->num_seqs) * a->q_len * hkv > INT32_MAX) return BSP_ERR_UNSUPPORTED;  // int32 rows
  const int32_t tokens = a->num_seqs * a->q_len;
  const int32_t rows = tokens * hkv;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto mark = [&](int i) {
    if (events) cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), s);
  };
  bsp_status st = check_kv(a->kv);
  if (st != BSP_OK) return st;
  if (!reuse && (st = check_idx(a->idx)) != BSP_OK) return st;
  if (a->num_new_tokens < 0 || a->num_q_heads < 1) return BSP_ERR_INVALID_ARG;
  if (a->num_new_tokens && (!a->k_new || !a->v_new || !a->slot || !al(a->k_new, 16) || !al(a->v_new, 16) ||
                            !al(a->slot, 8) || (!reuse && (!a->idx_k_new || !al(a->idx_k_new, 16)))))
    return BSP_ERR_INVALID_ARG;
  if (!a->q || !al(a->q, 16)) return BSP_ERR_INVALID_ARG;
  if (reuse ? (!a->sparse_bt || !a->sparse_ctx)
            : (!a->idx_q || !al(a->idx_q, 16) || !a->seq_lens || !a->row_seq || !a->row_len))
    return BSP_ERR_INVALID_ARG;
  const bool cast_q = a->q_dtype == BSP_FP8_E4M3, cast_iq = !reuse && a->idx_q_dtype == BSP_FP8_E4M3;
  if ((cast_q && (!a->q_cast || !al(a->q_cast, 16))) || (cast_iq && (!a->idx_q_cast || !al(a->idx_q_cast, 16))))
    return BSP_ERR_INVALID_ARG;
  // the queries the scorer and the attention read
  const void* q = cast_q ? a->q_cast : a->q;
  const void* iq = cast_iq ? a->idx_q_cast : a->idx_q;
  // The step's rows are decode-ordered (row_seq = token / q_len, as the prep
  // kernel writes it): the scorer and the selector find a row's sequence
  // without reading row_seq first.  With sel_counters the scorer's last CTA
  // of each query group selects the group's rows (no selector launch).
  const int32_t topk_flags = a->flags & (BSP_FORCE_TAIL | BSP_SELECT_BLOCKS);
  const bool fused = !reuse && a->sel_counters &&
                     index_score_can_select(a->idx->dtype, a->idx_q_dtype, a->max_pages,
                                            (a->flags & BSP_SELECT_BLOCKS) != 0);
  // every later stage's checks too, so that an invalid step enqueues nothing
  TopkParams sel;
  if (!reuse) {
    if (fused && !al(a->sel_counters, 4)) return BSP_ERR_INVALID_ARG;
    if ((st = index_score_check(a->idx, iq, a->idx_q_dtype, a->block_table, a->bt_stride, a->row_seq, a->row_len,
                                rows, a->q_len, a->max_pages, a->scores)) != BSP_OK ||
        (st = topk_params(a->scores, rows, a->max_pages, a->row_seq, a->row_len, a->block_table, a->bt_stride,
                          a->kv->dtype, a->k_pages, topk_flags, a->topk_idx, a->sparse_bt, a->sparse_ctx,
                          a->q_len * hkv, sel)) != BSP_OK)
      return st;
  }
  if ((st = sparse_pa_check_args(a->kv, q, a->q_dtype, a->num_q_heads, a->sparse_bt, a->sparse_ctx, rows, a->k_pages,
                                 a->out)) != BSP_OK ||
      (st = sparse_pa_ws_check(a->kv->dtype, rows, a->k_pages, a->ws, a->ws_bytes)) != BSP_OK)
    return st;
  mark(0);
  // write + e4m3 casts + row lengths: one launch
  DecodePrepParams pp{};
  KvWriteParams& w = pp.write;
  w.kv_dtype = a->kv->dtype;
  w.hkv = hkv;
  w.k_base = static_cast<uint8_t*>(a->kv->k_base);
  w.v_base = static_cast<uint8_t*>(a->kv->v_base);
  w.id_stride = a->kv->id_stride_bytes;
  w.num_blocks = a->kv->num_blocks;
  w.k_scale = a->kv->k_scale;
  w.v_scale = a->kv->v_scale;
  w.hidx = hidx;  // 0: no index-key write
  if (!reuse) {
    w.idx_dtype = a->idx->dtype;
    w.idx_base = static_cast<uint8_t*>(a->idx->base);
    w.idx_block_stride = a->idx->block_stride_bytes;
    w.idx_num_blocks = a->idx->num_blocks;
    w.idx_k = static_cast<const uint16_t*>(a->idx_k_new);
  }
  w.k = static_cast<const uint16_t*>(a->k_new);
  w.v = static_cast<const uint16_t*>(a->v_new);
  w.slot = a->slot;
  w.num_tokens = a->num_new_tokens;
  w.err = a->dev_err;
  if (cast_q) {
    pp.cast_src[0] = static_cast<const uint16_t*>(a->q);
    pp.cast_dst[0] = static_cast<uint8_t*>(a->q_cast);
    pp.cast_n[0] = static_cast<int64_t>(tokens) * a->num_q_heads * kDim;
  }
  if (cast_iq) {
    pp.cast_src[1] = static_cast<const uint16_t*>(a->idx_q);
    pp.cast_dst[1] = static_cast<uint8_t*>(a->idx_q_cast);
    pp.cast_n[1] = static_cast<int64_t>(tokens) * hidx * kDim;
  }
  if (!reuse) {  // the selection's rows; nothing to compute when it is reused
    pp.seq_lens = a->seq_lens;
    pp.num_seqs = a->num_seqs;
    pp.q_len = a->q_len;
    pp.heads = hkv;
    pp.row_seq = a->row_seq;
    pp.row_len = a->row_len;
  }
  if ((st = cuda_status(launch_decode_prep(pp, s))) != BSP_OK) return st;
  ++g_launches;
  mark(1);
  if (!reuse &&
      (st = index_score_impl(a->idx, iq, a->idx_q_dtype, a->block_table, a->bt_stride, a->row_seq, a->row_len, rows,
                             a->q_len, a->max_pages, a->scores, a->dev_err, stream, 1, fused ? &sel : nullptr,
                             fused ? a->sel_counters : nullptr)) != BSP_OK)
    return st;
  mark(2);
  if (!reuse && !fused &&
      (st = topk_impl(a->scores, rows, a->max_pages, a->row_seq, a->row_len, a->block_table, a->bt_stride,
                      a->kv->dtype, a->k_pages, topk_flags, a->topk_idx, a->sparse_bt, a->sparse_ctx, stream,
                      a->q_len * hkv)) != BSP_OK)
    return st;
  mark(3);
  // the attention's queries were written two launches back (or are the
  // caller's bf16 input) unless the prep kernel right before it cast them
  const bool q_early = !(reuse && a->q_dtype == BSP_FP8_E4M3);
  if ((st = sparse_pa_common(a->kv, q, a->q_dtype, a->num_q_heads, a->sparse_bt, a->sparse_ctx, rows, a->k_pages,
                             a->sm_scale, a->out, a->ws, a->ws_bytes, a->dev_err, stream, true, q_early)) != BSP_OK)
    return st;
  mark(4);
  return BSP_OK;
}

const char* bsp_status_str(bsp_status s) {
  switch (s) {
    case BSP_OK:
      return "ok";
    case BSP_ERR_INVALID_ARG:
      return "invalid argument";
    case BSP_ERR_UNSUPPORTED:
      return "unsupported size or dtype";
    case BSP_ERR_WORKSPACE:
      return "workspace too small";
    case BSP_ERR_CUDA:
      return "CUDA error";
  }
  return "unknown status";
}

int32_t bsp_last_cuda_error(void) { return g_last_cuda_error.load(); }
int64_t bsp_launch_count(void) { return g_launches.load(); }
int32_t bsp_version(void) { return 110; }

}  // extern "C"
