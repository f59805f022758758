// kernels.h -- launch parameters and host launchers of the libbsp kernels.
// Host-side only types; the C ABI in api.cu validates arguments and calls
// these.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/bsp.h"

namespace bsp {

// Per-device host state.  A kernel's dynamic shared-memory opt-in and the
// occupancy it allows belong to the current device's context, so they are
// kept per device (one process may drive several GPUs) and in atomics
// (several host threads may call the library at once; every writer stores
// the same value).
constexpr int kMaxDevices = 64;
inline int current_device() {
  int d = -1;
  return (cudaGetDevice(&d) == cudaSuccess && d >= 0 && d < kMaxDevices) ? d : -1;
}
// set() once per device; `done` holds one bit per device that has it (a
// device outside the table runs set() every time)
template <typename F>
inline cudaError_t once_per_device(std::atomic<uint64_t>& done, F set) {
  const int d = current_device();
  const uint64_t bit = d >= 0 ? (uint64_t{1} << d) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  const cudaError_t e = set();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}
// a positive value per device, computed by get() the first time
template <typename F>
inline int cached_per_device(std::atomic<int> (&table)[kMaxDevices], F get) {
  const int d = current_device();
  if (d < 0) return get();
  int v = table[d].load(std::memory_order_acquire);
  if (!v) {
    v = get();
    table[d].store(v, std::memory_order_release);
  }
  return v;
}

// Every kernel of the library goes through this launch: programmatic stream
// serialization (the kernel may be scheduled while the previous kernel on the
// stream drains; it waits on griddepcontrol before touching global memory)
// and, for cluster > 1, a 1-D thread-block cluster of that size.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

struct KvWriteParams {
  int32_t kv_dtype, hkv;
  uint8_t* k_base;
  uint8_t* v_base;
  int64_t id_stride, num_blocks;
  float k_scale, v_scale;
  int32_t idx_dtype, hidx;  // hidx = 0: no index write
  uint8_t* idx_base;
  int64_t idx_block_stride, idx_num_blocks;
  const uint16_t* k;
  const uint16_t* v;
  const uint16_t* idx_k;
  const int64_t* slot;
  int32_t num_tokens;
  int32_t* err;
};
cudaError_t launch_kv_page_write(const KvWriteParams& p, cudaStream_t s);

// write + the two e4m3 query casts + decode row lengths in one launch
struct DecodePrepParams {
  KvWriteParams write;
  const uint16_t* cast_src[2];  // NULL: no cast
  uint8_t* cast_dst[2];
  int64_t cast_n[2];
  const int32_t* seq_lens;
  int32_t num_seqs, q_len, heads;
  int32_t* row_seq;
  int32_t* row_len;
  int64_t write_blocks, cast_blocks[2];  // filled by the launcher
};
cudaError_t launch_decode_prep(DecodePrepParams p, cudaStream_t s);
cudaError_t launch_cast_e4m3(const uint16_t* x, uint8_t* out, int64_t n, cudaStream_t s);
cudaError_t launch_row_lengths_decode(const int32_t* seq_lens, int32_t num_seqs, int32_t q_len, int32_t heads,
                                      int32_t* row_seq, int32_t* row_len, cudaStream_t s);
cudaError_t launch_row_lengths_prefill(const int32_t* req, const int32_t* pos, int32_t n, int32_t heads,
                                       int32_t* row_seq, int32_t* row_len, cudaStream_t s);

struct TopkParams {
  const float* scores;
  int32_t num_rows, max_pages;
  const int32_t* row_seq;
  const int32_t* row_len;
  const int32_t* block_table;
  int32_t bt_stride, id_mul;  // id = block * id_mul + p % 8
  int32_t k_pages, force_tail;
  int32_t rows_per_seq;  // > 0: row r belongs to sequence r / rows_per_seq (no row_seq lookup first)
  int32_t blocks;        // 1: select 128-token blocks (k_pages / 8 of them), each emitting its pages
  int32_t* topk_idx;
  int32_t* sparse_bt;
  int32_t* sparse_ctx;
};
cudaError_t launch_topk_select(const TopkParams& p, cudaStream_t s);

struct IndexScoreParams {
  int32_t idx_dtype, hidx;
  const uint8_t* idx_base;
  int64_t block_stride, num_blocks;
  const void* q;
  int32_t q_dtype;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* row_seq;
  const int32_t* row_len;
  int32_t num_rows, num_tokens, q_group, max_pages;
  int32_t blocks_per_chunk, num_groups, stages;  // filled by the launcher
  int32_t seq_is_group;  // 1: rows are decode-ordered, group g is sequence g (no row_seq lookup first)
  float* scores;
  int32_t* err;
  // decode step, optional (NULL: off): the scorer also selects.  One int32
  // per (group, index head), zero on entry and left zero: the last CTA of a
  // group to finish its chunk selects the group's rows with `sel` (see
  // index_score_can_select).
  int32_t* sel_counters;
  TopkParams sel;
};
cudaError_t launch_index_score(IndexScoreParams p, int num_sms, cudaStream_t s);
// the tcgen05 scorer for MXFP4 keys and e4m3 queries (launch_index_score
// takes it when supported)
bool index_score_mx_tc_supported(const IndexScoreParams& p);
int index_score_mx_tc_occupancy();
cudaError_t launch_index_score_mx_tc(const IndexScoreParams& p, dim3 grid, cudaStream_t s);
// whether launch_index_score fuses the selection for these rows (else the
// caller launches the selector)
bool index_score_can_select(int32_t idx_dtype, int32_t q_dtype, int32_t max_pages, int32_t blocks);



struct SparsePaParams {
  int32_t kv_dtype, hkv;
  const uint8_t* k_base;
  const uint8_t* v_base;
  int64_t id_stride, num_ids;
  float k_scale, v_scale;
  const void* q;
  int32_t q_dtype, group;
  const int32_t* sparse_bt;
  const int32_t* sparse_ctx;
  int32_t num_rows, k_pages;
  float sm_scale;
  void* out;
  float* ws;  // partials when nsplit > 8 (not clustered)
  int32_t nsplit, pages_per_split;
  int32_t cluster;  // 2..8: the row's splits form a cluster and merge on chip
  int32_t ring;     // pages in flight per warp
  int32_t q_early;  // 1: q was written before the kernel launched ahead of this one (load it before the wait)
  int32_t* err;
};
// split plan shared by the launcher and the workspace query
struct PaPlan {
  int32_t nsplit, pages_per_split, cluster, ring;
};
PaPlan sparse_pa_plan(int32_t kv_dtype, int32_t num_rows, int32_t k_pages, int num_sms);
// prefill: one CTA per row, written directly
PaPlan sparse_pa_prefill_plan(int32_t kv_dtype, int32_t k_pages);
size_t sparse_pa_ws_bytes(int32_t num_rows, const PaPlan& plan);
// bytes of the per-row arrival counters at the start of the workspace
size_t sparse_pa_counter_bytes(int32_t num_rows);
cudaError_t launch_sparse_pa(const SparsePaParams& p, cudaStream_t s, int* launches);
// the argument checks of the attention calls (the status they return before
// anything is enqueued)
bsp_status sparse_pa_check_args(const bsp_kv_cache* kv, const void* q, int32_t q_dtype, int32_t num_q_heads,
                                const int32_t* sparse_bt, const int32_t* sparse_ctx, int32_t num_rows,
                                int32_t k_pages, const void* out);
// workspace bytes the decode plan of this KV format needs on the current device
size_t sparse_pa_decode_ws_need(int32_t kv_dtype, int32_t num_rows, int32_t k_pages);

struct PrefillScoreParams {
  const uint8_t* idx_base;
  int64_t block_stride, num_blocks;
  const uint8_t* q;  // e4m3 [tokens, 128]
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* row_seq;
  const int32_t* row_len;
  int32_t num_rows;
  const int32_t* cu_tokens;
  int32_t num_chunks, max_tiles, max_pages;
  float* scores;
  int32_t* err;
};
cudaError_t launch_index_score_prefill(const PrefillScoreParams& p, cudaStream_t s);
// the same for an MXFP4 index cache (e2m1 keys, e8m0 scales per 32 dims)
cudaError_t launch_index_score_prefill_mx(const PrefillScoreParams& p, cudaStream_t s);

}  // namespace bsp
