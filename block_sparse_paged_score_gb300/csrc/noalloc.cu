// noalloc.cu -- bsp_sparse_pa_decode for callers that cannot allocate device
// memory.
//
// The split-K decode attention needs a workspace for its per-split partial
// results.  bsp_sparse_pa_decode takes that workspace from the caller.  Some
// callers have no way to provide one: code embedded in a host application
// that plans and reserves all device memory at start-up and forbids further
// allocation, or a caller reaching this library through the C ABI from a
// language or runtime with no device allocator at hand.  This entry point
// serves them with a fixed scratch array that lives in the library itself.
//
// The scratch is a file-scope __device__ array of kScratchBytes.  Every GPU
// that loads the library holds it until the process exits.  The first call
// on a device looks up the array's device address with cudaGetSymbolAddress
// (with that device current) and caches it; that first call should come
// before any stream capture.  The cached address does not survive
// cudaDeviceReset (the module, and with it the array, may then move).  All
// calls share the array, which keeps the last call's contents.  When this
// format's split-K plan needs a workspace, its head holds the per-row arrival
// counters the merge needs at zero, and the call clears them (an async memset
// on the caller's stream, no allocation) before it launches.  Calls that
// overlap on the GPU (concurrent streams) race on the array.
#include <mutex>

#include "../../include/bsp.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB
__device__ __align__(256) uint8_t g_pa_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

}  // namespace

extern "C" bsp_status bsp_sparse_pa_decode_noalloc(const bsp_kv_cache* kv, const void* q, int32_t q_dtype,
                                                   int32_t num_q_heads, const int32_t* sparse_bt,
                                                   const int32_t* sparse_ctx, int32_t num_rows, int32_t k_pages,
                                                   float sm_scale, void* out, int32_t* dev_err,
                                                   bsp_stream_t stream) {
  // the attention's own checks first: an invalid call enqueues nothing
  const bsp_status st =
      bsp::sparse_pa_check_args(kv, q, q_dtype, num_q_heads, sparse_bt, sparse_ctx, num_rows, k_pages, out);
  if (st != BSP_OK || num_rows == 0) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSP_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_pa_scratch) != cudaSuccess || !p) return BSP_ERR_CUDA;
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  // this format's plan: most plans merge on chip and need no workspace at
  // all; a plan that does needs its counters zeroed, and both fit the
  // scratch whenever `need` does (the counters sit at its head)
  const size_t need = bsp::sparse_pa_decode_ws_need(kv->dtype, num_rows, k_pages);
  if (need > kScratchBytes) return BSP_ERR_WORKSPACE;
  if (need > 0 &&
      cudaMemsetAsync(scratch, 0, bsp::sparse_pa_counter_bytes(num_rows), reinterpret_cast<cudaStream_t>(stream)) !=
          cudaSuccess)
    return BSP_ERR_CUDA;
  return bsp_sparse_pa_decode(kv, q, q_dtype, num_q_heads, sparse_bt, sparse_ctx, num_rows, k_pages, sm_scale, out,
                              scratch, kScratchBytes, dev_err, stream);
}
