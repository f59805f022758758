// topk_row.cuh -- one row's top-k of pages by one CTA, shared by the
// selector kernels (topk_select.cu) and the scorer's fused selection tail
// (index_score.cu): the order-preserving key of a score, the register radix
// select, the packed CTA scan and the per-row selection with its emission
// (ROCm/ATOM PR 2962: selection per row, _emit_sparse_block_table_row, "the
// tail page is always selected"; vLLM API docs of the metadata builder: the
// page-16 rebase B*16 + j).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace bsp {

// Scores as order-preserving uint32 keys; -0 folds onto +0.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Radix select over keys held in registers by a CTA: thread t holds NK keys
// of candidates first..first+NK-1 (valid below n_cand).  Up to four 8-bit
// passes, most significant digit first, each with one shared-memory
// histogram (the four are zeroed by the caller before its first
// __syncthreads) and one warp scanning its 256 bins from the top, find tau,
// the need-th largest key, and take_eq, how many keys equal to tau are taken.
// When the bin holding the need-th key holds exactly the keys still needed,
// every key of the bin is taken and the passes stop there: tau becomes the
// bin's lowest key value (the digits below zero), so "key > tau, or key ==
// tau" is exactly the bin.  Block-wide: every thread of the CTA calls it.
template <int NK>
__device__ __forceinline__ void radix_select_regs(const uint32_t (&key)[NK], int first, int n_cand, int need,
                                                  int (&s_hist)[4][256], uint32_t& s_digit, int& s_above, int warp,
                                                  int lane, uint32_t& tau, int& take_eq) {
  uint32_t prefix = 0, mask = 0;
  int krem = need;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    __syncthreads();  // histograms zeroed; the previous pass's digit read
#pragma unroll
    for (int j = 0; j < NK; ++j)
      if (first + j < n_cand && (key[j] & mask) == prefix) atomicAdd(&s_hist[pass][(key[j] >> shift) & 255], 1);
    __syncthreads();
    if (warp == 0) {
      // lane owns bins 255-8*lane .. 248-8*lane (descending); find the digit
      // where the running count from the top first reaches krem
      int c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = s_hist[pass][255 - 8 * lane - j];
        sum += c[j];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int run = incl - sum;  // keys in higher bins
      if (run < krem && krem <= incl) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run < krem && krem <= run + c[j]) {
            s_digit = static_cast<uint32_t>(255 - 8 * lane - j) | (static_cast<uint32_t>(c[j]) << 8);
            s_above = run;
          }
          run += c[j];
        }
      }
    }
    __syncthreads();
    const uint32_t dc = s_digit;
    krem -= s_above;
    prefix |= (dc & 255u) << shift;
    mask |= 255u << shift;
    if (static_cast<int>(dc >> 8) == krem) break;  // the whole bin is taken
  }
  tau = prefix;
  take_eq = krem;
}

// exclusive prefix over the CTA (in thread order) of a per-thread count
// packed as (gt << 16) | eq; both fields stay below 2^16
__device__ __forceinline__ int cta_exclusive_packed(int packed, int* s_warp, int warp, int lane) {
  int x = packed;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  int before = x - packed;
  for (int w = 0; w < warp; ++w) before += s_warp[w];
  return before;
}

// One row of up to NT*KPT pages selected by a CTA of NT threads.  Thread t
// owns the KPT consecutive pages t*KPT.. in registers (and the ids of the one
// or two 128-token blocks they lie in, loaded up front).  A radix select of
// four 8-bit passes (one shared-memory histogram per pass, one warp scans its
// 256 bins) finds tau, the need-th largest key, and how many keys equal to
// tau are taken.  One block-wide scan of the packed per-thread counts (keys >
// tau, keys == tau) then gives every thread the output slot of its first
// selected page: the keys > tau before it, plus the ties before it up to the
// number taken (the lower page wins a tie).  Pages come out in ascending
// order with no sort.  s_hist must be zero on entry.  With wait_scores the
// CTA waits for the kernel before (griddepcontrol) just before it reads the
// scores, and before it returns early.  L2_ONLY reads the scores through L2
// (for scores written by other CTAs of the same kernel).
template <int KPT, int NT, bool L2_ONLY>
__device__ __forceinline__ void select_row_cta(const TopkParams& p, int r, int (&s_hist)[4][256], int* s_warp,
                                               uint32_t& s_digit, int& s_above, bool wait_scores) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int max_len = p.max_pages * kPage;
  const int L = min(max(p.row_len[r], 0), max_len);
  const int n = (L + kPage - 1) / kPage;
  const int kk = min(p.k_pages, n);
  int32_t* ti = p.topk_idx + static_cast<int64_t>(r) * p.k_pages;
  int32_t* bt = p.sparse_bt + static_cast<int64_t>(r) * p.k_pages;
  for (int m = kk + tid; m < p.k_pages; m += NT) ti[m] = bt[m] = -1;
  if (kk == 0) {
    if (tid == 0) p.sparse_ctx[r] = 0;
    if (wait_scores) pdl_wait();
    return;
  }
  const int n_cand = p.force_tail ? n - 1 : n;
  const int need = p.force_tail ? kk - 1 : kk;
  const bool all = need >= n_cand, none = need == 0, radix = !all && !none;

  // independent loads: the ids of the blocks this thread's pages lie in
  // (pages first.. first+KPT-1 span NB blocks from b0) and its scores
  constexpr int NB = KPT >= kPagesPerSide ? KPT / kPagesPerSide : 1;
  const int first = tid * KPT;
  const int nblk = (p.max_pages + kPagesPerSide - 1) / kPagesPerSide;
  const int b0 = first / kPagesPerSide;
  const int64_t bt_row = static_cast<int64_t>(p.rows_per_seq > 0 ? r / p.rows_per_seq : p.row_seq[r]) * p.bt_stride;
  int32_t ids[NB];
#pragma unroll
  for (int k = 0; k < NB; ++k) ids[k] = b0 + k < nblk ? p.block_table[bt_row + b0 + k] * p.id_mul : 0;
  if (wait_scores) {
    pdl_wait();  // the scores
    pdl_trigger();
  }
  const float* srow = p.scores + static_cast<int64_t>(r) * p.max_pages;
  uint32_t key[KPT];
  if (KPT % 4 == 0 && (p.max_pages & 3) == 0 && (reinterpret_cast<uintptr_t>(p.scores) & 15) == 0 &&
      first + KPT <= n_cand) {
    // whole 16-byte runs (the rows start 16-byte aligned)
#pragma unroll
    for (int j = 0; j < KPT; j += 4) {
      const float4* a = reinterpret_cast<const float4*>(srow + first + j);
      const float4 v = L2_ONLY ? __ldcg(a) : *a;
      key[j] = radix ? order_key(v.x) : 0u;
      key[j + 1] = radix ? order_key(v.y) : 0u;
      key[j + 2] = radix ? order_key(v.z) : 0u;
      key[j + 3] = radix ? order_key(v.w) : 0u;
    }
  } else {
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      key[j] = (radix && first + j < n_cand) ? order_key(L2_ONLY ? __ldcg(srow + first + j) : srow[first + j]) : 0u;
  }

  uint32_t tau = 0;
  int take_eq = 0;
  if (radix) radix_select_regs<KPT>(key, first, n_cand, need, s_hist, s_digit, s_above, warp, lane, tau, take_eq);

  // keys > tau and keys == tau of this thread as bit masks (bit j: page
  // first + j), their counts scanned over the block in page order
  static_assert(KPT <= 32, "one bit a page");
  uint32_t gmask = 0, emask = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const bool valid = first + j < n_cand;
    gmask |= static_cast<uint32_t>(valid && (all || (radix && key[j] > tau))) << j;
    emask |= static_cast<uint32_t>(valid && radix && key[j] == tau) << j;
  }
  const int before = cta_exclusive_packed((__popc(gmask) << 16) | __popc(emask), s_warp, warp, lane);
  const int eqr = before & 0xFFFF;  // ties in earlier threads
  int pos = (before >> 16) + min(eqr, take_eq);
  // the selection: every key > tau, and the ties while fewer than take_eq
  // came before (the lower page wins)
  uint32_t smask = none ? 0u : gmask;
  uint32_t ties = emask;
  for (int left = take_eq - eqr; left > 0 && ties; --left) {
    smask |= ties & (0u - ties);  // the lowest remaining tie
    ties &= ties - 1;
  }
  const bool tail_sel = first <= n - 1 && n - 1 < first + KPT && ((smask >> (n - 1 - first)) & 1u);
  for (uint32_t m = smask; m && pos < need; m &= m - 1, ++pos) {
    const int j = __ffs(m) - 1, pg = first + j;
    int32_t id = ids[0];
#pragma unroll
    for (int k = 1; k < NB; ++k)
      if (j / kPagesPerSide == k) id = ids[k];
    ti[pos] = pg;
    bt[pos] = id + pg % kPagesPerSide;  // first % 8 == 0 when a thread spans blocks
  }
  // the owner of page n-1 finishes the row: the forced tail entry, and the
  // context length (the tail page, if selected, is the last entry)
  if (first <= n - 1 && n - 1 < first + KPT) {
    const int pg = n - 1;
    const int tail_len = L - kPage * (n - 1);
    if (p.force_tail) {
      ti[kk - 1] = pg;
      int32_t id = ids[0];
#pragma unroll
      for (int k = 1; k < NB; ++k)
        if (pg / kPagesPerSide - b0 == k) id = ids[k];
      bt[kk - 1] = id + pg % kPagesPerSide;
      p.sparse_ctx[r] = kPage * (kk - 1) + tail_len;
    } else {
      p.sparse_ctx[r] = kPage * (kk - 1) + (tail_sel ? tail_len : kPage);
    }
  }
}

}  // namespace bsp
