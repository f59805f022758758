// topk_select.cu -- a3: per-row top-k of 16-token pages and the emitted
// sparse block table (ROCm/ATOM PR 2962: selection per row,
// _emit_sparse_block_table_row with pages_per_block 8 or 1, the B12 clamp, "the
// tail page is always selected"; vLLM API docs of
// MiniMaxM3SparseAiterPAMetadataBuilder: the page-16 rebase B*16 + j).
//
// Rows of up to 128 pages: one warp per row (topk_warp_kernel).  Up to 8192:
// one CTA of 256 threads per row with the keys in registers
// (topk_cta_kernel); when there are fewer rows than twice the SMs, one CTA of
// 512 or 1024 threads per row instead, up to 32768 pages.  Longer rows: one
// CTA of 512 threads per row with the keys in shared memory
// (topk_select_kernel).  Scores become order-preserving
// uint32 keys (-0 folded onto +0).  A most-significant-digit
// radix select (four 8-bit passes, shared-memory histograms, one warp scans
// the 256 bins) finds the k'-th largest key tau and how many keys equal to
// tau still fit.  Selection is then "key > tau, or key == tau and among the
// first `need` such keys in page order" -- the lower page wins a tie --
// computed with a block-wide prefix count in page order, and a second prefix
// count over the selection flags gives each selected page its output slot,
// so the table comes out in ascending page order without a sort.
#include "common.cuh"
#include "kernels.h"
#include "topk_row.cuh"

namespace bsp {

namespace {

constexpr int kThreads = 512;
constexpr int kSmemKeys = 16384;  // rows with more candidates read keys from global memory

// exclusive prefix sum over the block; returns this thread's offset and the total
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kThreads / 32 ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kThreads / 32) s_warp[lane] = w;  // inclusive
  }
  __syncthreads();
  total = s_warp[kThreads / 32 - 1];
  const int before = (warp ? s_warp[warp - 1] : 0) + x - v;
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kThreads) topk_select_kernel(TopkParams p) {
  extern __shared__ uint32_t s_keys[];
  __shared__ int s_hist[256];
  __shared__ int s_warp[kThreads / 32];
  __shared__ uint32_t s_digit;
  __shared__ int s_gt;

  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  const int max_len = p.max_pages * kPage;
  pdl_wait();  // scores come from the kernel before
  pdl_trigger();
  const int L = min(max(p.row_len[r], 0), max_len);
  const int n = (L + kPage - 1) / kPage;
  const int kk = min(p.k_pages, n);
  int32_t* ti = p.topk_idx + static_cast<int64_t>(r) * p.k_pages;
  int32_t* bt = p.sparse_bt + static_cast<int64_t>(r) * p.k_pages;
  for (int m = kk + tid; m < p.k_pages; m += kThreads) ti[m] = bt[m] = -1;
  if (kk == 0) {
    if (tid == 0) p.sparse_ctx[r] = 0;
    return;
  }
  const int n_cand = p.force_tail ? n - 1 : n;
  const int need = p.force_tail ? kk - 1 : kk;
  const float* srow = p.scores + static_cast<int64_t>(r) * p.max_pages;
  const bool in_smem = n_cand <= kSmemKeys;
  auto key_at = [&](int i) -> uint32_t { return in_smem ? s_keys[i] : order_key(srow[i]); };

  // need >= n_cand: every candidate; need == 0: none; else a radix select
  const bool all = need >= n_cand, none = need == 0;
  const bool radix = !all && !none;
  uint32_t tau = 0;
  int take_eq = 0;
  if (radix) {
    if (in_smem)
      for (int i = tid; i < n_cand; i += kThreads) s_keys[i] = order_key(srow[i]);
    uint32_t prefix = 0, mask = 0;
    int krem = need;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (tid < 256) s_hist[tid] = 0;
      __syncthreads();
      for (int i = tid; i < n_cand; i += kThreads) {
        const uint32_t k = key_at(i);
        if ((k & mask) == prefix) atomicAdd(&s_hist[(k >> shift) & 255], 1);
      }
      __syncthreads();
      if (tid < 32) {
        // lane owns bins 255-8*lane .. 248-8*lane (descending); find the digit
        // where the running count from the top first reaches krem
        int c[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = s_hist[255 - 8 * tid - j];
          sum += c[j];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += y;
        }
        int run = incl - sum;  // keys in higher bins
        if (run < krem && krem <= incl) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (run < krem && krem <= run + c[j]) {
              s_digit = static_cast<uint32_t>(255 - 8 * tid - j);
              s_gt = run;
            }
            run += c[j];
          }
        }
      }
      __syncthreads();
      krem -= s_gt;
      prefix |= s_digit << shift;
      mask |= 255u << shift;
      __syncthreads();
    }
    tau = prefix;
    take_eq = krem;
  } else if (in_smem) {
    for (int i = tid; i < n_cand; i += kThreads) s_keys[i] = 0xFFFFFFFFu;  // unused
  }

  // each thread owns a contiguous run of candidates, in page order
  const int per = (n_cand + kThreads - 1) / kThreads;
  const int b = min(tid * per, n_cand), e = min(b + per, n_cand);
  int n_eq = 0;
  if (radix)
    for (int i = b; i < e; ++i) n_eq += key_at(i) == tau;
  int tot;
  int eq_before = block_exclusive_scan(n_eq, s_warp, tot);
  int n_sel = 0;
  {
    int eqr = eq_before;
    for (int i = b; i < e; ++i) {
      bool sel = !none;
      if (radix) {
        const uint32_t k = key_at(i);
        sel = k > tau || (k == tau && eqr < take_eq);
        eqr += k == tau;
      }
      n_sel += sel;
    }
  }
  int sel_before = block_exclusive_scan(n_sel, s_warp, tot);
  const int64_t bt_row = static_cast<int64_t>(p.rows_per_seq > 0 ? r / p.rows_per_seq : p.row_seq[r]) * p.bt_stride;
  {
    int eqr = eq_before, pos = sel_before;
    int cur_blk = -1, cur_id = 0;  // this thread's pages are contiguous: few distinct blocks
    for (int i = b; i < e; ++i) {
      bool sel = !none;
      if (radix) {
        const uint32_t k = key_at(i);
        sel = k > tau || (k == tau && eqr < take_eq);
        eqr += k == tau;
      }
      if (sel && pos < need) {  // exactly `need` are selected; the bound keeps writes in the row
        if (i / kPagesPerSide != cur_blk) {
          cur_blk = i / kPagesPerSide;
          cur_id = p.block_table[bt_row + cur_blk] * p.id_mul;
        }
        ti[pos] = i;
        bt[pos] = cur_id + i % kPagesPerSide;
        ++pos;
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    const int tail_len = L - kPage * (n - 1);
    if (p.force_tail) {
      const int i = n - 1;
      ti[kk - 1] = i;
      bt[kk - 1] = p.block_table[bt_row + i / kPagesPerSide] * p.id_mul + i % kPagesPerSide;
      p.sparse_ctx[r] = kPage * (kk - 1) + tail_len;
    } else {
      // the tail page, if selected, is the last entry
      p.sparse_ctx[r] = kPage * (kk - 1) + (ti[kk - 1] == n - 1 ? tail_len : kPage);
    }
  }
}

// One warp per row for rows of up to 32*KPL candidates, four rows per CTA.
// Lane l holds the keys of pages l, l+32, ... in registers.  The k'-th key
// tau is built bit by bit from the top (keep a bit when at least `need` keys
// are >= the prefix with that bit set; one warp reduction per bit).  Pages
// are then visited in page order, 32 at a time: ballots give each page its
// rank among the keys equal to tau (the lower page wins a tie) and its output
// slot, so the table is emitted ascending with no sort and no block barrier.
template <int KPL>
__global__ void __launch_bounds__(128) topk_warp_kernel(TopkParams p) {
  __shared__ int32_t s_bt[4][(32 * KPL + kPagesPerSide - 1) / kPagesPerSide];
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (r >= p.num_rows) return;
  pdl_wait();  // scores come from the kernel before
  pdl_trigger();
  int32_t* wbt = s_bt[threadIdx.x >> 5];
  const unsigned full = 0xffffffffu, lt = (1u << lane) - 1u;
  const int max_len = p.max_pages * kPage;
  // independent loads first: the row's length and sequence, every score of
  // the row and its block ids (valid memory whatever the length)
  const int L = min(max(p.row_len[r], 0), max_len);
  const int64_t bt_row = static_cast<int64_t>(p.rows_per_seq > 0 ? r / p.rows_per_seq : p.row_seq[r]) * p.bt_stride;
  const float* srow = p.scores + static_cast<int64_t>(r) * p.max_pages;
  float sv[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) sv[i] = lane + 32 * i < p.max_pages ? srow[lane + 32 * i] : 0.f;
  for (int b = lane; b < (p.max_pages + kPagesPerSide - 1) / kPagesPerSide; b += 32)
    wbt[b] = p.block_table[bt_row + b] * p.id_mul;
  __syncwarp();
  const int n = (L + kPage - 1) / kPage;
  const int kk = min(p.k_pages, n);
  int32_t* ti = p.topk_idx + static_cast<int64_t>(r) * p.k_pages;
  int32_t* bt = p.sparse_bt + static_cast<int64_t>(r) * p.k_pages;
  for (int m = kk + lane; m < p.k_pages; m += 32) ti[m] = bt[m] = -1;
  if (kk == 0) {
    if (lane == 0) p.sparse_ctx[r] = 0;
    return;
  }
  const int n_cand = p.force_tail ? n - 1 : n;
  const int need = p.force_tail ? kk - 1 : kk;
  const bool all = need >= n_cand, none = need == 0, radix = !all && !none;
  uint32_t key[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int pg = lane + 32 * i;
    key[i] = (radix && pg < n_cand) ? order_key(sv[i]) : 0u;
  }
  uint32_t tau = 0;
  int take_eq = 0;
  if (radix) {
    // keys of real candidates are > 0 (order_key(-inf) = 0x007fffff), padding is 0
    uint32_t prefix = 0;
    for (int b = 31; b >= 0; --b) {
      const uint32_t cand = prefix | (1u << b);
      unsigned c[4] = {0u, 0u, 0u, 0u};  // four chains: no long dependent add
#pragma unroll
      for (int i = 0; i < KPL; ++i) c[i & 3] += key[i] >= cand;
      if (static_cast<int>(__reduce_add_sync(full, (c[0] + c[1]) + (c[2] + c[3]))) >= need) prefix = cand;
    }
    tau = prefix;
    unsigned gt = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) gt += key[i] > tau;
    take_eq = need - static_cast<int>(__reduce_add_sync(full, gt));
  }
  int base = 0, eq_base = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    if (32 * i >= n_cand) break;
    const int pg = lane + 32 * i;
    const bool valid = pg < n_cand;
    const bool eq = radix && valid && key[i] == tau;
    const unsigned beq = __ballot_sync(full, eq);
    const int eq_rank = eq_base + __popc(beq & lt);
    const bool sel = valid && !none && (all || key[i] > tau || (eq && eq_rank < take_eq));
    const unsigned bsel = __ballot_sync(full, sel);
    const int pos = base + __popc(bsel & lt);
    if (sel && pos < need) {
      ti[pos] = pg;
      bt[pos] = wbt[pg / kPagesPerSide] + pg % kPagesPerSide;
    }
    base += __popc(bsel);
    eq_base += __popc(beq);
  }
  if (lane == 0) {
    const int tail_len = L - kPage * (n - 1);
    if (p.force_tail) {
      const int pg = n - 1;
      ti[kk - 1] = pg;
      bt[kk - 1] = wbt[pg / kPagesPerSide] + pg % kPagesPerSide;
      p.sparse_ctx[r] = kPage * (kk - 1) + tail_len;
    }
  }
  if (!p.force_tail) {
    __syncwarp();
    if (lane == 0) p.sparse_ctx[r] = kPage * (kk - 1) + (ti[kk - 1] == n - 1 ? L - kPage * (n - 1) : kPage);
  }
}

// One CTA of 256 threads per row of up to 256*KPT pages (select_row_cta).
// Inside the decode step (rows_per_seq > 0) the row lengths come from the
// step's first kernel, done before the scorer started: only the scores need
// the wait, so the lengths, the unused tail of the outputs and the block ids
// go first.  Every CTA still waits before it exits.
constexpr int kCtaThreads = 256;

template <int KPT, int NT = kCtaThreads>
__global__ void __launch_bounds__(NT, NT == 256 ? (KPT >= 32 ? 4 : 5) : 1024 / NT) topk_cta_kernel(TopkParams p) {
  __shared__ int s_hist[4][256];
  __shared__ int s_warp[NT / 32];
  __shared__ uint32_t s_digit;
  __shared__ int s_above;
  for (int i = threadIdx.x; i < 4 * 256; i += NT) (&s_hist[0][0])[i] = 0;
  const bool in_step = p.rows_per_seq > 0;
  if (!in_step) {
    pdl_wait();  // scores (and the row lengths) come from earlier kernels
    pdl_trigger();
  }
  // a row much shorter than the kernel's width (an early prefill chunk in a
  // batch sized for the longest row) runs with fewer keys a thread: its
  // per-key work is then not spent on pages past its length
  const int n = (min(max(p.row_len[blockIdx.x], 0), p.max_pages * kPage) + kPage - 1) / kPage;
  if constexpr (KPT >= 16) {
    if (n <= NT * (KPT / 4)) {
      select_row_cta<KPT / 4, NT, false>(p, blockIdx.x, s_hist, s_warp, s_digit, s_above, in_step);
      return;
    }
  }
  if constexpr (KPT >= 8) {
    if (n <= NT * (KPT / 2)) {
      select_row_cta<KPT / 2, NT, false>(p, blockIdx.x, s_hist, s_warp, s_digit, s_above, in_step);
      return;
    }
  }
  select_row_cta<KPT, NT, false>(p, blockIdx.x, s_hist, s_warp, s_digit, s_above, in_step);
}

// 128-token blocks as the unit of selection (pages_per_block = 8).  One CTA
// of 256 threads per row; thread t owns blocks t*BPT.. with their ids in
// registers.  A block's key is the order key of the largest page score among
// its pages below n.  The same radix select and block scan as the
// page-granular CTA kernel find the selected blocks and their ranks; the
// block of rank j emits its pages (all 8, or the row's last n - 8*(nb-1)) at
// table positions 8j.., so the pages come out ascending.  With force_tail the
// tail block nb-1 is always selected and takes the last rank.
template <int BPT>
__global__ void __launch_bounds__(kCtaThreads) topk_block_kernel(TopkParams p) {
  __shared__ int s_hist[4][256];
  __shared__ int s_warp[kCtaThreads / 32];
  __shared__ uint32_t s_digit;
  __shared__ int s_above;
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 4 * 256; i += kCtaThreads) (&s_hist[0][0])[i] = 0;
  const bool in_step = p.rows_per_seq > 0;  // as in the page-granular kernel
  if (!in_step) {
    pdl_wait();
    pdl_trigger();
  }
  const int max_len = p.max_pages * kPage;
  const int L = min(max(p.row_len[r], 0), max_len);
  const int n = (L + kPage - 1) / kPage;
  const int nb = (n + kPagesPerSide - 1) / kPagesPerSide;
  const int kb = min(p.k_pages / kPagesPerSide, nb);
  int32_t* ti = p.topk_idx + static_cast<int64_t>(r) * p.k_pages;
  int32_t* bt = p.sparse_bt + static_cast<int64_t>(r) * p.k_pages;
  for (int m = tid; m < p.k_pages; m += kCtaThreads) ti[m] = bt[m] = -1;  // emitted entries overwrite these
  if (kb == 0) {
    if (tid == 0) p.sparse_ctx[r] = 0;
    if (in_step) pdl_wait();
    return;
  }
  const int n_cand = p.force_tail ? nb - 1 : nb;
  const int need = p.force_tail ? kb - 1 : kb;
  const bool all = need >= n_cand, none = need == 0, radix = !all && !none;

  const int first = tid * BPT;
  const int64_t bt_row = static_cast<int64_t>(p.rows_per_seq > 0 ? r / p.rows_per_seq : p.row_seq[r]) * p.bt_stride;
  int32_t ids[BPT];
#pragma unroll
  for (int j = 0; j < BPT; ++j) ids[j] = first + j < nb ? p.block_table[bt_row + first + j] * p.id_mul : 0;
  if (in_step) {
    pdl_wait();  // the scores
    pdl_trigger();
  }
  const float* srow = p.scores + static_cast<int64_t>(r) * p.max_pages;
  // rows of a multiple of 8 pages: a block's 8 scores are two aligned float4
  // (the score buffer is 16-byte aligned), masked to the pages below n
  const bool vec = (p.max_pages & 7) == 0;
  uint32_t key[BPT];
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    key[j] = 0u;
    const int b = first + j;
    if (radix && b < n_cand) {
      const int p0 = b * kPagesPerSide, np = min(kPagesPerSide, n - p0);
      float best;
      if (vec) {
        const float4 x = reinterpret_cast<const float4*>(srow + p0)[0];
        const float4 y = reinterpret_cast<const float4*>(srow + p0)[1];
        const float v[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
        best = v[0];
#pragma unroll
        for (int k = 1; k < 8; ++k) best = k < np ? fmaxf(best, v[k]) : best;
      } else {
        best = srow[p0];
        for (int pg = p0 + 1; pg < p0 + np; ++pg) best = fmaxf(best, srow[pg]);
      }
      key[j] = order_key(best);
    }
  }

  uint32_t tau = 0;
  int take_eq = 0;
  if (radix) radix_select_regs<BPT>(key, first, n_cand, need, s_hist, s_digit, s_above, warp, lane, tau, take_eq);

  int gt = 0, eq = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    const bool valid = first + j < n_cand;
    gt += valid && (all || (radix && key[j] > tau));
    eq += valid && radix && key[j] == tau;
  }
  const int before = cta_exclusive_packed((gt << 16) | eq, s_warp, warp, lane);
  int eqr = before & 0xFFFF;
  int rank = (before >> 16) + min(eqr, take_eq);
  bool tail_sel = false;
  const int tail_pages = n - kPagesPerSide * (nb - 1);  // pages of the row's last block
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    const int b = first + j;
    const bool valid = b < n_cand;
    const bool is_eq = valid && radix && key[j] == tau;
    const bool sel = valid && !none && (all || (radix && key[j] > tau) || (is_eq && eqr < take_eq));
    eqr += is_eq;
    if (sel && rank < need) {
      const int np = b == nb - 1 ? tail_pages : kPagesPerSide;
      for (int k = 0; k < np; ++k) {
        ti[kPagesPerSide * rank + k] = kPagesPerSide * b + k;
        bt[kPagesPerSide * rank + k] = ids[j] + k;
      }
      ++rank;
    }
    if (b == nb - 1) tail_sel = sel;
  }
  // the owner of block nb-1 finishes the row: the forced tail block, and the
  // context length (the tail block, if selected, holds the last entries)
  const int tail_len = L - kPage * (n - 1);
  if (first <= nb - 1 && nb - 1 < first + BPT) {
    int32_t id = ids[0];
#pragma unroll
    for (int j = 1; j < BPT; ++j)
      if (nb - 1 - first == j) id = ids[j];
    if (p.force_tail)
      for (int k = 0; k < tail_pages; ++k) {
        ti[kPagesPerSide * (kb - 1) + k] = kPagesPerSide * (nb - 1) + k;
        bt[kPagesPerSide * (kb - 1) + k] = id + k;
      }
    p.sparse_ctx[r] = (p.force_tail || tail_sel)
                          ? kPage * (kPagesPerSide * (kb - 1) + tail_pages - 1) + tail_len
                          : kPage * kPagesPerSide * kb;
  }
}

template <int BPT>
cudaError_t launch_blocks(const TopkParams& p, cudaStream_t s) {
  const cudaError_t e = launch_kernel(topk_block_kernel<BPT>, dim3(p.num_rows), dim3(kCtaThreads), 0, s, 0, p);
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

int device_sms_count() {
  static std::atomic<int> table[kMaxDevices];
  return cached_per_device(table, [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
      v = 0;
    return v > 0 ? v : 1;
  });
}

template <int KPT, int NT = kCtaThreads>
cudaError_t launch_cta(const TopkParams& p, cudaStream_t s) {
  const cudaError_t e = launch_kernel(topk_cta_kernel<KPT, NT>, dim3(p.num_rows), dim3(NT), 0, s, 0, p);
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

template <int KPL>
cudaError_t launch_warp(const TopkParams& p, cudaStream_t s) {
  const cudaError_t e = launch_kernel(topk_warp_kernel<KPL>, dim3((p.num_rows + 3) / 4), dim3(128), 0, s, 0, p);
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

}  // namespace

cudaError_t launch_topk_select(const TopkParams& p, cudaStream_t s) {
  if (p.num_rows == 0) return cudaSuccess;
  if (p.blocks) {
    const int nblk = (p.max_pages + kPagesPerSide - 1) / kPagesPerSide;
    if (nblk <= 1 * kCtaThreads) return launch_blocks<1>(p, s);
    if (nblk <= 2 * kCtaThreads) return launch_blocks<2>(p, s);
    if (nblk <= 4 * kCtaThreads) return launch_blocks<4>(p, s);
    if (nblk <= 8 * kCtaThreads) return launch_blocks<8>(p, s);
    if (nblk <= 16 * kCtaThreads) return launch_blocks<16>(p, s);
    return launch_blocks<32>(p, s);  // max_pages <= 65536
  }
  if (p.max_pages <= 128) return launch_warp<4>(p, s);  // one warp a row (longer rows measured slower)
  // Few long rows leave most SMs idle with one 256-thread CTA a row: give
  // each row a 512- or 1024-thread CTA instead (fewer keys per thread)
  if (p.max_pages > kCtaThreads && p.max_pages <= 32 * 1024 &&
      p.num_rows < 2 * device_sms_count()) {
    if (p.max_pages <= 512) return launch_cta<1, 512>(p, s);
    if (p.max_pages <= 2 * 1024) return launch_cta<2, 1024>(p, s);
    if (p.max_pages <= 4 * 1024) return launch_cta<4, 1024>(p, s);
    if (p.max_pages <= 8 * 1024) return launch_cta<8, 1024>(p, s);
    if (p.max_pages <= 16 * 1024) return launch_cta<16, 1024>(p, s);
    return launch_cta<32, 1024>(p, s);
  }
  if (p.max_pages <= 1 * kCtaThreads) return launch_cta<1>(p, s);
  if (p.max_pages <= 2 * kCtaThreads) return launch_cta<2>(p, s);
  if (p.max_pages <= 4 * kCtaThreads) return launch_cta<4>(p, s);
  if (p.max_pages <= 8 * kCtaThreads) return launch_cta<8>(p, s);
  if (p.max_pages <= 16 * kCtaThreads) return launch_cta<16>(p, s);
  if (p.max_pages <= 32 * kCtaThreads) return launch_cta<32>(p, s);
  const int cand = p.max_pages < kSmemKeys ? p.max_pages : kSmemKeys;
  const size_t bytes = static_cast<size_t>(cand) * 4;
  static std::atomic<uint64_t> configured{0};
  {
    const cudaError_t e = once_per_device(configured, [] {
      return cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemKeys * 4);
    });
    if (e != cudaSuccess) return e;
  }
  const cudaError_t e = launch_kernel(topk_select_kernel, dim3(p.num_rows), dim3(kThreads), bytes, s, 0, p);
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

}  // namespace bsp
