// index_score_prefill_tc.cu -- a2': index scores of prefill chunks as a dense
// fp8 contraction on the 5th-generation tensor cores (ROCm/ATOM PR 2962,
// commit "... page-128 block table": the prefill scorer; its scores are laid
// out as the decode scorer's, so selection and emission are shared).
//
//   S[i, t] = s_t * sum_d q[i, d] * k8[t, d]      (e4m3 x e4m3, fp32 accumulate)
//   scores[i, p] = max_{t in page p, t < L_i} S[i, t],  -inf past ceil(L_i/16)
//
// One CTA = one tile of 128 consecutive query rows of one chunk (a chunk is
// a run of query tokens of one sequence) x a range of 64 key blocks (8192
// keys).  Warp 0, lane 0 is the producer and the MMA issuer:
//   - the query tile and each pair of key blocks arrive by 2-D TMA tensor
//     loads with 128-byte swizzle (box 128 rows x 128 B) on mbarriers; key
//     rows of block b start at row b * (block_stride / 128) of the index
//     cache seen as a [rows, 128 B] tensor; a missing block loads from an
//     out-of-range row and is zero-filled;
//   - tcgen05.mma.cta_group::1.kind::f8f6f4, M = 128 queries, N = 256 keys,
//     K = 4 x 32 dims, into one of two 256-column fp32 TMEM accumulators;
//     tcgen05.commit releases the key stage and signals the accumulator.
// Warps 1..16 are the epilogue: warp w reads TMEM lanes 32*(w%4).. (its
// quarter) and a quarter of the 256 columns (64 keys = 4 pages) with two
// tcgen05.ld in flight, multiplies by the per-token fp32 scales (packed
// f32x2 multiplies), masks keys at or past the row's causal length only on
// the tile that crosses it, max-pools 16 keys into a page score by a tree of
// three-input maxima and stores 4 pages per row per tile.  The producer
// copies each tile's scales with its keys, by a 1-D TMA into a ring of 8
// shared-memory slots, so they land as early as the keys and never hold the
// accumulators up.  Accumulator double-buffering lets the MMAs of the next
// tile run under the epilogue of this one.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace bsp {

namespace {

// instruction descriptor: A = B = e4m3, N = 256 keys, M = 128 queries
constexpr uint32_t kIdesc = idesc_f8f6f4(kFmtE4m3, kFmtE4m3, 256, 128);
constexpr int kStages = 4;
constexpr int kKeyBlocksPerCta = 64;
constexpr int kEpiWarps = 16;
constexpr int kThreads = 32 * (1 + kEpiWarps);
constexpr int kTileBytes = 128 * 128;  // 128 rows x 128 B
// key scales: a ring of slots, one per tile (256 keys), filled with the
// tile's keys; a slot is reused 8 tiles later, when its epilogue is long done
constexpr int kScaleSlots = 8;
constexpr int kNumBars = 1 + 2 * kStages + 4 + kScaleSlots;
constexpr int kSmemBytes = 1024 /*align slack*/ + kTileBytes /*A*/ + kStages * 2 * kTileBytes /*B*/ +
                           kScaleSlots * 256 * 4 /*scales*/ + kNumBars * 8 /*barriers*/ + 16;

struct SmemLayout {
  uint8_t* a;
  uint8_t* b;  // [stage][256 rows][128 B]
  float* scales;  // [kScaleSlots][256]
  uint64_t* bars;  // a_full, b_full[S], b_empty[S], acc_full[2], acc_empty[2], scale_full[kScaleSlots]
  uint32_t* tmem_slot;
};

__device__ __forceinline__ SmemLayout carve(uint8_t* raw) {
  SmemLayout L;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  L.a = base;
  L.b = base + kTileBytes;
  L.scales = reinterpret_cast<float*>(L.b + kStages * 2 * kTileBytes);
  L.bars = reinterpret_cast<uint64_t*>(L.scales + kScaleSlots * 256);
  L.tmem_slot = reinterpret_cast<uint32_t*>(L.bars + kNumBars);
  return L;
}

__global__ void __launch_bounds__(kThreads, 1)
    index_score_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                               PrefillScoreParams p, int32_t oob_row) {
  extern __shared__ uint8_t smem_raw[];
  const SmemLayout sm = carve(smem_raw);
  uint64_t* a_full = sm.bars;
  uint64_t* b_full = sm.bars + 1;
  uint64_t* b_empty = sm.bars + 1 + kStages;
  uint64_t* acc_full = sm.bars + 1 + 2 * kStages;
  uint64_t* acc_empty = sm.bars + 3 + 2 * kStages;
  uint64_t* scale_full = sm.bars + 5 + 2 * kStages;  // [kScaleSlots]: a tile's key scales landed
  __shared__ int s_tok0, s_tok1, s_lmax, s_seq;
  __shared__ int s_bid[kKeyBlocksPerCta];  // the key range's block ids (-1: missing)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kb0 = blockIdx.y * kKeyBlocksPerCta;
  const int rows_per_block = static_cast<int>(p.block_stride / 128);

  pdl_wait();  // queries and row lengths come from earlier kernels
  pdl_trigger();
  if (tid == 0) {
    // locate this tile: chunks in order, ceil(size/128) tiles each
    int t = blockIdx.x, tok0 = -1, tok1 = -1;
    for (int c = 0; c < p.num_chunks; ++c) {
      const int a = p.cu_tokens[c], b = p.cu_tokens[c + 1];
      const int nt = (b - a + 127) / 128;
      if (t < nt) {
        tok0 = a + 128 * t;
        tok1 = min(b, tok0 + 128);
        break;
      }
      t -= nt;
    }
    s_tok0 = tok0;
    s_tok1 = tok1;
    s_lmax = 0;
    s_seq = tok0 >= 0 ? p.row_seq[tok0] : 0;
    mbar_init(a_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 32 * kEpiWarps);
    }
    for (int i = 0; i < kScaleSlots; ++i) mbar_init(&scale_full[i], 1);
    mbar_fence_init();
  }
  __syncthreads();
  const int tok0 = s_tok0, tok1 = s_tok1;
  if (tok0 < 0) return;  // past the last tile (the grid is an upper bound)

  // the epilogue's row and its causal length; the tile's longest row
  const int quarter = warp & 3;
  const int row = 32 * quarter + lane;
  const int tok = tok0 + row;
  const bool row_ok = warp >= 1 && tok < tok1;
  const int max_len = p.max_pages * kPage;
  int L = 0;
  if (row_ok) {
    L = min(max(p.row_len[tok], 0), max_len);
    if (p.row_seq[tok] != s_seq) set_err(p.err, BSP_DEVERR_GROUP_SEQ);
    if (warp <= 4) atomicMax(&s_lmax, L);
  }
  __syncthreads();
  const int nb = max(0, min(kKeyBlocksPerCta, (s_lmax + kBlock - 1) / kBlock - kb0));
  const int ntiles = (nb + 1) / 2;
  const int page_end = min((kb0 + kKeyBlocksPerCta) * kPagesPerSide, p.max_pages);
  const int seq = s_seq;

  if (ntiles == 0) {  // nothing of this key range below the tile's longest row
    fill_neg_inf(p.scores, p.max_pages, tok0, tok1, kb0 * kPagesPerSide, page_end);
    return;
  }

  if (tid < nb) {
    int bid = p.block_table[static_cast<int64_t>(seq) * p.bt_stride + kb0 + tid];
    if (bid < 0 || bid >= p.num_blocks) {
      set_err(p.err, BSP_DEVERR_BLOCK_ID);
      bid = -1;
    }
    s_bid[tid] = bid;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(sm.tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *sm.tmem_slot;

  auto block_row = [&](int blk) -> int {
    if (blk >= kb0 + nb) return oob_row;
    const int bid = s_bid[blk - kb0];
    return bid < 0 ? oob_row : bid * rows_per_block;
  };

  if (warp == 0) {
    if (lane == 0) {
      // key tile j (two blocks) into stage j % S, and its fp32 per-key
      // scales (512 B a block) into scale slot j % kScaleSlots; that slot's
      // previous tile, j - kScaleSlots, has finished its epilogue (the
      // producer has already seen the epilogue of tile j - S - 1 release its
      // accumulator)
      auto load_b = [&](int j) {
        const int st = j % kStages, ss = j % kScaleSlots;
        mbar_arrive_expect_tx(&b_full[st], 2 * kTileBytes);
        for (int h = 0; h < 2; ++h)
          tma_load_2d(sm.b + (st * 2 + h) * kTileBytes, &tmap_k, 0, block_row(kb0 + 2 * j + h), &b_full[st]);
        fence_proxy_async();  // the slot's earlier readers (generic proxy) before the copy's writes
        uint32_t bytes = 0;
        for (int h = 0; h < 2; ++h) {
          const int blk = kb0 + 2 * j + h;
          if (blk < kb0 + nb && s_bid[blk - kb0] >= 0) bytes += 512;
        }
        mbar_arrive_expect_tx(&scale_full[ss], bytes);
        for (int h = 0; h < 2; ++h) {
          const int blk = kb0 + 2 * j + h;
          if (blk < kb0 + nb && s_bid[blk - kb0] >= 0)
            bulk_g2s(sm.scales + ss * 256 + 128 * h,
                     p.idx_base + static_cast<int64_t>(s_bid[blk - kb0]) * p.block_stride + kFp8IndexScaleOff, 512,
                     &scale_full[ss]);
        }
      };
      mbar_arrive_expect_tx(a_full, kTileBytes);
      tma_load_2d(sm.a, &tmap_q, 0, tok0, a_full);
      for (int j = 0; j < min(kStages, ntiles); ++j) load_b(j);
      mbar_wait_sleep(a_full, 0, p.err);
      const uint32_t a_addr = smem_u32(sm.a);
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % kStages, buf = j & 1;
        mbar_wait_sleep(&b_full[st], (j / kStages) & 1, p.err);
        mbar_wait_sleep(&acc_empty[buf], ((j >> 1) & 1) ^ 1, p.err);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t b_addr = smem_u32(sm.b + st * 2 * kTileBytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_f8(tmem + buf * 256, smem_desc_sw128(a_addr + 32 * k), smem_desc_sw128(b_addr + 32 * k), kIdesc, k > 0);
        umma_commit(&b_empty[st]);
        umma_commit(&acc_full[buf]);
        // refill the previous tile's stage (its MMAs were issued an iteration
        // ago), so the MMAs just issued queue behind them without a wait
        const int jp = j - 1;
        if (jp >= 0 && jp + kStages < ntiles) {
          mbar_wait_sleep(&b_empty[jp % kStages], (jp / kStages) & 1, p.err);
          load_b(jp + kStages);
        }
      }
    }
    __syncwarp();
  } else {
    const int col0 = 64 * ((warp - 1) >> 2);  // this warp's quarter of the 256 columns (4 pages)
    for (int j = 0; j < ntiles; ++j) {
      const int buf = j & 1;
      // the tile's key scales (a missing block leaves stale but finite
      // scales: its keys lie past every row's length and are masked)
      mbar_wait_sleep(&scale_full[j % kScaleSlots], (j / kScaleSlots) & 1, p.err);
      mbar_wait_sleep(&acc_full[buf], (j >> 1) & 1, p.err);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      float v[64];
      tmem_ld32x2(tmem + (static_cast<uint32_t>(32 * quarter) << 16) + buf * 256 + col0, v);
      const float* sc = sm.scales + (j % kScaleSlots) * 256 + col0;
      const int kcol0 = (kb0 + 2 * j) * kBlock + col0;  // key of this warp's first column
      const bool whole = kcol0 + 64 <= L;  // every key of the 4 pages inside the row's causal length
      float pv[4];
#pragma unroll
      for (int pg = 0; pg < 4; ++pg) {
        float x[16];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float2 pr = fmul2(make_float2(v[16 * pg + 2 * c], v[16 * pg + 2 * c + 1]),
                                  *reinterpret_cast<const float2*>(sc + 16 * pg + 2 * c));
          x[2 * c] = pr.x, x[2 * c + 1] = pr.y;
        }
        if (!whole) {
#pragma unroll
          for (int c = 0; c < 16; ++c) x[c] = kcol0 + 16 * pg + c < L ? x[c] : -INFINITY;
        }
        pv[pg] = max16(x);
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(&acc_empty[buf]);  // the accumulator is free again
      if (row_ok) {
        const int pg0 = (kb0 + 2 * j) * kPagesPerSide + col0 / kPage;
        float* dst = p.scores + static_cast<int64_t>(tok) * p.max_pages + pg0;
        if (pg0 + 4 <= p.max_pages && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
          *reinterpret_cast<float4*>(dst) = make_float4(pv[0], pv[1], pv[2], pv[3]);
        } else {
          for (int i = 0; i < 4; ++i)
            if (pg0 + i < p.max_pages) dst[i] = pv[i];
        }
      }
    }
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
  // pages of this key range past every tile (beyond the tile's longest row)
  fill_neg_inf(p.scores, p.max_pages, tok0, tok1, (kb0 + 2 * ntiles) * kPagesPerSide, page_end);
}

}  // namespace

cudaError_t launch_index_score_prefill(const PrefillScoreParams& p, cudaStream_t s) {
  CUtensorMap tq, tk;
  const uint64_t key_rows = static_cast<uint64_t>(p.num_blocks) * (p.block_stride / 128);
  if (!make_map_u8(&tq, p.q, static_cast<uint64_t>(p.num_rows)) || !make_map_u8(&tk, p.idx_base, key_rows))
    return cudaErrorInvalidValue;
  static std::atomic<uint64_t> configured{0};
  {
    const cudaError_t e = once_per_device(configured, [] {
      return cudaFuncSetAttribute(index_score_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (e != cudaSuccess) return e;
  }
  const int max_blocks = (p.max_pages + kPagesPerSide - 1) / kPagesPerSide;
  const dim3 grid(static_cast<unsigned>(p.max_tiles),
                  static_cast<unsigned>((max_blocks + kKeyBlocksPerCta - 1) / kKeyBlocksPerCta));
  const cudaError_t e = launch_kernel(index_score_prefill_kernel, grid, dim3(kThreads), kSmemBytes, s, 0, tq, tk, p,
                                      static_cast<int32_t>(key_rows));
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

}  // namespace bsp
