// index_score_prefill_mx_tc.cu -- a2' for an MXFP4 index cache: the index
// scores of prefill chunks as a dense contraction on the 5th-generation
// tensor cores, e4m3 queries against e2m1 keys with one e8m0 scale per 32
// dims (ROCm/ATOM PR 2962: the MXFP4 prefill scorer, "score_prefill" over
// the data and scale views of the index page; its scores laid out as the
// other scorers').
//
//   S[i, t] = sum_G 2^(e[t, G] - 127) * sum_{d in group G} q[i, d] * k[t, d]
//   scores[i, p] = max_{t in page p, t < L_i} S[i, t],  -inf past ceil(L_i/16)
//
// One CTA = one tile of 128 consecutive query rows of one chunk x a range of
// 64 key blocks, as the fp8 prefill scorer; a key tile is one 128-token
// block.  The group scales go to the tensor core itself: each key tile is
// four tcgen05.mma kind::mxf8f6f4.block_scale (A = queries, e4m3, M = 128;
// B = keys, e2m1, N = 128; K = 32 = one scale group each, the descriptor's
// scale-factor id picking group g's byte) accumulating into one fp32 TMEM
// accumulator of 128 columns, double-buffered.
//   - warp 0, lane 0: the query tile by a 2-D TMA load with 128-byte
//     swizzle; each key block by a 2-D TMA load of 4-bit data type
//     16U4_ALIGN16B (every 8 packed bytes of 16 e2m1 values unpacked into a
//     16-byte slot, the layout the f8f6f4 kinds read), 128-byte swizzle,
//     into a 4-stage ring; the MMAs;
//   - warps 1..4: the scale factors in TMEM.  A cell of 32 bits holds the
//     four group scales of one key (the field stores them so: 4 bytes a
//     key); key n's cell goes to lane 32p + n % 32 of every 32-lane
//     sub-partition p, column (slot) + n / 32.  Each of the four warps
//     writes its own sub-partition's copy with tcgen05.st, one scale slot of
//     4 columns per ring stage, and the query scales (all 1.0) once;
//   - warps 5..12: the epilogue.  Warp w reads TMEM lanes 32*(w%4).. (its
//     quarter of the query rows) and 64 of the 128 keys (4 pages) with two
//     tcgen05.ld in flight, masks keys at or past the row's causal length on
//     the tile that crosses it and max-pools 16 keys into a page score (a
//     tree of three-input maxima); there is no per-key multiply left.
//
// Every wait is bounded; after a timed-out wait a role stops waiting (the
// error word is set) and the CTA frees its TMEM and returns.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace bsp {

namespace {

constexpr int kStages = 4;
constexpr int kKeyBlocksPerCta = 64;
constexpr int kKeys = 128;            // keys a tile (one block)
constexpr int kEpiWarps = 8;
constexpr int kScaleWarps = 4;
constexpr int kThreads = 32 * (1 + kScaleWarps + kEpiWarps);
constexpr int kQTile = 128 * 128;     // 128 query rows x 128 B
constexpr int kKeyTile = kKeys * 128;  // 128 keys x 128 padded bytes
constexpr uint32_t kKeyTx = kKeys * 64;  // the packed bytes the tensor load reads
// TMEM columns: two accumulators, the query scales, one key-scale slot per stage
constexpr uint32_t kColSfa = 256, kColSfb = 288, kSfbStride = 32;
constexpr int kSmemUsed = 1024 /*align slack*/ + kQTile + kStages * kKeyTile + 32 * 8 /*barriers*/ + 16;
// one CTA per SM: each holds all 512 TMEM columns, so a second resident CTA
// would only wait in tcgen05.alloc
constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;

struct SmemLayout {
  uint8_t* a;       // queries
  uint8_t* b;       // [stage][128 keys][128 B]
  uint64_t* bars;   // a_full, b_full[S], b_empty[S], sf_full[S], acc_full[2], acc_empty[2]
  uint32_t* tmem_slot;
};

__device__ __forceinline__ SmemLayout carve(uint8_t* raw) {
  SmemLayout L;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  L.a = base;
  L.b = base + kQTile;
  L.bars = reinterpret_cast<uint64_t*>(L.b + kStages * kKeyTile);
  L.tmem_slot = reinterpret_cast<uint32_t*>(L.bars + 32);
  return L;
}

__global__ void __launch_bounds__(kThreads, 1)
    index_score_prefill_mx_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                                  PrefillScoreParams p, int32_t oob_row) {
  extern __shared__ uint8_t smem_raw[];
  const SmemLayout sm = carve(smem_raw);
  uint64_t* a_full = sm.bars;
  uint64_t* b_full = sm.bars + 1;
  uint64_t* b_empty = sm.bars + 1 + kStages;
  uint64_t* sf_full = sm.bars + 1 + 2 * kStages;
  uint64_t* acc_full = sm.bars + 1 + 3 * kStages;
  uint64_t* acc_empty = sm.bars + 3 + 3 * kStages;
  __shared__ int s_tok0, s_tok1, s_lmax, s_seq;
  __shared__ int s_bid[kKeyBlocksPerCta];  // the key range's block ids (-1: missing)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kb0 = blockIdx.y * kKeyBlocksPerCta;

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
      mbar_init(&sf_full[i], 32 * kScaleWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 32 * kEpiWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();
  const int tok0 = s_tok0, tok1 = s_tok1;
  if (tok0 < 0) return;  // past the last tile (the grid is an upper bound)

  // the epilogue's row and its causal length; the tile's longest row
  const bool epi = warp >= 1 + kScaleWarps;
  const int quarter = warp & 3;
  const int row = 32 * quarter + lane;
  const int tok = tok0 + row;
  const bool row_ok = epi && tok < tok1;
  const bool first_epi = epi && warp < 1 + kScaleWarps + 4;  // one warp per quarter
  const int max_len = p.max_pages * kPage;
  int L = 0;
  if (row_ok) {
    L = min(max(p.row_len[tok], 0), max_len);
    if (p.row_seq[tok] != s_seq) set_err(p.err, BSP_DEVERR_GROUP_SEQ);
    if (first_epi) atomicMax(&s_lmax, L);
  }
  __syncthreads();
  const int ntiles = max(0, min(kKeyBlocksPerCta, (s_lmax + kBlock - 1) / kBlock - kb0));
  const int page_end = min((kb0 + kKeyBlocksPerCta) * kPagesPerSide, p.max_pages);
  const int seq = s_seq;

  if (ntiles == 0) {  // nothing of this key range below the tile's longest row
    fill_neg_inf(p.scores, p.max_pages, tok0, tok1, kb0 * kPagesPerSide, page_end);
    return;
  }

  if (tid < ntiles) {
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
  const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
  if (warp >= 1 && warp <= kScaleWarps) {  // the queries' scales: all 1.0, in each sub-partition's copy
    tmem_st4(tmem + lane_base + kColSfa, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  }
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  if (warp == 0) {
    if (lane == 0) {
      // key tile j = block kb0 + j
      auto load_b = [&](int j) {
        const int st = j % kStages;
        const int bid = s_bid[j];
        const int r0 = bid < 0 ? oob_row : static_cast<int>(static_cast<int64_t>(bid) * (p.block_stride / 64));
        mbar_arrive_expect_tx(&b_full[st], kKeyTx);
        tma_load_2d(sm.b + st * kKeyTile, &tmap_k, 0, r0, &b_full[st]);
      };
      bool alive = true;
      mbar_arrive_expect_tx(a_full, kQTile);
      tma_load_2d(sm.a, &tmap_q, 0, tok0, a_full);
      for (int j = 0; j < min(kStages, ntiles); ++j) load_b(j);
      alive = mbar_wait_sleep(a_full, 0, p.err);
      const uint32_t a_addr = smem_u32(sm.a);
      for (int j = 0; j < ntiles && alive; ++j) {
        const int st = j % kStages, buf = j & 1;
        alive = mbar_wait_sleep(&b_full[st], (j / kStages) & 1, p.err) &&
                mbar_wait_sleep(&sf_full[st], (j / kStages) & 1, p.err) &&
                mbar_wait_sleep(&acc_empty[buf], ((j >> 1) & 1) ^ 1, p.err);
        if (!alive) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t b_addr = smem_u32(sm.b + st * kKeyTile);
#pragma unroll
        for (int g = 0; g < 4; ++g)
          umma_mx(tmem + buf * kKeys, smem_desc_sw128(a_addr + 32 * g), smem_desc_sw128(b_addr + 32 * g),
                  idesc_mxf8f6f4(kFmtE4m3, kFmtE2m1, kKeys, 128, g, g), tmem + kColSfa,
                  tmem + kColSfb + kSfbStride * st, g > 0);
        umma_commit(&b_empty[st]);
        umma_commit(&acc_full[buf]);
        const int jp = j - 1;  // refill the previous tile's stage (its MMAs were issued an iteration ago)
        if (jp >= 0 && jp + kStages < ntiles) {
          alive = mbar_wait_sleep(&b_empty[jp % kStages], (jp / kStages) & 1, p.err);
          if (alive) load_b(jp + kStages);
        }
      }
      if (alive) mbar_wait_sleep(&b_empty[(ntiles - 1) % kStages], ((ntiles - 1) / kStages) & 1, p.err);
    }
    __syncwarp();
  } else if (warp <= kScaleWarps) {
    // key tile j's scale cells into slot j % S: lane l holds keys l, 32 + l,
    // 64 + l, 96 + l (columns 0..3 of the slot); every sub-partition its copy
    bool alive = true;
    for (int j = 0; j < ntiles && alive; ++j) {
      const int st = j % kStages;
      if (j >= kStages) alive = mbar_wait_sleep(&b_empty[st], ((j / kStages) - 1) & 1, p.err);  // the slot's MMAs are done
      if (!alive) break;
      const int bid = s_bid[j];
      uint32_t w[4] = {0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu};  // a missing block: zero keys, unit scales
      if (bid >= 0) {
        const uint32_t* cells = reinterpret_cast<const uint32_t*>(
            p.idx_base + static_cast<int64_t>(bid) * p.block_stride + kMxScaleOff);
#pragma unroll
        for (int c = 0; c < 4; ++c) w[c] = cells[32 * c + lane];
      }
      tmem_st4(tmem + lane_base + kColSfb + kSfbStride * st, w[0], w[1], w[2], w[3]);
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(&sf_full[st]);
    }
  } else {
    const int half = (warp - 1 - kScaleWarps) >> 2;  // this warp's 64 of the tile's 128 keys
    bool alive = true;
    for (int j = 0; j < ntiles; ++j) {
      const int buf = j & 1;
      if (alive) alive = mbar_wait_sleep(&acc_full[buf], (j >> 1) & 1, p.err);
      if (!alive) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      float v[64];
      tmem_ld32x2(tmem + lane_base + buf * kKeys + 64 * half, v);
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(&acc_empty[buf]);
      const int key0 = (kb0 + j) * kBlock + 64 * half;
      const bool whole = key0 + 64 <= L;  // every key of the 4 pages inside the row's causal length
      float pv[4];
#pragma unroll
      for (int pg = 0; pg < 4; ++pg) {
        float x[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) x[c] = (whole || key0 + 16 * pg + c < L) ? v[16 * pg + c] : -INFINITY;
        pv[pg] = max16(x);
      }
      if (row_ok) {
        const int pg0 = key0 / kPage;
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
  fill_neg_inf(p.scores, p.max_pages, tok0, tok1, (kb0 + ntiles) * kPagesPerSide, page_end);
}

}  // namespace

cudaError_t launch_index_score_prefill_mx(const PrefillScoreParams& p, cudaStream_t s) {
  CUtensorMap tq, tk;
  const uint64_t key_rows = static_cast<uint64_t>(p.num_blocks) * (p.block_stride / 64);
  if ((reinterpret_cast<uintptr_t>(p.idx_base) & 31) || p.block_stride % 64) return cudaErrorNotSupported;
  if (!make_map_u8(&tq, p.q, static_cast<uint64_t>(p.num_rows)) || !make_map_u4(&tk, p.idx_base, key_rows, kKeys))
    return cudaErrorInvalidValue;
  static std::atomic<uint64_t> configured{0};
  {
    const cudaError_t e = once_per_device(configured, [] {
      return cudaFuncSetAttribute(index_score_prefill_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (e != cudaSuccess) return e;
  }
  const int max_blocks = (p.max_pages + kPagesPerSide - 1) / kPagesPerSide;
  const dim3 grid(static_cast<unsigned>(p.max_tiles),
                  static_cast<unsigned>((max_blocks + kKeyBlocksPerCta - 1) / kKeyBlocksPerCta));
  const cudaError_t e = launch_kernel(index_score_prefill_mx_kernel, grid, dim3(kThreads), kSmemBytes, s, 0, tq, tk,
                                      p, static_cast<int32_t>(key_rows));
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

}  // namespace bsp
