// index_score_mx_tc.cu -- a2 for MXFP4 index keys and e4m3 index queries on
// the 5th-generation tensor cores (ROCm/ATOM PR 2962, commit "... page-128
// block table": the MXFP4 decode scorer, its scores laid out as the other
// scorers').
//
//   S[t, n] = sum_G 2^(e[t, G] - 127) * sum_{d in group G} k[t, d] * q[n, d]
//   scores[row n, p] = max_{t in page p, t < L_n} S[t, n],  -inf past ceil(L_n/16)
//
// The same work units as the mma.sync decode scorer: one CTA per (query
// group, index head, chunk of 128-token blocks).  Warp 0, lane 0 is the
// producer and MMA issuer:
//   - each block's 128 x 128 e2m1 keys arrive by a 2-D TMA tensor load whose
//     4-bit data type unpacks every 8 packed bytes into a 16-byte slot
//     (8 bytes of 16 values, 8 unused), the layout the f8f6f4 MMA reads, with
//     128-byte swizzle; its 512 B of e8m0 scales follow by a 1-D copy into
//     one of two slots beside the accumulator they belong to;
//   - the group's query rows (at most 8, zero-padded to N = 16) are staged
//     once, by the other warps, in the same swizzled layout;
//   - tcgen05.mma kind::f8f6f4, A = keys (M = 128 tokens), B = queries
//     (N = 16), one MMA of K = 32 per 32-dim scale group into an accumulator
//     of its own (4 x 16 fp32 TMEM columns), double-buffered, so the MMAs of
//     the next block run under the epilogue of this one.
// Warps 1..4 are the epilogue: warp w reads TMEM lanes 32*(w%4).. (32
// tokens) with tcgen05.ld, applies the four e8m0 scales of its token to the
// group accumulators, masks tokens at or past each row's length and
// max-reduces 16 tokens (lanes) into a page score.
//
// Every wait is bounded; after a timed-out wait a role stops waiting (the
// error word is set) and the CTA frees its TMEM and returns.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace bsp {

namespace {

constexpr int kStages = 3;  // 53 KB of shared memory: 4 CTAs per SM
constexpr int kScaleSlots = kStages + 2;  // a block's scales live until its epilogue is done
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (1 + kEpiWarps);
constexpr int kN = 16;  // query columns: the group's rows, zero-padded
constexpr int kAccCols = 4 * kN;
constexpr int kKeyTile = 128 * 128;                      // shared bytes of one block's keys
constexpr uint32_t kKeyTx = 128 * 64;  // the transaction count: the packed bytes read, not the padded ones
constexpr uint32_t kIdesc = idesc_f8f6f4(kFmtE2m1, kFmtE4m3, kN, 128);
constexpr int kSmemBytes = 1024 /*align slack*/ + kStages * kKeyTile + kN * 128 /*queries*/ +
                           kScaleSlots * 512 /*scales*/ + 24 * 8 /*barriers*/ + 16;

struct SmemLayout {
  uint8_t* keys;    // [stage][128 rows][128 B]
  uint8_t* q;       // [16 rows][128 B]
  uint8_t* scales;  // [kScaleSlots][128 tokens][4]
  uint64_t* bars;   // full[S], empty[S], acc_full[2], acc_empty[2], scale_full[kScaleSlots]
  uint32_t* tmem_slot;
};

__device__ __forceinline__ SmemLayout carve(uint8_t* raw) {
  SmemLayout L;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  L.keys = base;
  L.q = base + kStages * kKeyTile;
  L.scales = L.q + kN * 128;
  L.bars = reinterpret_cast<uint64_t*>(L.scales + kScaleSlots * 512);
  L.tmem_slot = reinterpret_cast<uint32_t*>(L.bars + 24);
  return L;
}

__global__ void __launch_bounds__(kThreads, 1)
    index_score_mx_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, IndexScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  const SmemLayout sm = carve(smem_raw);
  uint64_t* full = sm.bars;
  uint64_t* empty = sm.bars + kStages;
  uint64_t* acc_full = sm.bars + 2 * kStages;
  uint64_t* acc_empty = sm.bars + 2 * kStages + 2;
  uint64_t* scale_full = sm.bars + 2 * kStages + 4;
  __shared__ int s_len[8], s_row[8];
  __shared__ int s_bid[32];  // the chunk's block ids (blocks_per_chunk <= 32)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int group = blockIdx.x / p.hidx, h = blockIdx.x % p.hidx;
  const int tok0 = group * p.q_group;
  const int ntok = min(p.q_group, p.num_tokens - tok0);
  const int max_len = p.max_pages * kPage;
  const int blk0 = blockIdx.y * p.blocks_per_chunk;

  pdl_wait();  // row lengths and the cast queries come from earlier kernels
  pdl_trigger();
  int32_t bid_early = 0;
  if (p.seq_is_group && tid < p.blocks_per_chunk && (blk0 + tid) * kPagesPerSide < p.max_pages)
    bid_early = p.block_table[static_cast<int64_t>(group) * p.bt_stride + blk0 + tid];
  if (tid < 8) {
    int L = 0, r = -1;
    if (tid < ntok) {
      r = (tok0 + tid) * p.hidx + h;
      L = min(max(p.row_len[r], 0), max_len);
      if (p.row_seq[r] != p.row_seq[tok0 * p.hidx + h]) set_err(p.err, BSP_DEVERR_GROUP_SEQ);
    }
    s_len[tid] = L;
    s_row[tid] = r;
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 32 * kEpiWarps);
    }
    for (int i = 0; i < kScaleSlots; ++i) mbar_init(&scale_full[i], 1);
    mbar_fence_init();
  }
  __syncthreads();

  int lmax = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) lmax = max(lmax, s_len[i]);
  const int seq = p.seq_is_group ? group : p.row_seq[tok0 * p.hidx + h];
  const int nb = max(0, min(p.blocks_per_chunk, (lmax + kBlock - 1) / kBlock - blk0));
  const int page_end = min((blk0 + p.blocks_per_chunk) * kPagesPerSide, p.max_pages);
  {  // pages of this chunk past every row's context: -inf
    const int pfirst = (blk0 + nb) * kPagesPerSide;
    const int npg = max(0, page_end - pfirst);
    for (int i = tid; i < ntok * npg; i += blockDim.x)
      p.scores[static_cast<int64_t>(s_row[i / npg]) * p.max_pages + pfirst + i % npg] = -INFINITY;
  }
  if (nb == 0) return;

  if (tid < nb) {
    int bid = p.seq_is_group ? bid_early : p.block_table[static_cast<int64_t>(seq) * p.bt_stride + blk0 + tid];
    if (bid < 0 || bid >= p.num_blocks) {
      set_err(p.err, BSP_DEVERR_BLOCK_ID);
      bid = 0;
    }
    s_bid[tid] = bid;
  }
  if (warp >= 1) {
    // the query tile: row n < ntok is row (tok0+n)*hidx + h of the e4m3
    // queries, the rest zero; 16-byte chunk j of row n sits at chunk
    // j ^ (n % 8) (128-byte swizzle)
    const int c = tid - 32;  // 0..127: 16 rows x 8 chunks
    const int n = c >> 3, j = c & 7;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < ntok)
      v = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.q) +
                                          (static_cast<int64_t>(tok0 + n) * p.hidx + h) * kDim + 16 * j);
    *reinterpret_cast<uint4*>(sm.q + n * 128 + ((j ^ (n & 7)) << 4)) = v;
    fence_proxy_async();  // the tensor core reads the tile through the async proxy
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;" ::"r"(smem_u32(sm.tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *sm.tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint8_t* field0 = p.idx_base + static_cast<int64_t>(h) * kMxField;
      // block i: its keys into ring slot i % S, its e8m0 scales into scale
      // slot i % (S+2) -- whose last user, block i-S-2, has finished its
      // epilogue once the MMAs of block i-S were issued
      auto load_block = [&](int i) {
        const int st = i % kStages, ss = i % kScaleSlots;
        const int64_t row = (static_cast<int64_t>(s_bid[i]) * p.block_stride + static_cast<int64_t>(h) * kMxField) / 64;
        mbar_arrive_expect_tx(&full[st], kKeyTx);
        tma_load_2d(sm.keys + st * kKeyTile, &tmap_k, 0, static_cast<int>(row), &full[st]);
        fence_proxy_async();  // the epilogue's reads of the slot's previous scales
        mbar_arrive_expect_tx(&scale_full[ss], 512);
        bulk_g2s(sm.scales + ss * 512, field0 + static_cast<int64_t>(s_bid[i]) * p.block_stride + kMxScaleOff, 512,
                 &scale_full[ss]);
      };
      bool alive = true;
      for (int i = 0; i < min(kStages, nb); ++i) load_block(i);
      const uint32_t q_addr = smem_u32(sm.q);
      for (int i = 0; i < nb && alive; ++i) {
        const int st = i % kStages, buf = i & 1;
        alive = mbar_wait_sleep(&full[st], (i / kStages) & 1, p.err) &&
                mbar_wait_sleep(&acc_empty[buf], ((i >> 1) & 1) ^ 1, p.err);
        if (!alive) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t k_addr = smem_u32(sm.keys + st * kKeyTile);
#pragma unroll
        for (int g = 0; g < 4; ++g)
          umma_f8(tmem + buf * kAccCols + kN * g, smem_desc_sw128(k_addr + 32 * g), smem_desc_sw128(q_addr + 32 * g),
                  kIdesc, 0);
        umma_commit(&empty[st]);
        umma_commit(&acc_full[buf]);
        // refill the previous block's slot: its MMAs were issued an iteration
        // ago, so this wait overlaps the ones just issued
        const int j = i - 1;
        if (j >= 0 && j + kStages < nb) {
          alive = mbar_wait_sleep(&empty[j % kStages], (j / kStages) & 1, p.err);
          if (alive) load_block(j + kStages);
        }
      }
      // nothing may still be writing shared memory or TMEM when the CTA
      // leaves: wait (bounded) for the last MMAs
      if (alive && nb > 0) mbar_wait_sleep(&empty[(nb - 1) % kStages], ((nb - 1) / kStages) & 1, p.err);
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    const int t = 32 * quarter + lane;  // this thread's token of the block
    bool alive = true;
    for (int i = 0; i < nb && alive; ++i) {
      const int buf = i & 1;
      const int ss = i % kScaleSlots;
      alive = mbar_wait_sleep(&scale_full[ss], (i / kScaleSlots) & 1, p.err) &&
              mbar_wait_sleep(&acc_full[buf], (i >> 1) & 1, p.err);
      alive = __all_sync(0xffffffffu, alive);  // tcgen05.ld below is warp-wide
      if (!alive) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + buf * kAccCols;
      float a[4][8];
      tmem_ld8x4(taddr, kN, a);  // each group's first 8 query columns
      const uint32_t sc = *reinterpret_cast<const uint32_t*>(sm.scales + ss * 512 + 4 * t);
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(&acc_empty[buf]);
      float f[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) f[g] = e8m0_to_float((sc >> (8 * g)) & 0xFF);
      const int pos = (blk0 + i) * kBlock + t;
      const int page = (blk0 + i) * kPagesPerSide + (t >> 4);
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        if (n >= ntok) break;  // warp-uniform
        float v = a[0][n] * f[0];
        v = fmaf(a[1][n], f[1], v);
        v = fmaf(a[2][n], f[2], v);
        v = fmaf(a[3][n], f[3], v);
        float m = pos < s_len[n] ? v : -INFINITY;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((lane & 15) == 0 && page < p.max_pages)
          p.scores[static_cast<int64_t>(s_row[n]) * p.max_pages + page] =
              page < (s_len[n] + kPage - 1) / kPage ? m : -INFINITY;
      }
    }
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;" ::"r"(tmem));
  }
}

}  // namespace

bool index_score_mx_tc_supported(const IndexScoreParams& p) {
  return p.idx_dtype == BSP_MXFP4 && p.q_dtype == BSP_FP8_E4M3 && p.q_group <= 8 &&
         (reinterpret_cast<uintptr_t>(p.idx_base) & 31) == 0 && p.block_stride % 64 == 0 &&
         (reinterpret_cast<uintptr_t>(p.q) & 15) == 0;
}

int index_score_mx_tc_occupancy() {
  static std::atomic<int> table[kMaxDevices];
  return cached_per_device(table, [] {
    int v = 0;
    if (cudaFuncSetAttribute(index_score_mx_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, index_score_mx_tc_kernel, kThreads, kSmemBytes) !=
            cudaSuccess)
      v = 1;
    return std::max(1, std::min(v, 512 / (2 * kAccCols)));  // TMEM: 128 columns a CTA
  });
}

cudaError_t launch_index_score_mx_tc(const IndexScoreParams& p, dim3 grid, cudaStream_t s) {
  CUtensorMap tk;
  const uint64_t rows = static_cast<uint64_t>(p.num_blocks) * (p.block_stride / 64);
  if (!make_map_u4(&tk, p.idx_base, rows, 128)) return cudaErrorInvalidValue;
  index_score_mx_tc_occupancy();  // the shared-memory opt-in
  const cudaError_t e = launch_kernel(index_score_mx_tc_kernel, grid, dim3(kThreads), kSmemBytes, s, 0, tk, p);
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

}  // namespace bsp
