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
// 64 key blocks, as the fp8 prefill scorer.  Warp 0, lane 0 is the producer
// and MMA issuer:
//   - the query tile (e4m3) by a 2-D TMA load with 128-byte swizzle;
//   - each half block of 64 keys by a 2-D TMA load of 4-bit data type
//     16U4_ALIGN16B (every 8 packed bytes of 16 e2m1 values unpacked into a
//     16-byte slot, the layout kind::f8f6f4 reads), 128-byte swizzle; its
//     64 x 4 e8m0 scales by a 1-D copy into one of two scale slots beside the
//     accumulator they belong to;
//   - four tcgen05.mma kind::f8f6f4 (A = queries, M = 128; B = keys, N = 64;
//     K = 32 = one scale group each) into four fp32 accumulators of 64 TMEM
//     columns, double-buffered (2 x 256 columns).
// Warps 1..8 are the epilogue: warp w reads TMEM lanes 32*(w%4).. (its
// quarter of the query rows) and half of the 64 keys, scales the four group
// sums of each key by its 2^(e-127) (decoded once per tile into shared
// memory by the epilogue warps together), masks keys at or past the row's
// causal length and max-pools 16 keys into a page score.
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
constexpr int kKeysPerTile = 64;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (1 + kEpiWarps);
constexpr int kAccCols = 4 * kKeysPerTile;  // four scale groups
constexpr int kQTile = 128 * 128;           // 128 query rows x 128 B
constexpr int kKeyTile = kKeysPerTile * 128;  // 64 keys x 128 padded bytes
constexpr uint32_t kKeyTx = kKeysPerTile * 64;  // the packed bytes the tensor load reads
constexpr uint32_t kIdesc = idesc_f8f6f4(kFmtE4m3, kFmtE2m1, kKeysPerTile, 128);
constexpr int kSmemUsed = 1024 /*align slack*/ + kQTile + kStages * kKeyTile + 2 * 256 /*e8m0*/ +
                          2 * 256 * 4 /*decoded scales*/ + 16 * 8 /*barriers*/ + 16;
// one CTA per SM: each holds all 512 TMEM columns, so a second resident CTA
// would only wait in tcgen05.alloc
constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;

struct SmemLayout {
  uint8_t* a;       // queries
  uint8_t* b;       // [stage][64 keys][128 B]
  uint8_t* e8;      // [2][64 keys][4] raw scales
  float* scales;    // [2][64 keys][4] decoded
  uint64_t* bars;   // a_full, b_full[S], b_empty[S], acc_full[2], acc_empty[2], scale_full[2]
  uint32_t* tmem_slot;
};

__device__ __forceinline__ SmemLayout carve(uint8_t* raw) {
  SmemLayout L;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  L.a = base;
  L.b = base + kQTile;
  L.e8 = L.b + kStages * kKeyTile;
  L.scales = reinterpret_cast<float*>(L.e8 + 2 * 256);
  L.bars = reinterpret_cast<uint64_t*>(L.scales + 2 * 256);
  L.tmem_slot = reinterpret_cast<uint32_t*>(L.bars + 16);
  return L;
}

// the epilogue warps' own barrier (named barrier 1, 256 threads)
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory"); }

__global__ void __launch_bounds__(kThreads, 1)
    index_score_prefill_mx_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                                  PrefillScoreParams p, int32_t oob_row) {
  extern __shared__ uint8_t smem_raw[];
  const SmemLayout sm = carve(smem_raw);
  uint64_t* a_full = sm.bars;
  uint64_t* b_full = sm.bars + 1;
  uint64_t* b_empty = sm.bars + 1 + kStages;
  uint64_t* acc_full = sm.bars + 1 + 2 * kStages;
  uint64_t* acc_empty = sm.bars + 3 + 2 * kStages;
  uint64_t* scale_full = sm.bars + 5 + 2 * kStages;
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
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 32 * kEpiWarps);
      mbar_init(&scale_full[i], 1);
    }
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
  const int ntiles = 2 * nb;  // half blocks of 64 keys
  const int page_end = min((kb0 + kKeyBlocksPerCta) * kPagesPerSide, p.max_pages);
  const int seq = s_seq;

  if (ntiles == 0) {
    if (row_ok && warp <= 4)
      for (int pg = kb0 * kPagesPerSide; pg < page_end; ++pg)
        p.scores[static_cast<int64_t>(tok) * p.max_pages + pg] = -INFINITY;
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

  if (warp == 0) {
    if (lane == 0) {
      // key tile j: keys 64*(j%2).. of block kb0 + j/2
      auto load_b = [&](int j) {
        const int st = j % kStages;
        const int bid = s_bid[j >> 1];
        const int r0 = bid < 0 ? oob_row
                               : static_cast<int>(static_cast<int64_t>(bid) * (p.block_stride / 64) +
                                                  (j & 1) * kKeysPerTile);
        mbar_arrive_expect_tx(&b_full[st], kKeyTx);
        tma_load_2d(sm.b + st * kKeyTile, &tmap_k, 0, r0, &b_full[st]);
      };
      bool alive = true;
      mbar_arrive_expect_tx(a_full, kQTile);
      tma_load_2d(sm.a, &tmap_q, 0, tok0, a_full);
      for (int j = 0; j < min(kStages, ntiles); ++j) load_b(j);
      alive = mbar_wait(a_full, 0, p.err);
      const uint32_t a_addr = smem_u32(sm.a);
      for (int j = 0; j < ntiles && alive; ++j) {
        const int st = j % kStages, buf = j & 1;
        alive = mbar_wait(&b_full[st], (j / kStages) & 1, p.err) &&
                mbar_wait(&acc_empty[buf], ((j >> 1) & 1) ^ 1, p.err);
        if (!alive) break;
        {  // the tile's e8m0 scales (64 keys x 4 B) into this buffer's slot
          const int bid = s_bid[j >> 1];
          fence_proxy_async();
          mbar_arrive_expect_tx(&scale_full[buf], bid >= 0 ? 256 : 0);
          if (bid >= 0)
            bulk_g2s(sm.e8 + buf * 256,
                     p.idx_base + static_cast<int64_t>(bid) * p.block_stride + kMxScaleOff + (j & 1) * 256, 256,
                     &scale_full[buf]);
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t b_addr = smem_u32(sm.b + st * kKeyTile);
#pragma unroll
        for (int g = 0; g < 4; ++g)
          umma_f8(tmem + buf * kAccCols + kKeysPerTile * g, smem_desc_sw128(a_addr + 32 * g),
                  smem_desc_sw128(b_addr + 32 * g), kIdesc, 0);
        umma_commit(&b_empty[st]);
        umma_commit(&acc_full[buf]);
        const int jp = j - 1;  // refill the previous tile's slot (its MMAs were issued an iteration ago)
        if (jp >= 0 && jp + kStages < ntiles) {
          alive = mbar_wait(&b_empty[jp % kStages], (jp / kStages) & 1, p.err);
          if (alive) load_b(jp + kStages);
        }
      }
      if (alive) mbar_wait(&b_empty[(ntiles - 1) % kStages], ((ntiles - 1) / kStages) & 1, p.err);
    }
    __syncwarp();
  } else {
    const int half = (warp - 1) >> 2;  // this warp's 32 of the tile's 64 keys
    const int et = tid - 32;           // 0..255 among the epilogue threads
    // every epilogue thread runs every iteration (the named barrier needs all
    // 256); after a timed-out wait a warp stops waiting and reading TMEM
    bool alive = true;
    for (int j = 0; j < ntiles; ++j) {
      const int buf = j & 1;
      if (alive) alive = __all_sync(0xffffffffu, mbar_wait(&scale_full[buf], (j >> 1) & 1, p.err));
      if (alive) {  // decode the tile's 256 scales once, shared by every row
        const uint8_t e = sm.e8[buf * 256 + et];
        sm.scales[buf * 256 + et] = e8m0_to_float(e);
      }
      epi_sync();  // the decoded scales, for every row; and buffer buf^1's readers are done
      if (alive) alive = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (j >> 1) & 1, p.err));
      if (!alive) continue;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + buf * kAccCols + 32 * half;
      float a0[32], a1[32], a2[32], a3[32];
      tmem_ld32(taddr, a0);
      tmem_ld32(taddr + kKeysPerTile, a1);
      tmem_ld32(taddr + 2 * kKeysPerTile, a2);
      tmem_ld32(taddr + 3 * kKeysPerTile, a3);
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(&acc_empty[buf]);
      const float4* sc = reinterpret_cast<const float4*>(sm.scales + buf * 256) + 32 * half;
      const int key0 = (kb0 + (j >> 1)) * kBlock + (j & 1) * kKeysPerTile + 32 * half;
      float pv[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float m = -INFINITY;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int k = 16 * hh + c;
          const float4 f = sc[k];
          float v = a0[k] * f.x;
          v = fmaf(a1[k], f.y, v);
          v = fmaf(a2[k], f.z, v);
          v = fmaf(a3[k], f.w, v);
          m = key0 + k < L ? fmaxf(m, v) : m;
        }
        pv[hh] = m;
      }
      if (row_ok) {
        const int pg0 = key0 / kPage;
        float* dst = p.scores + static_cast<int64_t>(tok) * p.max_pages + pg0;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          if (pg0 + hh < p.max_pages) dst[hh] = pv[hh];
      }
    }
    // pages of this key range that no tile covered
    if (row_ok && warp <= 4)
      for (int pg = (kb0 + nb) * kPagesPerSide; pg < page_end; ++pg)
        p.scores[static_cast<int64_t>(tok) * p.max_pages + pg] = -INFINITY;
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

}  // namespace

cudaError_t launch_index_score_prefill_mx(const PrefillScoreParams& p, cudaStream_t s) {
  CUtensorMap tq, tk;
  const uint64_t key_rows = static_cast<uint64_t>(p.num_blocks) * (p.block_stride / 64);
  if ((reinterpret_cast<uintptr_t>(p.idx_base) & 31) || p.block_stride % 64) return cudaErrorNotSupported;
  if (!make_map_u8(&tq, p.q, static_cast<uint64_t>(p.num_rows)) || !make_map_u4(&tk, p.idx_base, key_rows, 64))
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
