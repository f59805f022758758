// index_score.cu -- a2: page scores of the index query against the index-key
// cache (ROCm/ATOM PR 2962, commit "... page-128 block table": fp32 scores of
// each row over its context, -inf where nothing is scored; "Known limits":
// the scorer runs at the score workspace's full width).
//
//   scores[r, p] = max_{t in page p, t < L_r} sum_d q[r, d] * k[t, d]
//   scores[r, p] = -inf for p >= ceil(L_r / 16)
//
// Work unit: one CTA per (query group, index head, chunk of 128-token
// blocks).  A query group is q_group consecutive tokens of one sequence (the
// decode query length), so the index cache of a sequence is read once per
// group.  The chunk length is planned from the kernel's occupancy, trading
// each CTA's fixed start against the grid's tail.  Thread 0 streams whole
// index fields (16896 B fp8, 32768 B bf16, 8704 B MXFP4 per block and head)
// into a shared-memory ring with 1-D TMA bulk copies completing on
// mbarriers; the four warps each score 32 tokens of a block (two 16-token
// pages) on the tensor cores:
//   A = 16 keys x 16 dims (fp8 -> f16 exactly, e2m1 -> f16 exactly, or bf16),
//   B = 16 dims x 8 query rows (the group's rows; unused columns are zero),
//   C = fp32.
// fp8 keys with an e4m3 query run on the fp8 mma (m16n8k32 e4m3 x e4m3 ->
// f32) straight from the cached bytes.  The dims of each mma are a
// permutation of the real dims chosen so that every thread reads 16-byte (or
// 4-byte) runs of a key row; A and B use the same permutation, so each dot
// product is unchanged.  The per-token fp8 scale and the per-32-dim e8m0
// scales are applied to the fp32 partial sums, then the page max is a shuffle
// reduction over the 16 tokens of the tile.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "topk_row.cuh"

namespace bsp {

namespace {

// Per format: the index field of one block and head, a key row's bytes,
// where the per-token scales start in the field (0: none), and the deepest
// ring the plan may give a CTA.
template <int KEY>
struct KeyFmt;
template <>
struct KeyFmt<BSP_BF16> {
  static constexpr int kField = kBf16IndexField, kRow = 2 * kDim, kScaleOff = 0;
  static constexpr int kStages = 3;
};
// fp8 rings stop at 2 fields (6 CTAs per SM): with 3 or 4 (4 or 3 CTAs per
// SM) the mma work of a block no longer hides behind the copies (measured
// 117 us against 92 on the 32k-token batch)
template <>
struct KeyFmt<BSP_FP8_E4M3> {
  static constexpr int kField = kFp8IndexField, kRow = kDim, kScaleOff = kFp8IndexScaleOff;
  static constexpr int kStages = 2;
};
template <>
struct KeyFmt<BSP_MXFP4> {
  static constexpr int kField = kMxField, kRow = kDim / 2, kScaleOff = kMxScaleOff;
  static constexpr int kStages = 6;
};
// fp8 keys scored against an e4m3 query: the fp8 mma takes the cached bytes
// as they are (no conversion)
constexpr int kFp8KeysE4m3Q = 3;
template <>
struct KeyFmt<kFp8KeysE4m3Q> {
  static constexpr int kField = kFp8IndexField, kRow = kDim, kScaleOff = kFp8IndexScaleOff;
  static constexpr int kStages = 2;
};
template <int KEY>
constexpr int smem_bytes(int stages) {
  return stages * KeyFmt<KEY>::kField + stages * 8;
}

// first of the four real dims that B fragment m of thread t covers
template <int KEY>
__device__ __forceinline__ int frag_dim(int m, int t) {
  if (KEY == BSP_FP8_E4M3) return 16 * (t + 4 * (m >> 2)) + 4 * (m & 3);
  if (KEY == BSP_MXFP4) return 32 * (m >> 1) + 8 * t + 4 * (m & 1);
  return 8 * (t + 4 * (m >> 1)) + 4 * (m & 1);
}

__device__ __forceinline__ void load_q4(const void* q, int q_dtype, int64_t off, float (&v)[4]) {
  if (q_dtype == BSP_BF16) {
    const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(q) + off);
    v[0] = bf16_bits_to_float(w.x & 0xFFFF);
    v[1] = bf16_bits_to_float(w.x >> 16);
    v[2] = bf16_bits_to_float(w.y & 0xFFFF);
    v[3] = bf16_bits_to_float(w.y >> 16);
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(q) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = e4m3_to_float(w >> (8 * i));
  }
}

// B fragments of the group's query rows tok0 .. tok0+ntok-1 (index head h):
// thread (g, t) holds row g's dims in the permutation frag_dim / the fp8 mma
// uses; columns past the group are zero.
template <int KEY>
__device__ __forceinline__ void load_qb(const IndexScoreParams& p, int tok0, int ntok, int h, int g, int t,
                                        uint32_t (&qb)[8][2]) {
  if (KEY == kFp8KeysE4m3Q) {
    // mma m (< 4): this thread's 16-dim chunk c = t + 4*(m/2), dims 8*(m%2) + 0..7
    const uint8_t* qrow = static_cast<const uint8_t*>(p.q) + (static_cast<int64_t>(tok0 + g) * p.hidx + h) * kDim;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int d = 16 * (t + 4 * (m >> 1)) + 8 * (m & 1);
      qb[m][0] = g < ntok ? *reinterpret_cast<const uint32_t*>(qrow + d) : 0u;
      qb[m][1] = g < ntok ? *reinterpret_cast<const uint32_t*>(qrow + d + 4) : 0u;
    }
  }
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    if (KEY == kFp8KeysE4m3Q) break;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (g < ntok) load_q4(p.q, p.q_dtype, (static_cast<int64_t>(tok0 + g) * p.hidx + h) * kDim + frag_dim<KEY>(m, t), v);
    if (KEY == BSP_BF16) {
      qb[m][0] = pack_bf16x2(v[0], v[1]);
      qb[m][1] = pack_bf16x2(v[2], v[3]);
    } else {
      qb[m][0] = pack_f16x2(v[0], v[1]);
      qb[m][1] = pack_f16x2(v[2], v[3]);
    }
  }
}

// Scores of one 16-key tile against the group's query columns (mma C
// layout): v0 / v1 for key g and query rows 2t / 2t+1, v2 / v3 for key g+8.
// `rows` is the shared-memory address of the tile's first key row, `scales`
// of its first per-key scale (fp8 and MXFP4 fields).
template <int KEY>
__device__ __forceinline__ void tile_scores(uint32_t rows, uint32_t scales, const uint32_t (&qb)[8][2], int g, int t,
                                            float& v0, float& v1, float& v2, float& v3) {
  if (KEY == kFp8KeysE4m3Q) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t ra_row = rows + g * 128, rb_row = ra_row + 8 * 128;
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
      const uint4 ra = lds128(ra_row + 16 * (t + 4 * ii));
      const uint4 rb = lds128(rb_row + 16 * (t + 4 * ii));
      mma_e4m3(acc, ra.x, rb.x, ra.y, rb.y, qb[2 * ii][0], qb[2 * ii][1]);
      mma_e4m3(acc, ra.z, rb.z, ra.w, rb.w, qb[2 * ii + 1][0], qb[2 * ii + 1][1]);
    }
    const float sg = __uint_as_float(lds32(scales + g * 4));
    const float sg8 = __uint_as_float(lds32(scales + (g + 8) * 4));
    v0 = acc[0] * sg, v1 = acc[1] * sg, v2 = acc[2] * sg8, v3 = acc[3] * sg8;
  } else if (KEY == BSP_FP8_E4M3) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t ra_row = rows + g * 128, rb_row = ra_row + 8 * 128;
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
      const uint4 ra = lds128(ra_row + 16 * (t + 4 * ii));
      const uint4 rb = lds128(rb_row + 16 * (t + 4 * ii));
      const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2_scaled(wa[j], a0, a2);
        e4m3x4_to_f16x2_scaled(wb[j], a1, a3);
        mma_f16(acc, a0, a1, a2, a3, qb[4 * ii + j][0], qb[4 * ii + j][1]);
      }
    }
    // per-token scale; the f16 keys hold value * 2^-8
    const float sg = __uint_as_float(lds32(scales + g * 4)) * 256.f;
    const float sg8 = __uint_as_float(lds32(scales + (g + 8) * 4)) * 256.f;
    v0 = acc[0] * sg, v1 = acc[1] * sg, v2 = acc[2] * sg8, v3 = acc[3] * sg8;
  } else if (KEY == BSP_MXFP4) {
    float acc[4][4];
#pragma unroll
    for (int G = 0; G < 4; ++G) acc[G][0] = acc[G][1] = acc[G][2] = acc[G][3] = 0.f;
    const uint32_t ra_row = rows + g * 64, rb_row = ra_row + 8 * 64;
#pragma unroll
    for (int G = 0; G < 4; ++G) {
      const uint32_t wa = lds32(ra_row + 16 * G + 4 * t), wb = lds32(rb_row + 16 * G + 4 * t);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t a0 = e2m1x2_to_f16x2((wa >> (16 * hh)) & 0xFF);
        const uint32_t a2 = e2m1x2_to_f16x2((wa >> (16 * hh + 8)) & 0xFF);
        const uint32_t a1 = e2m1x2_to_f16x2((wb >> (16 * hh)) & 0xFF);
        const uint32_t a3 = e2m1x2_to_f16x2((wb >> (16 * hh + 8)) & 0xFF);
        mma_f16(acc[G], a0, a1, a2, a3, qb[2 * G + hh][0], qb[2 * G + hh][1]);
      }
    }
    const uint32_t sa = lds32(scales + g * 4);
    const uint32_t sb = lds32(scales + (g + 8) * 4);
    v0 = v1 = v2 = v3 = 0.f;
#pragma unroll
    for (int G = 0; G < 4; ++G) {
      const float ca = e8m0_to_float((sa >> (8 * G)) & 0xFF), cb = e8m0_to_float((sb >> (8 * G)) & 0xFF);
      v0 = fmaf(acc[G][0], ca, v0);
      v1 = fmaf(acc[G][1], ca, v1);
      v2 = fmaf(acc[G][2], cb, v2);
      v3 = fmaf(acc[G][3], cb, v3);
    }
  } else {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t ra_row = rows + g * 256, rb_row = ra_row + 8 * 256;
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const uint4 ra = lds128(ra_row + 16 * (t + 4 * ii));
      const uint4 rb = lds128(rb_row + 16 * (t + 4 * ii));
      mma_bf16(acc, ra.x, rb.x, ra.y, rb.y, qb[2 * ii][0], qb[2 * ii][1]);
      mma_bf16(acc, ra.z, rb.z, ra.w, rb.w, qb[2 * ii + 1][0], qb[2 * ii + 1][1]);
    }
    v0 = acc[0], v1 = acc[1], v2 = acc[2], v3 = acc[3];
  }
}

// The selection tail of the decode step's scorer: every CTA of a (query
// group, index head) unit has written its chunk's scores; the last one to
// finish -- an arrival count per unit -- reads the unit's score rows back
// through L2 and selects each row (select_row_cta with 128 threads, SEL
// pages a thread), then zeroes the count for the next step.  The ring is
// idle by then and holds the histograms.
template <int SEL>
__device__ __forceinline__ void select_unit(const IndexScoreParams& p, const int* s_row, int ntok, uint8_t* smem) {
  __shared__ int s_last;
  __threadfence();  // this thread's score stores, before the count
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&p.sel_counters[blockIdx.x], 1) == static_cast<int>(gridDim.y) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();  // the other CTAs' scores, after the count
  auto& hist = *reinterpret_cast<int(*)[4][256]>(smem);
  int* s_warp = reinterpret_cast<int*>(smem + 4096);
  uint32_t& s_digit = *reinterpret_cast<uint32_t*>(smem + 4096 + 16);
  int& s_above = *reinterpret_cast<int*>(smem + 4096 + 20);
  for (int j = 0; j < ntok; ++j) {
    for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x) (&hist[0][0])[i] = 0;
    select_row_cta<SEL, 128, true>(p.sel, s_row[j], hist, s_warp, s_digit, s_above, false);
    __syncthreads();  // the next row reuses the histograms and the scan slots
  }
  if (threadIdx.x == 0) p.sel_counters[blockIdx.x] = 0;
}

template <int KEY, int SEL>
__global__ void __launch_bounds__(128) index_score_kernel(IndexScoreParams p) {
  constexpr int FB = KeyFmt<KEY>::kField;
  const int S = p.stages;  // ring depth, 1..kStages
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * FB);
  __shared__ int s_len[8], s_row[8], s_seq;
  __shared__ int s_bid[32];  // the chunk's block ids (blocks_per_chunk <= 32)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int group = blockIdx.x / p.hidx, h = blockIdx.x % p.hidx;
  const int chunk = blockIdx.y;
  const int tok0 = group * p.q_group;
  const int ntok = min(p.q_group, p.num_tokens - tok0);
  const int max_len = p.max_pages * kPage;
  const int blk0 = chunk * p.blocks_per_chunk;

  pdl_wait();  // row lengths come from the kernel before
  pdl_trigger();
  // decode-ordered rows: the chunk's block ids load alongside the rows'
  // lengths instead of after them (entries past the context go unused)
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
    s_seq = p.seq_is_group ? group : p.row_seq[tok0 * p.hidx + h];
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
  __syncthreads();

  int lmax = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) lmax = max(lmax, s_len[i]);
  const int seq = s_seq;
  const int nb = max(0, min(p.blocks_per_chunk, (lmax + kBlock - 1) / kBlock - blk0));
  const int page_end = min((blk0 + p.blocks_per_chunk) * kPagesPerSide, p.max_pages);

  // pages of this chunk past every row's context: -inf
  {
    const int pfirst = (blk0 + nb) * kPagesPerSide;
    const int npg = max(0, page_end - pfirst);
    for (int i = tid; i < ntok * npg; i += blockDim.x)
      p.scores[static_cast<int64_t>(s_row[i / npg]) * p.max_pages + pfirst + i % npg] = -INFINITY;
  }
  if (nb > 0) {
  if (tid < nb) {
    int bid = p.seq_is_group ? bid_early : p.block_table[static_cast<int64_t>(seq) * p.bt_stride + blk0 + tid];
    if (bid < 0 || bid >= p.num_blocks) {
      set_err(p.err, BSP_DEVERR_BLOCK_ID);
      bid = 0;
    }
    s_bid[tid] = bid;
  }
  __syncthreads();

  auto issue = [&](int i) {
    const int bid = s_bid[i];
    const int st = i % S;
    mbar_arrive_expect_tx(&bars[st], FB);
    bulk_g2s(smem + st * FB, p.idx_base + static_cast<int64_t>(bid) * p.block_stride + static_cast<int64_t>(h) * FB,
             FB, &bars[st]);
  };
  if (tid == 0)
    for (int i = 0; i < min(S, nb); ++i) issue(i);

  // B fragments: query row g of the group (zero beyond the group)
  uint32_t qb[8][2];
  load_qb<KEY>(p, tok0, ntok, h, g, t, qb);
  const int len_lo = s_len[min(2 * t, 7)], len_hi = s_len[min(2 * t + 1, 7)];

  for (int i = 0; i < nb; ++i) {
    const int st = i % S;
    mbar_wait(&bars[st], (i / S) & 1, p.err);
    const uint32_t sbase = smem_u32(smem + st * FB);
    const int blk_pos = (blk0 + i) * kBlock;
#pragma unroll
    for (int tile = 0; tile < 2; ++tile) {
      const int tokb = 32 * warp + 16 * tile;
      float v0, v1, v2, v3;
      tile_scores<KEY>(sbase + tokb * KeyFmt<KEY>::kRow, sbase + KeyFmt<KEY>::kScaleOff + tokb * 4, qb, g, t, v0, v1, v2,
                       v3);
      // mask tokens past each row's length, then the page max over 16 tokens
      const int pos = blk_pos + tokb + g;
      float m_lo = fmaxf(pos < len_lo ? v0 : -INFINITY, pos + 8 < len_lo ? v2 : -INFINITY);
      float m_hi = fmaxf(pos < len_hi ? v1 : -INFINITY, pos + 8 < len_hi ? v3 : -INFINITY);
#pragma unroll
      for (int m = 4; m < 32; m <<= 1) {
        m_lo = fmaxf(m_lo, __shfl_xor_sync(0xffffffffu, m_lo, m));
        m_hi = fmaxf(m_hi, __shfl_xor_sync(0xffffffffu, m_hi, m));
      }
      const int page = (blk0 + i) * kPagesPerSide + 2 * warp + tile;
      if (g == 0 && page < p.max_pages) {
        if (2 * t < ntok)
          p.scores[static_cast<int64_t>(s_row[2 * t]) * p.max_pages + page] =
              page < (len_lo + kPage - 1) / kPage ? m_lo : -INFINITY;
        if (2 * t + 1 < ntok)
          p.scores[static_cast<int64_t>(s_row[2 * t + 1]) * p.max_pages + page] =
              page < (len_hi + kPage - 1) / kPage ? m_hi : -INFINITY;
      }
    }
    __syncthreads();
    if (tid == 0 && i + S < nb) {
      fence_proxy_async();
      issue(i + S);
    }
  }
  }  // nb > 0
  if constexpr (SEL > 0) select_unit<SEL>(p, s_row, ntok, smem);
}

// the dynamic shared-memory opt-in (once per device; per function)
template <int KEY, int SEL>
cudaError_t configure_key() {
  static std::atomic<uint64_t> done{0};
  return once_per_device(done, [] {
    return cudaFuncSetAttribute(index_score_kernel<KEY, SEL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_bytes<KEY>(KeyFmt<KEY>::kStages));
  });
}

// resident CTAs per SM with a ring of `stages` fields (queried once per depth;
// a failed query assumes 1)
template <int KEY, int SEL>
int occupancy_key(int stages) {
  static std::atomic<int> cache[KeyFmt<KEY>::kStages + 1][kMaxDevices];
  return cached_per_device(cache[stages], [stages] {
    int n = 0;
    cudaError_t e = configure_key<KEY, SEL>();
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, index_score_kernel<KEY, SEL>, 128,
                                                        smem_bytes<KEY>(stages));
    return (e == cudaSuccess && n > 0) ? n : 1;
  });
}

// Blocks per CTA (cb) and ring depth.  With W blocks per SM and `occ`
// resident CTAs per SM sharing its bandwidth, the plan minimises
//   W * (1 + s / cb) + occ * cb / 2
// over cb = 1..32: every CTA pays a fixed start (row lengths, block ids, the
// first copy) worth about s blocks of streaming, and the grid ends in a tail
// of about half a CTA, whose blocks each take occ block-times.  s is a time
// (kStartBytes of streaming), so it is worth more of the small MXFP4 fields
// than of the fp8 ones.  The ring holds min(cb, kStages) fields.  On a
// 128-sequence, 32k-token batch (256 fp8 blocks per sequence) this picks
// cb = 6: measured 91.8 us, against 92.3 at cb = 4, 93.6 at 8, 92.8 at 12,
// 101.5 at 16 and 96.5 at 2 (the wave-count plan before it).
constexpr double kStartBytes = 0.5 * kFp8IndexField;

template <int KEY, int SEL>
void plan_key(IndexScoreParams& p, int64_t max_blocks, int num_sms) {
  const double W = static_cast<double>(p.num_groups) * p.hidx * max_blocks / num_sms;
  const double s = kStartBytes / KeyFmt<KEY>::kField;
  double best = 0.0;
  for (int cb = 1; cb <= 32; ++cb) {
    const int stages = std::min(cb, KeyFmt<KEY>::kStages);
    const double occ = occupancy_key<KEY, SEL>(stages);
    const double cost = W * (1.0 + s / cb) + occ * cb / 2.0;
    if (cb == 1 || cost < best) {
      best = cost;
      p.blocks_per_chunk = cb;
      p.stages = stages;
    }
    if (cb >= max_blocks) break;
  }
}

template <int KEY, int SEL>
cudaError_t launch_key(IndexScoreParams p, int64_t max_blocks, int num_sms, cudaStream_t s) {
  plan_key<KEY, SEL>(p, max_blocks, num_sms);
  const cudaError_t c = configure_key<KEY, SEL>();
  if (c != cudaSuccess) return c;
  const int64_t cb = p.blocks_per_chunk;
  const dim3 grid(static_cast<unsigned>(p.num_groups * p.hidx), static_cast<unsigned>((max_blocks + cb - 1) / cb));
  const cudaError_t e =
      launch_kernel(index_score_kernel<KEY, SEL>, grid, dim3(128), smem_bytes<KEY>(p.stages), s, 0, p);
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

// the fused selection's pages per thread (128 threads); 0: not fused
int select_width(int32_t idx_dtype, int32_t q_dtype, int32_t max_pages, int32_t blocks) {
  if (idx_dtype != BSP_FP8_E4M3 || q_dtype != BSP_FP8_E4M3 || blocks) return 0;
  for (int w = 4; w <= 32; w *= 2)
    if (max_pages <= 128 * w) return w;
  return 0;
}

}  // namespace

bool index_score_can_select(int32_t idx_dtype, int32_t q_dtype, int32_t max_pages, int32_t blocks) {
  return select_width(idx_dtype, q_dtype, max_pages, blocks) != 0;
}

// MXFP4 keys with e4m3 queries on tcgen05: the same chunk grid, planned with
// that kernel's occupancy and a 4-deep ring.  Its plan counts whole waves of
// resident CTAs, each costing (cb + s) block-times, with s the time of
// streaming 1.5 fp8 fields.
void plan_mx_tc(IndexScoreParams& p, int64_t max_blocks, int num_sms) {
  const int64_t units = static_cast<int64_t>(p.num_groups) * p.hidx;
  const double start_blocks = 1.5 * kFp8IndexField / kMxField;
  const int64_t resident = static_cast<int64_t>(index_score_mx_tc_occupancy()) * num_sms;
  double best = 0.0;
  for (int cb = 1; cb <= 32; ++cb) {
    const int64_t ctas = units * ((max_blocks + cb - 1) / cb);
    const int64_t waves = (ctas + resident - 1) / resident;
    const double cost = static_cast<double>(waves) * (cb + start_blocks);
    if (cb == 1 || cost < best) {
      best = cost;
      p.blocks_per_chunk = cb;
      p.stages = 4;
    }
    if (cb >= max_blocks) break;
  }
}

cudaError_t launch_index_score(IndexScoreParams p, int num_sms, cudaStream_t s) {
  if (p.num_rows == 0 || p.max_pages == 0) return cudaSuccess;
  p.num_groups = (p.num_tokens + p.q_group - 1) / p.q_group;
  const int64_t max_blocks = (p.max_pages + kPagesPerSide - 1) / kPagesPerSide;
  if (!p.sel_counters && index_score_mx_tc_supported(p)) {
    plan_mx_tc(p, max_blocks, num_sms);
    const int64_t cb = p.blocks_per_chunk;
    return launch_index_score_mx_tc(
        p, dim3(static_cast<unsigned>(p.num_groups * p.hidx), static_cast<unsigned>((max_blocks + cb - 1) / cb)), s);
  }
  const int sel = p.sel_counters ? select_width(p.idx_dtype, p.q_dtype, p.max_pages, p.sel.blocks) : 0;
  if (p.sel_counters && !sel) return cudaErrorInvalidValue;  // the caller checks index_score_can_select
  switch (p.idx_dtype) {
    case BSP_BF16:
      return launch_key<BSP_BF16, 0>(p, max_blocks, num_sms, s);
    case BSP_FP8_E4M3:
      if (p.q_dtype != BSP_FP8_E4M3) return launch_key<BSP_FP8_E4M3, 0>(p, max_blocks, num_sms, s);
      switch (sel) {
        case 4:
          return launch_key<kFp8KeysE4m3Q, 4>(p, max_blocks, num_sms, s);
        case 8:
          return launch_key<kFp8KeysE4m3Q, 8>(p, max_blocks, num_sms, s);
        case 16:
          return launch_key<kFp8KeysE4m3Q, 16>(p, max_blocks, num_sms, s);
        case 32:
          return launch_key<kFp8KeysE4m3Q, 32>(p, max_blocks, num_sms, s);
        default:
          return launch_key<kFp8KeysE4m3Q, 0>(p, max_blocks, num_sms, s);
      }
    default:
      return launch_key<BSP_MXFP4, 0>(p, max_blocks, num_sms, s);
  }
}

}  // namespace bsp
