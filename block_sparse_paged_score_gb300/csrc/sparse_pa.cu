// sparse_pa.cu -- a4/a5: attention of each row over the tokens its sparse
// block table selects (vLLM API docs of MiniMaxM3SparseAiterPAImpl.forward:
// decode and prefill attend through sparse_block_table / sparse_context_lens;
// vLLM PR 61889, Details: one page id addresses K and V; ROCm/ATOM PR 2962:
// MXFP4 K/V with an e4m3 query, one row per (token, KV head), prefill
// plan-free with one direct write per row).
//
// Row r = token*Hkv + h attends its G query heads (G <= 16 fill the M=16 rows
// of an mma tile; unused rows are zero) over tokens m < sparse_ctx[r]; token
// m is token m%16 of page sparse_bt[r, m/16].
//
// CTA = 4 warps = one (row, split); a split is a run of pages and warp w
// takes pages w, w+4, ... of it.  Each warp streams its pages through a ring
// of shared-memory slots with 1-D TMA bulk copies (K page + V page of its
// head; MXFP4: the 1 KB data and 64 B scales of both sides) completing on
// mbarriers, and keeps its own online softmax.  Per 16-token page:
//   S  = Q Kt : 2 n-tiles (8 tokens) x 8 k-steps of mma.sync m16n8k16
//   P  = 2^(S*scale - m)     (log2 domain, running max m and sum l per head;
//                             the hardware ex2.approx)
//   O += P V  : 16 n-tiles (8 dims) of mma.sync m16n8k16
// The Q fragments sit in shared memory (loaded once per CTA), which keeps the
// fp8 kernel within 128 registers: four CTAs (16 warps) per SM.  fp8 pages
// are converted to f16 in registers right after ldmatrix (exact; the k/v
// scales are folded into the softmax scale and the output scale).  For fp8
// the 16 tokens of a page enter the mma in the order 0,1,4,5,8,9,12,13 |
// 2,3,6,7,... so that the S accumulator lands as the P fragment whose tokens
// match the V rows a ldmatrix of the dim-major V page hands each thread
// (tokens 4t..4t+3); bf16 pages use the natural order.  MXFP4 pages are
// dequantised by the warp into a bf16 page (e2m1 * 2^(e-127) is exact in
// bf16) and then take the bf16 path.
//
// The 4 warps merge in shared memory (log-sum-exp).  A row with one split is
// written directly; 2..8 splits form a thread-block cluster and merge through
// distributed shared memory; more splits (very few rows) publish (m, l, O) to
// the workspace and the last CTA of the row to arrive merges them.  The plan
// splits rows only as far as one wave of resident CTAs needs, and deepens the
// per-warp ring (a launch parameter) when the grid leaves room for it.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace bsp {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// fp8 -> f16 of the K/V pages with the hardware cvt (exact)
__device__ __forceinline__ void kv_e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  e4m3x4_to_f16x2_cvt(w, lo, hi);
}
constexpr float kRescaleLog2 = 8.f;

template <int KV>
struct PaFmt;
constexpr int kMaxCluster = 8;  // portable thread-block cluster size

// Per format: kRing, the default pages in flight per warp (the plan deepens
// it up to kRingMax while the grid fits one wave); kSlot, the bytes of one
// page of K and V; kDeq, the bf16 page a warp dequantises MXFP4 into;
// kMinCtas, the resident CTAs per SM the kernel is compiled for (its register
// budget: fp8 fits four, 16 warps per SM, with a 3-page ring; MXFP4 fits
// four with a 2-page ring, the most its dequant pages leave room for).  All
// measured.
template <>
struct PaFmt<BSP_FP8_E4M3> {
  static constexpr int kRing = 3, kRingMax = 6, kSlot = 4096, kDeq = 0, kMinCtas = 4;
};
template <>
struct PaFmt<BSP_BF16> {
  static constexpr int kRing = 2, kRingMax = 4, kSlot = 8192, kDeq = 0, kMinCtas = 2;
};
template <>
struct PaFmt<BSP_MXFP4> {
  // K data 1024 | K scales 64 | V data 1024 | V scales 64
  static constexpr int kRing = 2, kRingMax = 6, kSlot = 2176, kDeq = 8192, kMinCtas = 4;
};

// shared memory: the rings (and MXFP4 dequant pages) during the page loop,
// reused after it for the four warps' merge ([4][16] m, [4][16] l,
// [4][16][136] O); the mbarriers sit after the larger of the two
constexpr int kCombineFloats = 128 + 4 * 16 * (128 + 8);
// plus this CTA's partial (m[16], l[16], O[16][128]) that cluster peers read
constexpr int kCombineBytes = (kCombineFloats + 32 + 16 * 128) * 4;
template <int KV>
__host__ __device__ constexpr int pa_bar_offset(int ring) {
  return (4 * ring * PaFmt<KV>::kSlot + 4 * PaFmt<KV>::kDeq) > kCombineBytes
             ? 4 * ring * PaFmt<KV>::kSlot + 4 * PaFmt<KV>::kDeq
             : kCombineBytes;
}
// the row's Q fragments (4 KB) follow the ring / merge area, then the mbarriers
constexpr int kQFragBytes = 8 * 32 * 16;
template <int KV>
__host__ __device__ constexpr int pa_smem_bytes(int ring) {
  return pa_bar_offset<KV>(ring) + kQFragBytes + 4 * ring * 8;
}

// Row of dim d in a dequantised V page: the 16-byte rows (8 tokens of one
// dim) are rotated within each group of 8 by d/8, so that the dequant's
// stores (lane L writes dims 4L..4L+3) spread over all 32 banks; a
// ldmatrix of 8 consecutive dims still reads one 128-byte block.
__device__ __forceinline__ int mx_vrow(int d) { return (d & ~7) | ((d + (d >> 3)) & 7); }

// dequantise one MXFP4 page (K and V, 16 tokens) into the bf16 page layout
// K [d/8][16 t][8], V [t/8][128 rows][8] (dim d at row mx_vrow(d))
__device__ __forceinline__ void mx_page_to_bf16(const uint8_t* slot, uint8_t* dq, int lane) {
  {  // K: lane = (token, half of the dims)
    const int tk = lane >> 1, hf = lane & 1;
    const uint4* src = reinterpret_cast<const uint4*>(slot + tk * 64 + hf * 32);
    const uint4 w0 = src[0], w1 = src[1];
    const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const uint32_t sc = *reinterpret_cast<const uint16_t*>(slot + 1024 + tk * 4 + 2 * hf);
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // 8 dims per word
      const float s = e8m0_to_float((sc >> (8 * (j >> 2))) & 0xFF);
      uint32_t out[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 f = f16x2_to_float2(e2m1x2_to_f16x2((words[j] >> (8 * b)) & 0xFF));
        out[b] = pack_bf16x2(f.x * s, f.y * s);
      }
      *reinterpret_cast<uint4*>(dq + (hf * 8 + j) * 256 + tk * 16) = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
  {  // V: lane = dims 4*lane..+3; 8 tokens at a time
    const uint8_t* vd = slot + 1088;
    const uint8_t* vs = slot + 2112;
#pragma unroll
    for (int th = 0; th < 2; ++th) {
      float v[8][4];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int tk = 8 * th + k;
        const uint32_t two = *reinterpret_cast<const uint16_t*>(vd + tk * 64 + 2 * lane);
        const float s = e8m0_to_float(vs[tk * 4 + (lane >> 3)]);
        const float2 f0 = f16x2_to_float2(e2m1x2_to_f16x2(two & 0xFF));
        const float2 f1 = f16x2_to_float2(e2m1x2_to_f16x2(two >> 8));
        v[k][0] = f0.x * s, v[k][1] = f0.y * s, v[k][2] = f1.x * s, v[k][3] = f1.y * s;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 w;
        w.x = pack_bf16x2(v[0][i], v[1][i]);
        w.y = pack_bf16x2(v[2][i], v[3][i]);
        w.z = pack_bf16x2(v[4][i], v[5][i]);
        w.w = pack_bf16x2(v[6][i], v[7][i]);
        *reinterpret_cast<uint4*>(dq + 4096 + th * 2048 + mx_vrow(4 * lane + i) * 16) = w;
      }
    }
  }
}

// the workspace starts with one int32 arrival counter per row, padded to 256 B
__host__ __device__ constexpr int64_t ws_counter_floats(int64_t rows) { return (rows + 63) / 64 * 64; }




// running state of one warp's online softmax: O (16 heads x 128 dims as 16
// n-tiles of the mma accumulator), max m and sum l of heads g and g+8
struct PaState {
  float o[16][4];
  float m0, m1, l0, l1;
};

__device__ __forceinline__ void pa_state_init(PaState& a) {
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) a.o[nd][0] = a.o[nd][1] = a.o[nd][2] = a.o[nd][3] = 0.f;
  a.m0 = a.m1 = -INFINITY;
  a.l0 = a.l1 = 0.f;
}

// Q fragments (A operand) of one row: tile rows = query heads g and g+8 of
// the row's KV head.  Warp w builds k-steps 2w and 2w+1 and stores them to
// shared memory at qs as [kc][lane] uint4 (4 KB); the caller synchronises the
// CTA before they are read.  Split in two so that the global loads are in
// flight while the warp does other work: load_q_raw issues them (raw q
// words, zero for heads past the group), store_q_raw converts and stores.
struct QRaw {
  uint32_t w[2][2][2];  // [k-step][head half][word]
};

template <int KV>
__device__ __forceinline__ QRaw load_q_raw(const void* q, int q_dtype, int64_t qrow, int group, int warp, int lane) {
  constexpr bool F16 = KV == BSP_FP8_E4M3;
  const int g = lane >> 2, t = lane & 3;
  QRaw r;
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    const int kc = 2 * warp + kk;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int head = g + 8 * half;
      const int64_t e = qrow + head * kDim + 16 * kc;
      uint32_t w0 = 0, w1 = 0;
      if (head < group) {
        if (q_dtype == BSP_BF16) {
          const uint16_t* b = static_cast<const uint16_t*>(q) + e;
          if (F16) {  // elements 4t..4t+3
            const uint2 v = *reinterpret_cast<const uint2*>(b + 4 * t);
            w0 = v.x, w1 = v.y;
          } else {  // elements 2t, 2t+1 and 8+2t, 9+2t
            w0 = *reinterpret_cast<const uint32_t*>(b + 2 * t);
            w1 = *reinterpret_cast<const uint32_t*>(b + 8 + 2 * t);
          }
        } else {
          const uint8_t* b = static_cast<const uint8_t*>(q) + e;
          if (F16) {
            w0 = *reinterpret_cast<const uint32_t*>(b + 4 * t);
          } else {
            w0 = *reinterpret_cast<const uint16_t*>(b + 2 * t);
            w1 = *reinterpret_cast<const uint16_t*>(b + 8 + 2 * t);
          }
        }
      }
      r.w[kk][half][0] = w0;
      r.w[kk][half][1] = w1;
    }
  }
  return r;
}

template <int KV>
__device__ __forceinline__ void store_q_raw(uint32_t qs, const QRaw& r, int q_dtype, int warp, int lane) {
  constexpr bool F16 = KV == BSP_FP8_E4M3;
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    const int kc = 2 * warp + kk;
    uint32_t f[4];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t w0 = r.w[kk][half][0], w1 = r.w[kk][half][1];
      float v[4];
      if (q_dtype == BSP_BF16) {
        v[0] = bf16_bits_to_float(w0 & 0xFFFF), v[1] = bf16_bits_to_float(w0 >> 16);
        v[2] = bf16_bits_to_float(w1 & 0xFFFF), v[3] = bf16_bits_to_float(w1 >> 16);
      } else if (F16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = e4m3_to_float(w0 >> (8 * i));
      } else {
        v[0] = e4m3_to_float(w0), v[1] = e4m3_to_float(w0 >> 8);
        v[2] = e4m3_to_float(w1), v[3] = e4m3_to_float(w1 >> 8);
      }
      if (F16) {
        f[half] = pack_f16x2(v[0], v[1]);
        f[2 + half] = pack_f16x2(v[2], v[3]);
      } else {
        f[half] = pack_bf16x2(v[0], v[1]);
        f[2 + half] = pack_bf16x2(v[2], v[3]);
      }
    }
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(qs + (kc * 32 + lane) * 16), "r"(f[0]), "r"(f[1]),
                 "r"(f[2]), "r"(f[3])
                 : "memory");
  }
}

// One 16-token page of one warp: K at shared address kaddr, V at vaddr (fp8
// layouts for KV = fp8, bf16 layouts otherwise); tok0 = the page's first
// token in the row, tokens >= ctx are masked.
template <int KV>
__device__ __forceinline__ void pa_page(PaState& a, uint32_t qs, uint32_t kaddr, uint32_t vaddr, int tok0, int ctx,
                                        float qk_scale, int lane) {
  constexpr bool F16 = KV == BSP_FP8_E4M3;
  const int t = lane & 3;
  // S = Q Kt: both 8-token n-tiles interleaved, two accumulators each, so no
  // mma waits on the one before it for more than 4 steps
  float s[2][4];
  {
    float acc[2][2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) acc[nt][e][0] = acc[nt][e][1] = acc[nt][e][2] = acc[nt][e][3] = 0.f;
    if (F16) {
      const int rr = lane & 7;
#pragma unroll
      for (int q4 = 0; q4 < 2; ++q4) {
        uint32_t r[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int tok = 4 * (rr >> 1) + 2 * nt + (rr & 1);
          ldsm_x4(r[nt][0], r[nt][1], r[nt][2], r[nt][3], kaddr + (4 * q4 + (lane >> 3)) * 256 + tok * 16);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kc = 4 * q4 + j;
          const uint4 qa = lds128(qs + (kc * 32 + lane) * 16);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            uint32_t b0, b1;
            kv_e4m3x4_to_f16x2(r[nt][j], b0, b1);
            mma_f16(acc[nt][j & 1], qa.x, qa.y, qa.z, qa.w, b0, b1);
          }
        }
      }
    } else {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int kc = 2 * q4;
        const uint4 qa0 = lds128(qs + (kc * 32 + lane) * 16), qa1 = lds128(qs + ((kc + 1) * 32 + lane) * 16);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t r[4];
          ldsm_x4(r[0], r[1], r[2], r[3], kaddr + (4 * q4 + (lane >> 3)) * 256 + (8 * nt + (lane & 7)) * 16);
          mma_bf16(acc[nt][0], qa0.x, qa0.y, qa0.z, qa0.w, r[0], r[1]);
          mma_bf16(acc[nt][1], qa1.x, qa1.y, qa1.z, qa1.w, r[2], r[3]);
        }
      }
    }
    // only a row's last page can reach past its context; the others skip
    // the per-token test (a warp-uniform branch)
    if (tok0 + kPage <= ctx) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[nt][j] = (acc[nt][0][j] + acc[nt][1][j]) * qk_scale;
    } else {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tok = F16 ? 4 * t + 2 * nt + (j & 1) : 8 * nt + 2 * t + (j & 1);
          s[nt][j] = tok0 + tok < ctx ? (acc[nt][0][j] + acc[nt][1][j]) * qk_scale : -INFINITY;
        }
    }
  }

  // online softmax (log2 domain); rows g (regs 0,1) and g+8 (regs 2,3)
  float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
  float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  // The reference max moves only when a row's max grows by more than 2^8
  // (kRescaleLog2): P then stays below 256, exact enough in f16/bf16 and far
  // from overflow, and O is rescaled only on the (warp-uniform) pages where
  // some row's max moved.  softmax = exp2(s - m) / sum is the same for any m.
  const bool move0 = mx0 > a.m0 + kRescaleLog2, move1 = mx1 > a.m1 + kRescaleLog2;
  const float mn0 = move0 ? mx0 : a.m0, mn1 = move1 ? mx1 : a.m1;
  const float al0 = ex2_approx(a.m0 - mn0), al1 = ex2_approx(a.m1 - mn1);
  a.m0 = mn0, a.m1 = mn1;
  float pr[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    pr[nt][0] = ex2_approx(s[nt][0] - mn0);
    pr[nt][1] = ex2_approx(s[nt][1] - mn0);
    pr[nt][2] = ex2_approx(s[nt][2] - mn1);
    pr[nt][3] = ex2_approx(s[nt][3] - mn1);
  }
  a.l0 = a.l0 * al0 + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
  a.l1 = a.l1 * al1 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
  if (__any_sync(0xffffffffu, move0 || move1)) {
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      a.o[nd][0] *= al0, a.o[nd][1] *= al0, a.o[nd][2] *= al1, a.o[nd][3] *= al1;
    }
  }

  // O += P V
  uint32_t pa0, pa1, pa2, pa3;
  if (F16) {
    pa0 = pack_f16x2(pr[0][0], pr[0][1]);
    pa1 = pack_f16x2(pr[0][2], pr[0][3]);
    pa2 = pack_f16x2(pr[1][0], pr[1][1]);
    pa3 = pack_f16x2(pr[1][2], pr[1][3]);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint32_t r[4];
      ldsm_x4(r[0], r[1], r[2], r[3], vaddr + (8 * (4 * q4 + (lane >> 3)) + (lane & 7)) * 16);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t b0, b1;
        kv_e4m3x4_to_f16x2(r[j], b0, b1);
        mma_f16(a.o[4 * q4 + j], pa0, pa1, pa2, pa3, b0, b1);
      }
    }
  } else {
    // bf16 P carries 8 significant bits; P = hi + lo (both bf16) keeps ~16
    uint32_t lo0, lo1, lo2, lo3;
    split_bf16x2(pr[0][0], pr[0][1], pa0, lo0);
    split_bf16x2(pr[0][2], pr[0][3], pa1, lo1);
    split_bf16x2(pr[1][0], pr[1][1], pa2, lo2);
    split_bf16x2(pr[1][2], pr[1][3], pa3, lo3);
#pragma unroll
    for (int q8 = 0; q8 < 8; ++q8) {
      uint32_t r[4];
      const int d = 8 * (2 * q8 + (lane >> 4)) + (lane & 7);
      ldsm_x4(r[0], r[1], r[2], r[3], vaddr + ((lane >> 3) & 1) * 2048 + (KV == BSP_MXFP4 ? mx_vrow(d) : d) * 16);
      mma_bf16(a.o[2 * q8], pa0, pa1, pa2, pa3, r[0], r[1]);
      mma_bf16(a.o[2 * q8], lo0, lo1, lo2, lo3, r[0], r[1]);
      mma_bf16(a.o[2 * q8 + 1], pa0, pa1, pa2, pa3, r[2], r[3]);
      mma_bf16(a.o[2 * q8 + 1], lo0, lo1, lo2, lo3, r[2], r[3]);
    }
  }
}

// The four warps' states of one row merged through the shared-memory area
// cb (kCombineFloats floats; free on entry).  On return thread tid holds, for
// head hh = tid/8 and dims dq + 32j (dq = 4*(tid%8), j < 4), the merged max
// M (log2 domain), sum L and unnormalised output acc.  Rows are padded to 136
// floats so the fragment stores hit each bank twice at most.
__device__ __forceinline__ void pa_combine(float* cb, const PaState& a, int tid, float& M, float& L,
                                           float4 (&acc)[4]) {
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  // sum l over the quad (the 4 threads of a head row)
  float l0 = a.l0, l1 = a.l1;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  constexpr int kCo = kDim + 8;
  float* cm = cb;        // [4][16]
  float* cl = cm + 64;   // [4][16]
  float* co = cl + 64;   // [4][16][kCo]
  __syncthreads();
  if (t == 0) {
    cm[warp * 16 + g] = a.m0, cm[warp * 16 + g + 8] = a.m1;
    cl[warp * 16 + g] = l0, cl[warp * 16 + g + 8] = l1;
  }
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) {
    *reinterpret_cast<float2*>(co + (warp * 16 + g) * kCo + 8 * nd + 2 * t) = make_float2(a.o[nd][0], a.o[nd][1]);
    *reinterpret_cast<float2*>(co + (warp * 16 + g + 8) * kCo + 8 * nd + 2 * t) = make_float2(a.o[nd][2], a.o[nd][3]);
  }
  __syncthreads();
  const int hh = tid >> 3, dq = 4 * (tid & 7);
  M = -INFINITY;
#pragma unroll
  for (int w = 0; w < 4; ++w) M = fmaxf(M, cm[w * 16 + hh]);
  float wgt[4];
  L = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    wgt[w] = M == -INFINITY ? 0.f : exp2f(cm[w * 16 + hh] - M);
    L += wgt[w] * cl[w * 16 + hh];
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float4 c = *reinterpret_cast<const float4*>(co + (w * 16 + hh) * kCo + dq + 32 * j);
      acc[j].x += wgt[w] * c.x, acc[j].y += wgt[w] * c.y, acc[j].z += wgt[w] * c.z, acc[j].w += wgt[w] * c.w;
    }
  }
}

// dims dq + 32j of one head's output row, scaled by f, as bf16
__device__ __forceinline__ void store_out_row(uint16_t* orow, int dq, const float4 (&acc)[4], float f) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint2*>(orow + dq + 32 * j) =
        make_uint2(pack_bf16x2(acc[j].x * f, acc[j].y * f), pack_bf16x2(acc[j].z * f, acc[j].w * f));
}

// TMA copies of one page (K and V of KV head h) into a ring slot; bad ids
// are flagged and replaced by page 0
template <int KV>
__device__ __forceinline__ void issue_page(const SparsePaParams& p, int64_t id, int h, uint8_t* slot, uint64_t* bar) {
  constexpr int SB = PaFmt<KV>::kSlot;
  if (id < 0 || id >= p.num_ids) {
    set_err(p.err, BSP_DEVERR_PAGE_ID);
    id = 0;
  }
  mbar_arrive_expect_tx(bar, SB);
  if (KV == BSP_MXFP4) {
    const int64_t blk = id / kPagesPerSide, u = id % kPagesPerSide;
    const uint8_t* kf = p.k_base + blk * p.id_stride + static_cast<int64_t>(h) * kMxField;
    const uint8_t* vf = p.v_base + blk * p.id_stride + static_cast<int64_t>(h) * kMxField;
    bulk_g2s(slot, kf + u * 1024, 1024, bar);
    bulk_g2s(slot + 1024, kf + kMxScaleOff + u * 64, 64, bar);
    bulk_g2s(slot + 1088, vf + u * 1024, 1024, bar);
    bulk_g2s(slot + 2112, vf + kMxScaleOff + u * 64, 64, bar);
  } else {
    constexpr int PB = SB / 2;
    bulk_g2s(slot, p.k_base + id * p.id_stride + static_cast<int64_t>(h) * PB, PB, bar);
    bulk_g2s(slot + PB, p.v_base + id * p.id_stride + static_cast<int64_t>(h) * PB, PB, bar);
  }
}

// ---------------------------------------------------------------------------
// per-row schedule: CTA = (row, split)
template <int KV>
__global__ void __launch_bounds__(128, PaFmt<KV>::kMinCtas)
    sparse_pa_kernel(SparsePaParams p, float qk_scale, float out_scale) {
  constexpr int SB = PaFmt<KV>::kSlot, DQ = PaFmt<KV>::kDeq;
  const int R = p.ring;  // pages in flight per warp, 1..kRingMax
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t qs = smem_u32(smem + pa_bar_offset<KV>(R));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pa_bar_offset<KV>(R) + kQFragBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t cta = blockIdx.x;
  const int row = static_cast<int>(cta / p.nsplit), split = static_cast<int>(cta % p.nsplit);
  const int h = row % p.hkv;
  const int64_t token = row / p.hkv;
  const int hq = p.hkv * p.group;

  if (tid == 0) {
    for (int i = 0; i < 4 * R; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
  const int64_t q_off = (token * hq + static_cast<int64_t>(h) * p.group) * kDim;
  QRaw qraw;
  if (p.q_early) {  // the queries do not come from the kernel before: stage them before waiting
    qraw = load_q_raw<KV>(p.q, p.q_dtype, q_off, p.group, warp, lane);
    store_q_raw<KV>(qs, qraw, p.q_dtype, warp, lane);
  }
  __syncthreads();
  pdl_wait();  // the sparse table (and the queries, unless staged) come from earlier kernels
  pdl_trigger();

  // the queries' loads go out first; they land while the page ids and the
  // first pages are fetched
  if (!p.q_early) qraw = load_q_raw<KV>(p.q, p.q_dtype, q_off, p.group, warp, lane);
  // this warp's page ids, 32 at a time, loaded together ahead of use: lane j
  // holds the id of the warp's page 32*c + j (the ring issues its TMA copies
  // from these without a dependent global load).  The first 32 are loaded
  // alongside the row's context length, over the split's whole page range
  // (entries past the context are never used).
  const int p0 = split * p.pages_per_split;
  const int pmax = min(p0 + p.pages_per_split, p.k_pages);  // the split's pages, whatever the context
  const int32_t* sbt = p.sparse_bt + static_cast<int64_t>(row) * p.k_pages;
  int32_t my_id = 0;
  int id_chunk = 0;
  if (p0 + warp + 4 * lane < pmax) my_id = sbt[p0 + warp + 4 * lane];
  const int ctx = min(max(p.sparse_ctx[row], 0), p.k_pages * kPage);
  const int npages = (ctx + kPage - 1) / kPage;
  const int p1 = min(pmax, npages);
  const int nw = p1 > p0 + warp ? (p1 - p0 - warp + 3) / 4 : 0;
  uint8_t* wring = smem + warp * R * SB;
  uint64_t* wbar = bars + warp * R;
  uint8_t* wdq = smem + 4 * R * SB + warp * DQ;

  auto id_of = [&](int j) -> int32_t {  // warp-uniform j
    if ((j >> 5) != id_chunk) {
      id_chunk = j >> 5;
      const int jj = 32 * id_chunk + lane;
      my_id = jj < nw ? sbt[p0 + warp + 4 * jj] : 0;
    }
    return __shfl_sync(0xffffffffu, my_id, j & 31);
  };
  for (int i = 0; i < R; ++i) {
    const int32_t id = id_of(i);
    if (lane == 0 && i < nw) issue_page<KV>(p, id, h, wring + i * SB, &wbar[i]);
  }

  if (!p.q_early) {
    store_q_raw<KV>(qs, qraw, p.q_dtype, warp, lane);
    __syncthreads();
  }

  PaState a;
  pa_state_init(a);
  bool alive = true;  // false after a timed-out wait: no further waits
  int st = 0;         // ring slot of page i, and the parity of its phase
  uint32_t phase = 0;
  for (int i = 0; i < nw; ++i) {
    if (alive) alive = mbar_wait_sleep(&wbar[st], phase, p.err);
    const int pg = p0 + warp + 4 * i;
    if (KV == BSP_MXFP4) {
      __syncwarp();  // every lane is done reading the previous dequantised page
      mx_page_to_bf16(wring + st * SB, wdq, lane);
      __syncwarp();
      const int32_t id = id_of(i + R);
      if (lane == 0 && i + R < nw) {
        fence_proxy_async();
        issue_page<KV>(p, id, h, wring + st * SB, &wbar[st]);
      }
      pa_page<KV>(a, qs, smem_u32(wdq), smem_u32(wdq) + 4096, pg * kPage, ctx, qk_scale, lane);
    } else {
      pa_page<KV>(a, qs, smem_u32(wring + st * SB), smem_u32(wring + st * SB) + SB / 2, pg * kPage, ctx, qk_scale,
                  lane);
      __syncwarp();
      const int32_t id = id_of(i + R);
      if (lane == 0 && i + R < nw) {
        fence_proxy_async();
        issue_page<KV>(p, id, h, wring + st * SB, &wbar[st]);
      }
    }
    if (++st == R) st = 0, phase ^= 1;
  }

  // merge the four warps (the rings are no longer used)
  float* cm = reinterpret_cast<float*>(smem);
  float M, L;
  float4 acc[4];
  pa_combine(cm, a, tid, M, L, acc);
  const int hh = tid >> 3, dq = 4 * (tid & 7);
  uint16_t* orow = static_cast<uint16_t*>(p.out) + (token * hq + static_cast<int64_t>(h) * p.group + hh) * kDim;
  if (p.nsplit == 1) {
    if (hh < p.group) store_out_row(orow, dq, acc, L > 0.f ? out_scale / L : 0.f);
    return;
  }

  if (p.cluster > 1) {
    // The row's splits form one thread-block cluster: publish this split's
    // partial in shared memory, and after a cluster barrier CTA k merges
    // heads k, k+nsplit, ... reading every peer's partial through
    // distributed shared memory (no global round trip).
    float* pm = cm + kCombineFloats;  // [16]
    float* pl = pm + 16;              // [16]
    float* po = pl + 16;              // [16][128]
    if ((tid & 7) == 0) pm[hh] = M, pl[hh] = L;
#pragma unroll
    for (int j = 0; j < 4; ++j) *reinterpret_cast<float4*>(po + hh * kDim + dq + 32 * j) = acc[j];
    cluster_sync();
    // CTA `rank` finishes heads rank, rank + nsplit, ...: 32 threads per
    // head, 4 dims each; every peer's (m, l, O[4 dims]) is loaded at once
    const int rank = static_cast<int>(cluster_ctarank()), ns = p.nsplit;
    const int d = 4 * (tid & 31);
    for (int head = rank + (tid >> 5) * ns; head < p.group; head += 4 * ns) {
      float mv[kMaxCluster], lv[kMaxCluster];
      float4 ov[kMaxCluster];
#pragma unroll
      for (int sp = 0; sp < kMaxCluster; ++sp) {
        if (sp < ns) {
          mv[sp] = *cluster_map(pm + head, sp);
          lv[sp] = *cluster_map(pl + head, sp);
          ov[sp] = *reinterpret_cast<const float4*>(cluster_map(po + head * kDim + d, sp));
        }
      }
      float Mx = -INFINITY;
#pragma unroll
      for (int sp = 0; sp < kMaxCluster; ++sp)
        if (sp < ns) Mx = fmaxf(Mx, mv[sp]);
      float Ls = 0.f;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int sp = 0; sp < kMaxCluster; ++sp) {
        if (sp < ns) {
          const float w = (Mx == -INFINITY || mv[sp] == -INFINITY) ? 0.f : exp2f(mv[sp] - Mx);
          Ls += w * lv[sp];
          O.x += w * ov[sp].x, O.y += w * ov[sp].y, O.z += w * ov[sp].z, O.w += w * ov[sp].w;
        }
      }
      const float f = Ls > 0.f ? out_scale / Ls : 0.f;
      uint16_t* dst = static_cast<uint16_t*>(p.out) + (token * hq + static_cast<int64_t>(h) * p.group + head) * kDim + d;
      *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(O.x * f, O.y * f), pack_bf16x2(O.z * f, O.w * f));
    }
    cluster_sync_relaxed();  // peers are done reading this CTA's shared memory
    return;
  }

  // split-K: publish this split's (m, l, O), then the last CTA of the row to
  // arrive merges all splits (no second kernel, no waiting: the counter tells
  // the last one that every other split has been written)
  int32_t* counters = reinterpret_cast<int32_t*>(p.ws);
  float* wso = p.ws + ws_counter_floats(p.num_rows);
  float* wsml = wso + static_cast<int64_t>(p.num_rows) * p.nsplit * 16 * kDim;
  const int64_t unit = static_cast<int64_t>(row) * p.nsplit + split;
#pragma unroll
  for (int j = 0; j < 4; ++j) *reinterpret_cast<float4*>(wso + (unit * 16 + hh) * kDim + dq + 32 * j) = acc[j];
  if ((tid & 7) == 0) *reinterpret_cast<float2*>(wsml + (unit * 16 + hh) * 2) = make_float2(M, L);
  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) s_last = atomicAdd(&counters[row], 1) == p.nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  float* sw = cm;  // [nsplit][16] merge weights, then [16] 1/L
  float* sinv = cm + 16 * p.nsplit;
  if (tid < 16) {
    float Mx = -INFINITY;
    for (int sp = 0; sp < p.nsplit; ++sp)
      Mx = fmaxf(Mx, __ldcg(wsml + ((static_cast<int64_t>(row) * p.nsplit + sp) * 16 + tid) * 2));
    float Ls = 0.f;
    for (int sp = 0; sp < p.nsplit; ++sp) {
      const float2 ml =
          __ldcg(reinterpret_cast<const float2*>(wsml + ((static_cast<int64_t>(row) * p.nsplit + sp) * 16 + tid) * 2));
      const float w = (Mx == -INFINITY || ml.x == -INFINITY) ? 0.f : exp2f(ml.x - Mx);
      sw[sp * 16 + tid] = w;
      Ls += w * ml.y;
    }
    sinv[tid] = Ls > 0.f ? out_scale / Ls : 0.f;
  }
  __syncthreads();
  if (hh < p.group) {
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < p.nsplit; ++sp) {
      const float w = sw[sp * 16 + hh];
      const float* src = wso + ((static_cast<int64_t>(row) * p.nsplit + sp) * 16 + hh) * kDim + dq;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 c = __ldcg(reinterpret_cast<const float4*>(src + 32 * j));
        acc[j].x += w * c.x, acc[j].y += w * c.y, acc[j].z += w * c.z, acc[j].w += w * c.w;
      }
    }
    store_out_row(orow, dq, acc, sinv[hh]);
  }
  if (tid == 0) counters[row] = 0;  // ready for the next call
}

// the dynamic shared-memory opt-in of a kernel: its largest ring (once per device)
template <int KV>
cudaError_t configure_kv() {
  static std::atomic<uint64_t> done{0};
  return once_per_device(done, [] {
    return cudaFuncSetAttribute(sparse_pa_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                pa_smem_bytes<KV>(PaFmt<KV>::kRingMax));
  });
}

template <int KV>
cudaError_t launch_kv(const SparsePaParams& p, cudaStream_t s, int* launches) {
  if (p.ring < 1 || p.ring > PaFmt<KV>::kRingMax) return cudaErrorInvalidValue;
  {
    const cudaError_t e = configure_kv<KV>();
    if (e != cudaSuccess) return e;
  }
  const float kfold = KV == BSP_FP8_E4M3 ? p.k_scale : 1.f;
  const float vfold = KV == BSP_FP8_E4M3 ? p.v_scale : 1.f;
  const float qk_scale = p.sm_scale * kfold * kLog2e;
  const int64_t ctas = static_cast<int64_t>(p.num_rows) * p.nsplit;
  const cudaError_t e = launch_kernel(sparse_pa_kernel<KV>, dim3(static_cast<unsigned>(ctas)), dim3(128),
                                      pa_smem_bytes<KV>(p.ring), s, p.cluster, p, qk_scale, vfold);
  if (e != cudaSuccess) return e;
  ++*launches;
  return cudaPeekAtLastError();
}

// resident CTAs per SM of the per-row kernel with a ring of `ring` pages per
// warp (queried once per format and depth; a failed query assumes 1)
template <int KV>
int occupancy_kv(int ring) {
  static std::atomic<int> cache[PaFmt<KV>::kRingMax + 1][kMaxDevices];
  return cached_per_device(cache[ring], [ring] {
    int n = 0;
    cudaError_t e = configure_kv<KV>();
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sparse_pa_kernel<KV>, 128, pa_smem_bytes<KV>(ring));
    return (e == cudaSuccess && n > 0) ? n : 1;
  });
}

template <int KV>
PaPlan plan_kv(int32_t num_rows, int32_t k_pages, int num_sms) {
  PaPlan plan{};
  const int64_t rows = num_rows > 0 ? num_rows : 1;
  // split each row over floor(resident / rows) CTAs: the fewest CTAs that
  // fill one wave (fewer, longer CTAs stream better than many short ones);
  // up to 8 splits form one cluster and merge on chip, more (very few rows)
  // merge through the workspace
  const int base_ring = PaFmt<KV>::kRing;
  const int64_t per_sm = occupancy_kv<KV>(base_ring);
  int64_t ns = per_sm * num_sms / rows;
  const int64_t max_ns = std::min<int64_t>(64, (k_pages + 3) / 4);
  ns = ns < 1 ? 1 : (ns > max_ns ? max_ns : ns);
  if (ns > kMaxCluster && rows * kMaxCluster >= num_sms) ns = kMaxCluster;
  int64_t pps = (k_pages + ns - 1) / ns;
  pps = (pps + 3) / 4 * 4;
  if (pps < 4) pps = 4;
  ns = (k_pages + pps - 1) / pps;
  if (ns < 1) ns = 1;
  plan.nsplit = static_cast<int32_t>(ns);
  plan.pages_per_split = static_cast<int32_t>(pps);
  plan.cluster = (ns >= 2 && ns <= kMaxCluster) ? static_cast<int32_t>(ns) : 0;
  // deepen the ring while the grid still fits in one wave: a warp's pages
  // (pps / 4) all in flight at once when there is room
  const int64_t ctas = rows * ns, per_warp = (pps + 3) / 4;
  int ring = base_ring;
  while (ring < PaFmt<KV>::kRingMax && ring < per_warp &&
         static_cast<int64_t>(occupancy_kv<KV>(ring + 1)) * num_sms >= ctas)
    ++ring;
  plan.ring = ring;
  return plan;
}

}  // namespace

PaPlan sparse_pa_plan(int32_t kv_dtype, int32_t num_rows, int32_t k_pages, int num_sms) {
  switch (kv_dtype) {
    case BSP_FP8_E4M3:
      return plan_kv<BSP_FP8_E4M3>(num_rows, k_pages, num_sms);
    case BSP_BF16:
      return plan_kv<BSP_BF16>(num_rows, k_pages, num_sms);
    default:
      return plan_kv<BSP_MXFP4>(num_rows, k_pages, num_sms);
  }
}

PaPlan sparse_pa_prefill_plan(int32_t kv_dtype, int32_t k_pages) {
  PaPlan plan{};
  plan.nsplit = 1;
  plan.pages_per_split = (k_pages + 3) / 4 * 4;
  plan.ring = kv_dtype == BSP_FP8_E4M3 ? PaFmt<BSP_FP8_E4M3>::kRing
                                       : (kv_dtype == BSP_BF16 ? PaFmt<BSP_BF16>::kRing : PaFmt<BSP_MXFP4>::kRing);
  return plan;
}

size_t sparse_pa_ws_bytes(int32_t num_rows, const PaPlan& plan) {
  if (plan.nsplit <= kMaxCluster) return 0;  // no split, or merged on chip in a cluster
  const size_t partials = static_cast<size_t>(num_rows) * plan.nsplit;
  return (static_cast<size_t>(ws_counter_floats(num_rows)) + partials * 16 * (kDim + 2)) * sizeof(float);
}

size_t sparse_pa_counter_bytes(int32_t num_rows) { return static_cast<size_t>(ws_counter_floats(num_rows)) * 4; }

cudaError_t launch_sparse_pa(const SparsePaParams& p, cudaStream_t s, int* launches) {
  if (p.num_rows == 0) return cudaSuccess;
  switch (p.kv_dtype) {
    case BSP_FP8_E4M3:
      return launch_kv<BSP_FP8_E4M3>(p, s, launches);
    case BSP_BF16:
      return launch_kv<BSP_BF16>(p, s, launches);
    default:
      return launch_kv<BSP_MXFP4>(p, s, launches);
  }
}

}  // namespace bsp
