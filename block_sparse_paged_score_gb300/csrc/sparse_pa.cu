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
// CTA = 4 warps = one (row, split); a split is a run of pages and warp w takes
// pages w, w+4, ... of it.  Each warp streams its pages through a ring of
// shared-memory slots with 1-D TMA bulk copies (K page + V page of its head;
// MXFP4: the 1 KB data and 64 B scales of both sides) completing on mbarriers,
// and keeps its own online softmax.  Per 16-token page:
//   S  = Q Kt : 2 n-tiles (8 tokens) x 8 k-steps of mma.sync m16n8k16
//   P  = exp2(S*scale - m)   (log2 domain, running max m and sum l per head)
//   O += P V  : 16 n-tiles (8 dims) of mma.sync m16n8k16
// fp8 pages are converted to f16 in registers right after ldmatrix (exact:
// value * 2^-8; the k/v scales and 2^8 are folded into the softmax scale and
// the output scale).  For fp8 the 16 tokens of a page enter the mma in the
// order 0,1,4,5,8,9,12,13 | 2,3,6,7,... so that the S accumulator lands as the
// P fragment whose tokens match the V rows a ldmatrix of the dim-major V page
// hands each thread (tokens 4t..4t+3); bf16 pages use the natural order.
// MXFP4 pages are dequantised by the warp into a bf16 page (e2m1 * 2^(e-127)
// is exact in bf16) and then take the bf16 path.
// The 4 warps merge in shared memory (log-sum-exp); a row with one split is
// written directly, otherwise the CTA writes (m, l, O) to the workspace and
// sparse_pa_merge combines the splits.
#include "common.cuh"
#include "kernels.h"

namespace bsp {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int KV>
struct PaFmt;
template <>
struct PaFmt<BSP_FP8_E4M3> {
  static constexpr int kRing = 3, kSlot = 4096, kDeq = 0;
};
template <>
struct PaFmt<BSP_BF16> {
  static constexpr int kRing = 2, kSlot = 8192, kDeq = 0;
};
template <>
struct PaFmt<BSP_MXFP4> {
  // K data 1024 | K scales 64 | V data 1024 | V scales 64
  static constexpr int kRing = 3, kSlot = 2176, kDeq = 8192;
};

template <int KV>
constexpr int pa_smem_bytes() {
  return 4 * PaFmt<KV>::kRing * PaFmt<KV>::kSlot + 4 * PaFmt<KV>::kDeq + 4 * PaFmt<KV>::kRing * 8;
}
static_assert(4 * 3 * 4096 >= 4 * (16 * 128 + 32) * 4, "combine area fits the fp8 ring");

__device__ __forceinline__ void load_q_vals(const void* q, int q_dtype, int64_t off, int n, float* v) {
  if (q_dtype == BSP_BF16) {
    const uint16_t* p = static_cast<const uint16_t*>(q) + off;
    for (int i = 0; i < n; ++i) v[i] = bf16_bits_to_float(p[i]);
  } else {
    const uint8_t* p = static_cast<const uint8_t*>(q) + off;
    for (int i = 0; i < n; ++i) v[i] = e4m3_to_float(p[i]);
  }
}

// dequantise one MXFP4 page (K and V, 16 tokens) into the bf16 page layout
// K [d/8][16 t][8], V [t/8][128 d][8]
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
  {  // V: lane = dims 4*lane..+3, all 16 tokens
    const uint8_t* vd = slot + 1088;
    const uint8_t* vs = slot + 2112;
    float v[16][4];
#pragma unroll
    for (int tk = 0; tk < 16; ++tk) {
      const uint32_t two = *reinterpret_cast<const uint16_t*>(vd + tk * 64 + 2 * lane);
      const float s = e8m0_to_float(vs[tk * 4 + (lane >> 3)]);
      const float2 f0 = f16x2_to_float2(e2m1x2_to_f16x2(two & 0xFF));
      const float2 f1 = f16x2_to_float2(e2m1x2_to_f16x2(two >> 8));
      v[tk][0] = f0.x * s, v[tk][1] = f0.y * s, v[tk][2] = f1.x * s, v[tk][3] = f1.y * s;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int th = 0; th < 2; ++th) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * th + 0][i], v[8 * th + 1][i]);
        w.y = pack_bf16x2(v[8 * th + 2][i], v[8 * th + 3][i]);
        w.z = pack_bf16x2(v[8 * th + 4][i], v[8 * th + 5][i]);
        w.w = pack_bf16x2(v[8 * th + 6][i], v[8 * th + 7][i]);
        *reinterpret_cast<uint4*>(dq + 4096 + th * 2048 + (4 * lane + i) * 16) = w;
      }
  }
}

template <int KV>
__global__ void __launch_bounds__(128) sparse_pa_kernel(SparsePaParams p, float qk_scale, float out_scale) {
  constexpr int R = PaFmt<KV>::kRing, SB = PaFmt<KV>::kSlot, DQ = PaFmt<KV>::kDeq;
  constexpr bool F16 = KV == BSP_FP8_E4M3;  // f16 mma with permuted tokens; else bf16
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 4 * R * SB + 4 * DQ);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int64_t cta = blockIdx.x;
  const int row = static_cast<int>(cta / p.nsplit), split = static_cast<int>(cta % p.nsplit);
  const int h = row % p.hkv;
  const int64_t token = row / p.hkv;
  const int hq = p.hkv * p.group;
  const int ctx = min(max(p.sparse_ctx[row], 0), p.k_pages * kPage);
  const int npages = (ctx + kPage - 1) / kPage;
  const int p0 = split * p.pages_per_split, p1 = min(p0 + p.pages_per_split, npages);

  if (tid == 0) {
    for (int i = 0; i < 4 * R; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
  __syncthreads();

  const int nw = p1 > p0 + warp ? (p1 - p0 - warp + 3) / 4 : 0;
  const int32_t* sbt = p.sparse_bt + static_cast<int64_t>(row) * p.k_pages;
  uint8_t* wring = smem + warp * R * SB;
  uint64_t* wbar = bars + warp * R;
  uint8_t* wdq = smem + 4 * R * SB + warp * DQ;

  auto issue = [&](int i) {
    const int pg = p0 + warp + 4 * i;
    int64_t id = sbt[pg];
    if (id < 0 || id >= p.num_ids) {
      set_err(p.err, BSP_DEVERR_PAGE_ID);
      id = 0;
    }
    uint8_t* slot = wring + (i % R) * SB;
    uint64_t* bar = &wbar[i % R];
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
  };
  if (lane == 0)
    for (int i = 0; i < min(R, nw); ++i) issue(i);

  // Q fragments (A operand), rows = heads g and g+8 of this KV head
  uint32_t qa[8][4];
  {
    const int64_t qrow = (token * hq + static_cast<int64_t>(h) * p.group) * kDim;
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int head = g + 8 * half;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (F16) {
          if (head < p.group) load_q_vals(p.q, p.q_dtype, qrow + head * kDim + 16 * kc + 4 * t, 4, v);
          qa[kc][half] = pack_f16x2(v[0], v[1]);
          qa[kc][2 + half] = pack_f16x2(v[2], v[3]);
        } else {
          if (head < p.group) {
            load_q_vals(p.q, p.q_dtype, qrow + head * kDim + 16 * kc + 2 * t, 2, v);
            load_q_vals(p.q, p.q_dtype, qrow + head * kDim + 16 * kc + 8 + 2 * t, 2, v + 2);
          }
          qa[kc][half] = pack_bf16x2(v[0], v[1]);
          qa[kc][2 + half] = pack_bf16x2(v[2], v[3]);
        }
      }
    }
  }

  float o[16][4];
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int i = 0; i < nw; ++i) {
    const int st = i % R;
    mbar_wait(&wbar[st], (i / R) & 1, p.err);
    const int pg = p0 + warp + 4 * i;
    uint32_t kaddr, vaddr;
    if (KV == BSP_MXFP4) {
      mx_page_to_bf16(wring + st * SB, wdq, lane);
      __syncwarp();
      if (lane == 0 && i + R < nw) {
        fence_proxy_async();
        issue(i + R);
      }
      kaddr = smem_u32(wdq);
      vaddr = kaddr + 4096;
    } else {
      kaddr = smem_u32(wring + st * SB);
      vaddr = kaddr + SB / 2;
    }

    // S = Q Kt
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (F16) {
        const int rr = lane & 7;
        const int tok = 4 * (rr >> 1) + 2 * nt + (rr & 1);
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
          uint32_t r[4];
          ldsm_x4(r[0], r[1], r[2], r[3], kaddr + (4 * q4 + (lane >> 3)) * 256 + tok * 16);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t b0, b1;
            e4m3x4_to_f16x2_scaled(r[j], b0, b1);
            const int kc = 4 * q4 + j;
            mma_f16(acc, qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3], b0, b1);
          }
        }
      } else {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t r[4];
          ldsm_x4(r[0], r[1], r[2], r[3], kaddr + (4 * q4 + (lane >> 3)) * 256 + (8 * nt + (lane & 7)) * 16);
          const int kc = 2 * q4;
          mma_bf16(acc, qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3], r[0], r[1]);
          mma_bf16(acc, qa[kc + 1][0], qa[kc + 1][1], qa[kc + 1][2], qa[kc + 1][3], r[2], r[3]);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tok = F16 ? 4 * t + 2 * nt + (j & 1) : 8 * nt + 2 * t + (j & 1);
        s[nt][j] = pg * kPage + tok < ctx ? acc[j] * qk_scale : -INFINITY;
      }
    }

    // online softmax (log2 domain); rows g (regs 0,1) and g+8 (regs 2,3)
    float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    m0 = mn0, m1 = mn1;
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pr[nt][0] = exp2f(s[nt][0] - mn0);
      pr[nt][1] = exp2f(s[nt][1] - mn0);
      pr[nt][2] = exp2f(s[nt][2] - mn1);
      pr[nt][3] = exp2f(s[nt][3] - mn1);
    }
    l0 = l0 * al0 + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
    l1 = l1 * al1 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      o[nd][0] *= al0, o[nd][1] *= al0, o[nd][2] *= al1, o[nd][3] *= al1;
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
          e4m3x4_to_f16x2_scaled(r[j], b0, b1);
          mma_f16(o[4 * q4 + j], pa0, pa1, pa2, pa3, b0, b1);
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
        ldsm_x4(r[0], r[1], r[2], r[3],
                vaddr + ((lane >> 3) & 1) * 2048 + (8 * (2 * q8 + (lane >> 4)) + (lane & 7)) * 16);
        mma_bf16(o[2 * q8], pa0, pa1, pa2, pa3, r[0], r[1]);
        mma_bf16(o[2 * q8], lo0, lo1, lo2, lo3, r[0], r[1]);
        mma_bf16(o[2 * q8 + 1], pa0, pa1, pa2, pa3, r[2], r[3]);
        mma_bf16(o[2 * q8 + 1], lo0, lo1, lo2, lo3, r[2], r[3]);
      }
    }
    __syncwarp();
    if (KV != BSP_MXFP4 && lane == 0 && i + R < nw) {
      fence_proxy_async();
      issue(i + R);
    }
  }

  // sum l over the quad (the 4 threads of a head row)
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // merge the four warps in shared memory (the rings are no longer used)
  __syncthreads();
  float* cm = reinterpret_cast<float*>(smem);  // [4][16]
  float* cl = cm + 64;                         // [4][16]
  float* co = cl + 64;                         // [4][16][128]
  if (t == 0) {
    cm[warp * 16 + g] = m0, cm[warp * 16 + g + 8] = m1;
    cl[warp * 16 + g] = l0, cl[warp * 16 + g + 8] = l1;
  }
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) {
    *reinterpret_cast<float2*>(co + (warp * 16 + g) * kDim + 8 * nd + 2 * t) = make_float2(o[nd][0], o[nd][1]);
    *reinterpret_cast<float2*>(co + (warp * 16 + g + 8) * kDim + 8 * nd + 2 * t) = make_float2(o[nd][2], o[nd][3]);
  }
  __syncthreads();
  const int hh = tid >> 3, d0 = (tid & 7) * 16;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < 4; ++w) M = fmaxf(M, cm[w * 16 + hh]);
  float wgt[4], L = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    wgt[w] = M == -INFINITY ? 0.f : exp2f(cm[w * 16 + hh] - M);
    L += wgt[w] * cl[w * 16 + hh];
  }
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) a += wgt[w] * co[(w * 16 + hh) * kDim + d0 + j];
    acc[j] = a;
  }
  if (p.nsplit == 1) {
    if (hh < p.group) {
      const float f = L > 0.f ? out_scale / L : 0.f;
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2(acc[2 * j] * f, acc[2 * j + 1] * f);
      uint16_t* dst = static_cast<uint16_t*>(p.out) + (token * hq + static_cast<int64_t>(h) * p.group + hh) * kDim + d0;
      reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  } else {
    const int64_t unit = static_cast<int64_t>(row) * p.nsplit + split;
    float* wo = p.ws + (unit * 16 + hh) * kDim + d0;
#pragma unroll
    for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4*>(wo + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
    if ((tid & 7) == 0) {
      float* wml = p.ws + static_cast<int64_t>(p.num_rows) * p.nsplit * 16 * kDim + (unit * 16 + hh) * 2;
      wml[0] = M;
      wml[1] = L;
    }
  }
}

// combine the splits of a row: one CTA per row, thread = dim
__global__ void __launch_bounds__(128) sparse_pa_merge_kernel(SparsePaParams p, float out_scale) {
  const int row = blockIdx.x, d = threadIdx.x;
  const int h = row % p.hkv;
  const int64_t token = row / p.hkv;
  const int hq = p.hkv * p.group;
  const float* ml = p.ws + static_cast<int64_t>(p.num_rows) * p.nsplit * 16 * kDim;
  for (int hh = 0; hh < p.group; ++hh) {
    float M = -INFINITY;
    for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, ml[((static_cast<int64_t>(row) * p.nsplit + s) * 16 + hh) * 2]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < p.nsplit; ++s) {
        const int64_t unit = static_cast<int64_t>(row) * p.nsplit + s;
        const float m = ml[(unit * 16 + hh) * 2];
        if (m == -INFINITY) continue;
        const float w = exp2f(m - M);
        L += w * ml[(unit * 16 + hh) * 2 + 1];
        O += w * p.ws[(unit * 16 + hh) * kDim + d];
      }
    }
    const float v = L > 0.f ? O * (out_scale / L) : 0.f;
    reinterpret_cast<__nv_bfloat16*>(p.out)[(token * hq + static_cast<int64_t>(h) * p.group + hh) * kDim + d] =
        __float2bfloat16_rn(v);
  }
}

template <int KV>
cudaError_t launch_kv(const SparsePaParams& p, cudaStream_t s, int* launches) {
  constexpr int bytes = pa_smem_bytes<KV>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(sparse_pa_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const float kfold = KV == BSP_FP8_E4M3 ? p.k_scale * 256.f : 1.f;
  const float vfold = KV == BSP_FP8_E4M3 ? p.v_scale * 256.f : 1.f;
  const float qk_scale = p.sm_scale * kfold * kLog2e;
  const int64_t ctas = static_cast<int64_t>(p.num_rows) * p.nsplit;
  sparse_pa_kernel<KV><<<static_cast<unsigned>(ctas), 128, bytes, s>>>(p, qk_scale, vfold);
  ++*launches;
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess || p.nsplit == 1) return e;
  sparse_pa_merge_kernel<<<p.num_rows, 128, 0, s>>>(p, vfold);
  ++*launches;
  return cudaPeekAtLastError();
}

}  // namespace

void sparse_pa_plan(int32_t num_rows, int32_t k_pages, int num_sms, int32_t* nsplit, int32_t* pages_per_split) {
  int64_t rows = num_rows > 0 ? num_rows : 1;
  int64_t ns = (4LL * num_sms + rows - 1) / rows;
  const int64_t max_ns = (k_pages + 3) / 4;
  ns = ns < 1 ? 1 : (ns > max_ns ? max_ns : ns);
  int64_t pps = (k_pages + ns - 1) / ns;
  pps = (pps + 3) / 4 * 4;
  if (pps < 4) pps = 4;
  ns = (k_pages + pps - 1) / pps;
  if (ns < 1) ns = 1;
  *nsplit = static_cast<int32_t>(ns);
  *pages_per_split = static_cast<int32_t>(pps);
}

size_t sparse_pa_ws_bytes(int32_t num_rows, int32_t nsplit) {
  if (nsplit <= 1) return 0;
  return static_cast<size_t>(num_rows) * nsplit * 16 * (kDim + 2) * sizeof(float);
}

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
