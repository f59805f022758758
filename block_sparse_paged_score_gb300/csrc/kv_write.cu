// kv_write.cu -- a1: quantise new tokens and scatter them into the caches
// (ROCm/ATOM PR 2962, commit "... index key": the fused writer stores K, V and
// the index key straight onto the pool pages; vLLM PR 61889, Details:
// per-tensor fp8 scales), the writer's unit-scale e4m3 query cast, and the
// row-length helpers with the pad-row clamp (ATOM PR 2962, B12).
//
// One warp per (token, head, side); lane l owns dims 4l..4l+3, so a 32-element
// MXFP4 group is 8 lanes and its amax is an 8-lane shuffle reduction.  The
// page addresses follow the interleaved layout of vLLM PR 61889 (K page
// [128/x][16][x], V page [16/x][128][x] at V-base = K-base + 8 page slots) and
// the 8704 B MXFP4 field.  The writer is built without fast-math: divisions
// are IEEE round-to-nearest, so its bytes are reproducible bit for bit.
#include "common.cuh"
#include "kernels.h"

namespace bsp {

namespace {

// Shared exponent of an MXFP4 group: clamp(floor(log2(amax)) - 2, -127, 127),
// floor(log2) read exactly off the fp32 bits (OCP MX v1.0 rule).
__device__ __forceinline__ int mx_shared_exp(float amax) {
  uint32_t b = __float_as_uint(amax);
  if (b == 0) return -127;
  int ex = (b >> 23) & 0xFF;
  int E = ex ? ex - 127 : (31 - __clz(b & 0x7FFFFFu)) - 149;
  int e = E - 2;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Write dims 4*lane..+3 of token o of an MXFP4 field.
__device__ __forceinline__ void write_mx(uint8_t* field, int o, int lane, const float (&x)[4]) {
  float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
  int e = mx_shared_exp(a);
  float sc = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, normal for e in [-127, 125]
  uint32_t lo = float2_to_e2m1x2(x[0] * sc, x[1] * sc);
  uint32_t hi = float2_to_e2m1x2(x[2] * sc, x[3] * sc);
  *reinterpret_cast<uint16_t*>(field + o * 64 + 2 * lane) = static_cast<uint16_t>(lo | (hi << 8));
  if ((lane & 7) == 0) field[kMxScaleOff + o * 4 + (lane >> 3)] = static_cast<uint8_t>(e + 127);
}

__device__ __forceinline__ void kv_page_write_block(const KvWriteParams& p, int64_t block_idx) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = block_idx * 4 + (threadIdx.x >> 5);
  const int units = 2 * p.hkv + p.hidx;
  const int64_t token = gw / units;
  const int u = static_cast<int>(gw % units);
  if (token >= p.num_tokens) return;
  const int64_t slot = p.slot[token];
  if (slot < 0) return;
  const int64_t block = slot / kBlock;
  const int o = static_cast<int>(slot % kBlock);

  int side, h;  // side 0 K, 1 V, 2 index key
  if (u < p.hkv) {
    side = 0, h = u;
  } else if (u < 2 * p.hkv) {
    side = 1, h = u - p.hkv;
  } else {
    side = 2, h = u - 2 * p.hkv;
  }
  const int64_t nblk = side == 2 ? p.idx_num_blocks : p.num_blocks;
  if (block >= nblk) {
    if (lane == 0) set_err(p.err, BSP_DEVERR_SLOT);
    return;
  }
  const uint16_t* src = side == 0 ? p.k : (side == 1 ? p.v : p.idx_k);
  const int heads = side == 2 ? p.hidx : p.hkv;
  const uint2 raw = *reinterpret_cast<const uint2*>(src + (token * heads + h) * kDim + 4 * lane);
  float x[4] = {bf16_bits_to_float(raw.x & 0xFFFF), bf16_bits_to_float(raw.x >> 16),
                bf16_bits_to_float(raw.y & 0xFFFF), bf16_bits_to_float(raw.y >> 16)};

  if (side == 2) {
    uint8_t* field = p.idx_base + block * p.idx_block_stride +
                     static_cast<int64_t>(h) *
                         (p.idx_dtype == BSP_BF16 ? kBf16IndexField
                                                  : (p.idx_dtype == BSP_FP8_E4M3 ? kFp8IndexField : kMxField));
    if (p.idx_dtype == BSP_BF16) {
      *reinterpret_cast<uint2*>(field + o * 256 + 8 * lane) = raw;
    } else if (p.idx_dtype == BSP_FP8_E4M3) {
      float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
      const float s = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
      uint32_t w = float2_to_e4m3x2(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s)) |
                   (float2_to_e4m3x2(__fdiv_rn(x[2], s), __fdiv_rn(x[3], s)) << 16);
      *reinterpret_cast<uint32_t*>(field + o * 128 + 4 * lane) = w;
      if (lane == 0) *reinterpret_cast<float*>(field + kFp8IndexScaleOff + o * 4) = s;
    } else {
      write_mx(field, o, lane, x);
    }
    return;
  }

  uint8_t* base = side == 0 ? p.k_base : p.v_base;
  if (p.kv_dtype == BSP_MXFP4) {
    write_mx(base + block * p.id_stride + static_cast<int64_t>(h) * kMxField, o, lane, x);
    return;
  }
  const int64_t page_id = block * 16 + o / kPage;
  const int t = o % kPage;
  const int d0 = 4 * lane;
  if (p.kv_dtype == BSP_FP8_E4M3) {
    uint8_t* page = base + page_id * p.id_stride + static_cast<int64_t>(h) * 2048;
    const float sc = side == 0 ? p.k_scale : p.v_scale;
    uint32_t w = float2_to_e4m3x2(__fdiv_rn(x[0], sc), __fdiv_rn(x[1], sc)) |
                 (float2_to_e4m3x2(__fdiv_rn(x[2], sc), __fdiv_rn(x[3], sc)) << 16);
    if (side == 0) {  // K [d/16][t][16]
      *reinterpret_cast<uint32_t*>(page + (d0 >> 4) * 256 + t * 16 + (d0 & 15)) = w;
    } else {  // V [d][16 t]
#pragma unroll
      for (int i = 0; i < 4; ++i) page[(d0 + i) * 16 + t] = static_cast<uint8_t>(w >> (8 * i));
    }
  } else {  // bf16: K [d/8][t][8], V [t/8][d][8]
    uint16_t* page = reinterpret_cast<uint16_t*>(base + page_id * p.id_stride + static_cast<int64_t>(h) * 4096);
    if (side == 0) {
      *reinterpret_cast<uint2*>(page + (d0 >> 3) * 128 + t * 8 + (d0 & 7)) = raw;
    } else {
      const uint16_t e[4] = {static_cast<uint16_t>(raw.x & 0xFFFF), static_cast<uint16_t>(raw.x >> 16),
                             static_cast<uint16_t>(raw.y & 0xFFFF), static_cast<uint16_t>(raw.y >> 16)};
#pragma unroll
      for (int i = 0; i < 4; ++i) page[(t >> 3) * 1024 + (d0 + i) * 8 + (t & 7)] = e[i];
    }
  }
}

__global__ void __launch_bounds__(128) kv_page_write_kernel(KvWriteParams p) {
  pdl_wait();
  pdl_trigger();
  kv_page_write_block(p, blockIdx.x);
}

// 8 elements per thread, 128 threads per block
__device__ __forceinline__ void cast_e4m3_block(const uint16_t* __restrict__ x, uint8_t* __restrict__ out, int64_t n,
                                                int64_t block_idx) {
  const int64_t i = (block_idx * 128 + threadIdx.x) * 8;
  if (i + 8 <= n) {
    const uint4 v = *reinterpret_cast<const uint4*>(x + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t r[2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
      r[j] = float2_to_e4m3x2(bf16_bits_to_float(w[2 * j] & 0xFFFF), bf16_bits_to_float(w[2 * j] >> 16)) |
             (float2_to_e4m3x2(bf16_bits_to_float(w[2 * j + 1] & 0xFFFF),
                               bf16_bits_to_float(w[2 * j + 1] >> 16))
              << 16);
    *reinterpret_cast<uint2*>(out + i) = make_uint2(r[0], r[1]);
  } else {
    for (int64_t j = i; j < n; ++j) out[j] = static_cast<uint8_t>(float2_to_e4m3x2(bf16_bits_to_float(x[j]), 0.f));
  }
}

__global__ void __launch_bounds__(128) cast_e4m3_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ out,
                                                        int64_t n) {
  pdl_wait();
  pdl_trigger();
  cast_e4m3_block(x, out, n, blockIdx.x);
}

// 128 rows per block
__device__ __forceinline__ void row_lengths_decode_block(const int32_t* seq_lens, int32_t num_seqs, int32_t q_len,
                                                         int32_t heads, int32_t* row_seq, int32_t* row_len,
                                                         int64_t block_idx) {
  const int64_t r = block_idx * 128 + threadIdx.x;
  const int64_t rows = static_cast<int64_t>(num_seqs) * q_len * heads;
  if (r >= rows) return;
  const int64_t token = r / heads;
  const int s = static_cast<int>(token / q_len), j = static_cast<int>(token % q_len);
  const int64_t L = static_cast<int64_t>(seq_lens[s]) - (q_len - 1 - j);
  row_seq[r] = s;
  row_len[r] = static_cast<int32_t>(L < 0 ? 0 : L);
}

__global__ void __launch_bounds__(128) row_lengths_decode_kernel(const int32_t* seq_lens, int32_t num_seqs,
                                                                 int32_t q_len, int32_t heads, int32_t* row_seq,
                                                                 int32_t* row_len) {
  pdl_wait();
  pdl_trigger();
  row_lengths_decode_block(seq_lens, num_seqs, q_len, heads, row_seq, row_len, blockIdx.x);
}

// The decode step's preparation in one launch: blocks [0, w) write the new
// tokens, the next blocks cast the two query tensors to e4m3, the last ones
// compute the row lengths.  The parts are independent.
__global__ void __launch_bounds__(128) decode_prep_kernel(DecodePrepParams p) {
  pdl_wait();
  pdl_trigger();
  int64_t b = blockIdx.x;
  if (b < p.write_blocks) return kv_page_write_block(p.write, b);
  b -= p.write_blocks;
  for (int c = 0; c < 2; ++c) {
    if (b < p.cast_blocks[c]) return cast_e4m3_block(p.cast_src[c], p.cast_dst[c], p.cast_n[c], b);
    b -= p.cast_blocks[c];
  }
  row_lengths_decode_block(p.seq_lens, p.num_seqs, p.q_len, p.heads, p.row_seq, p.row_len, b);
}

__global__ void row_lengths_prefill_kernel(const int32_t* req, const int32_t* pos, int32_t n, int32_t heads,
                                           int32_t* row_seq, int32_t* row_len) {
  pdl_wait();
  pdl_trigger();
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= static_cast<int64_t>(n) * heads) return;
  const int64_t i = r / heads;
  const int64_t L = static_cast<int64_t>(pos[i]) + 1;
  row_seq[r] = req[i];
  row_len[r] = static_cast<int32_t>(L < 0 ? 0 : L);
}

}  // namespace

cudaError_t launch_kv_page_write(const KvWriteParams& p, cudaStream_t s) {
  const int64_t warps = static_cast<int64_t>(p.num_tokens) * (2 * p.hkv + p.hidx);
  if (warps == 0) return cudaSuccess;
  const cudaError_t e = launch_kernel(kv_page_write_kernel, dim3(static_cast<unsigned>((warps + 3) / 4)), dim3(128), 0,
                                      s, 0, p);
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

cudaError_t launch_cast_e4m3(const uint16_t* x, uint8_t* out, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const cudaError_t e =
      launch_kernel(cast_e4m3_kernel, dim3(static_cast<unsigned>((n + 1023) / 1024)), dim3(128), 0, s, 0, x, out, n);
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

cudaError_t launch_row_lengths_decode(const int32_t* seq_lens, int32_t num_seqs, int32_t q_len, int32_t heads,
                                      int32_t* row_seq, int32_t* row_len, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(num_seqs) * q_len * heads;
  if (rows == 0) return cudaSuccess;
  const cudaError_t e = launch_kernel(row_lengths_decode_kernel, dim3(static_cast<unsigned>((rows + 127) / 128)),
                                      dim3(128), 0, s, 0, seq_lens, num_seqs, q_len, heads, row_seq, row_len);
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

cudaError_t launch_decode_prep(DecodePrepParams p, cudaStream_t s) {
  p.write_blocks = (static_cast<int64_t>(p.write.num_tokens) * (2 * p.write.hkv + p.write.hidx) + 3) / 4;
  for (int c = 0; c < 2; ++c) p.cast_blocks[c] = p.cast_src[c] ? (p.cast_n[c] + 1023) / 1024 : 0;
  const int64_t rows = static_cast<int64_t>(p.num_seqs) * p.q_len * p.heads;
  const int64_t total = p.write_blocks + p.cast_blocks[0] + p.cast_blocks[1] + (rows + 127) / 128;
  if (total == 0) return cudaSuccess;
  const cudaError_t e = launch_kernel(decode_prep_kernel, dim3(static_cast<unsigned>(total)), dim3(128), 0, s, 0, p);
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

cudaError_t launch_row_lengths_prefill(const int32_t* req, const int32_t* pos, int32_t n, int32_t heads,
                                       int32_t* row_seq, int32_t* row_len, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(n) * heads;
  if (rows == 0) return cudaSuccess;
  const cudaError_t e = launch_kernel(row_lengths_prefill_kernel, dim3(static_cast<unsigned>((rows + 255) / 256)),
                                      dim3(256), 0, s, 0, req, pos, n, heads, row_seq, row_len);
  return e != cudaSuccess ? e : cudaPeekAtLastError();
}

}  // namespace bsp
