// bench_micro.cu -- microbenchmarks of the GB300 units the sparse path's
// kernels are built on: the roofline denominators and instruction choices
// behind them (run by bench_micro.py, not part of libbsp).
//   gather      4 KB page pairs (2 KB K + 2 KB V, 16 KB apart) gathered by
//               1-D TMA bulk copies into per-warp shared-memory rings, from
//               a pool that fits L2 or one that does not: the data-movement
//               ceiling of an attention that reads selected pages
//   stream      read-only streams over a 4 GB pool, every byte once: plain
//               16-byte loads, 4 KB page pairs by the gather kernel, and
//               whole 16.5 KB chunks through a CTA ring (thread 0 copies,
//               the CTA syncs per chunk)
//   tma_ring    the prefill scorer's key-tile loads alone: two 16 KB boxes a
//               tile into a ring of one CTA per SM, 2-D tensor loads with
//               128-byte swizzle against 1-D bulk copies of the same bytes
//   mma_sync    legacy warp MMA rates: m16n8k16 f16 and m16n8k32 e4m3
//   umma        tcgen05.mma rate from one issuing thread, M = 128 and N =
//               16 ... 256 (kind::f16, K = 16; kind::f8f6f4 e4m3, K = 32),
//               and N = 16 into 1 ... 16 independent accumulators
//   cvt         cvt.rn.f16x2.e4m3x2 throughput (the fp8 -> f16 conversion)
//   sf_layout   where kind::mxf8f6f4.block_scale reads its e8m0 scale
//               factors in TMEM (scale_vec::1X, M = N = 128)
#include <cuda_runtime.h>
#include <stdint.h>

#include "block_sparse_paged_score_gb300/csrc/common.cuh"
#include "block_sparse_paged_score_gb300/csrc/tcgen05.cuh"

using namespace bsp;

template <int R>
__global__ void __launch_bounds__(128) gather_kernel(const uint8_t* pool, const int32_t* ids, int pages_per_row,
                                                      uint32_t* sink, int32_t* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 4 * R * 4096);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 4 * R; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
  __syncthreads();
  const int32_t* rid = ids + static_cast<int64_t>(blockIdx.x) * pages_per_row;
  const int nw = pages_per_row / 4;
  uint8_t* ring = smem + warp * R * 4096;
  uint64_t* wb = bars + warp * R;
  auto issue = [&](int32_t id, uint8_t* slot, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, 4096);
    bulk_g2s(slot, pool + static_cast<int64_t>(id) * 2048, 2048, bar);
    bulk_g2s(slot + 2048, pool + static_cast<int64_t>(id + 8) * 2048, 2048, bar);
  };
  if (lane == 0)
    for (int i = 0; i < R && i < nw; ++i) issue(rid[warp + 4 * i], ring + i * 4096, &wb[i]);
  uint32_t acc = 0;
  int st = 0;
  uint32_t ph = 0;
  bool alive = true;
  for (int i = 0; i < nw; ++i) {
    if (alive) alive = mbar_wait(&wb[st], ph, err);
    const uint4 v = *reinterpret_cast<const uint4*>(ring + st * 4096 + lane * 128);
    acc ^= v.x ^ v.w;
    __syncwarp();
    if (lane == 0 && i + R < nw) {
      fence_proxy_async();
      issue(rid[warp + 4 * (i + R)], ring + st * 4096, &wb[st]);
    }
    if (++st == R) st = 0, ph ^= 1;
  }
  sink[static_cast<int64_t>(blockIdx.x) * 128 + tid] = acc;
}

// Read-only streams that touch every byte of the pool once (no L2 reuse):
// plain 16-byte loads in a grid-stride loop, four in flight per thread
__global__ void __launch_bounds__(256) stream_ld_kernel(const uint4* pool, int64_t n16, uint32_t* sink) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  uint32_t acc = 0;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldcs(pool + i), b = __ldcs(pool + i + stride), c = __ldcs(pool + i + 2 * stride),
                d = __ldcs(pool + i + 3 * stride);
    acc ^= a.x ^ b.y ^ c.z ^ d.w;
  }
  for (; i < n16; i += stride) acc ^= __ldcs(pool + i).x;
  sink[static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x] = acc;
}

// whole chunks (one bulk copy each, issued by thread 0) through a CTA ring
// of S stages; every warp waits for the stage, the CTA syncs, thread 0
// refills it: a streaming scorer's data movement without its arithmetic
__global__ void __launch_bounds__(128) chunk_kernel(const uint8_t* pool, const int32_t* ids, int chunks_per_cta,
                                                    int chunk, int S, uint32_t* sink, int32_t* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * chunk);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
  __syncthreads();
  const int32_t* cid = ids + static_cast<int64_t>(blockIdx.x) * chunks_per_cta;
  auto issue = [&](int i) {
    const int st = i % S;
    mbar_arrive_expect_tx(&bars[st], chunk);
    bulk_g2s(smem + st * chunk, pool + static_cast<int64_t>(cid[i]) * chunk, chunk, &bars[st]);
  };
  if (tid == 0)
    for (int i = 0; i < S && i < chunks_per_cta; ++i) issue(i);
  uint32_t acc = 0;
  bool alive = true;
  for (int i = 0; i < chunks_per_cta; ++i) {
    const int st = i % S;
    if (alive) alive = mbar_wait(&bars[st], (i / S) & 1, err);
    acc ^= *reinterpret_cast<const uint32_t*>(smem + st * chunk + tid * 4);
    __syncthreads();
    if (tid == 0 && i + S < chunks_per_cta) {
      fence_proxy_async();
      issue(i + S);
    }
  }
  sink[static_cast<int64_t>(blockIdx.x) * 128 + tid] = acc;
}

// Key tiles as the prefill scorer loads them: each tile is two 16 KB boxes
// (128 rows x 128 B) at block rows of the pool, into a ring of S stages of
// one CTA; thread 0 issues, waits for the stage S tiles back and reissues.
// mode 0: 2-D tensor loads (128-byte swizzle), mode 1: 1-D bulk copies of
// the same 16 KB.
__global__ void __launch_bounds__(32, 1) tma_ring_kernel(const __grid_constant__ CUtensorMap map, const uint8_t* pool,
                                                         const int32_t* rows, int tiles, int S, int mode,
                                                         uint32_t* sink, int32_t* err) {
  extern __shared__ uint8_t raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(S) * 32768);
  if (threadIdx.x != 0) return;
  for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
  mbar_fence_init();
  const int32_t* r = rows + static_cast<int64_t>(blockIdx.x) * tiles * 2;
  auto issue = [&](int j) {
    const int st = j % S;
    mbar_arrive_expect_tx(&bars[st], 32768);
    for (int h = 0; h < 2; ++h) {
      uint8_t* dst = ring + static_cast<size_t>(st) * 32768 + h * 16384;
      if (mode == 0)
        tma_load_2d(dst, &map, 0, r[2 * j + h], &bars[st]);
      else
        bulk_g2s(dst, pool + static_cast<int64_t>(r[2 * j + h]) * 128, 16384, &bars[st]);
    }
  };
  for (int j = 0; j < S && j < tiles; ++j) issue(j);
  uint32_t acc = 0;
  bool alive = true;
  for (int j = 0; j < tiles; ++j) {
    const int st = j % S;
    if (alive) alive = mbar_wait(&bars[st], (j / S) & 1, err);
    acc ^= *reinterpret_cast<const uint32_t*>(ring + static_cast<size_t>(st) * 32768 + (j & 63) * 4);
    if (j + S < tiles) {
      fence_proxy_async();
      issue(j + S);
    }
  }
  sink[blockIdx.x] = acc;
}

__global__ void __launch_bounds__(256) mma_sync_kernel(int iters, float* out) {
  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  const uint32_t a0 = pack_f16x2(threadIdx.x * 1e-3f, 0.5f), a1 = pack_f16x2(0.25f, threadIdx.x * 2e-3f);
  const uint32_t b0 = pack_f16x2(0.125f, 0.5f), b1 = pack_f16x2(1.f, -0.5f);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) mma_f16(acc[j], a0, a1, a1, a0, b0, b1);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += acc[j][0] + acc[j][1] + acc[j][2] + acc[j][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void __launch_bounds__(256) mma_sync_e4m3_kernel(int iters, float* out) {
  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  const uint32_t a0 = 0x38383838u ^ threadIdx.x, a1 = 0x30303030u;
  const uint32_t b0 = 0x38303830u, b1 = 0x28382838u;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) mma_e4m3(acc[j], a0, a1, a1, a0, b0, b1);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += acc[j][0] + acc[j][1] + acc[j][2] + acc[j][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// no-swizzle K-major descriptor: core matrices 8 rows x 16 B, LBO along K, SBO along M/N
__device__ __forceinline__ uint64_t desc_noswz(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>((lbo & 0x3FFFF) >> 4) << 16;
  d |= static_cast<uint64_t>((sbo & 0x3FFFF) >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// kind: 0 = f16 (K 16), 1 = f8f6f4 e4m3 (K 32); n columns (16..256, power of two for the alloc)
__global__ void __launch_bounds__(128, 1) umma_kernel(int iters, int n, int kind, int32_t* err, uint32_t* sink) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t done_bar;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < 16384; i += 128) reinterpret_cast<uint32_t*>(smem)[i] = 0x3C003C00u;  // 64 KB of 1.0h
  if (tid == 0) {
    mbar_init(&done_bar, 1);
    mbar_fence_init();
  }
  fence_proxy_async();
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(&tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_slot;
  if (tid == 0) {
    const uint32_t a = smem_u32(smem), b = smem_u32(smem + 16384);
    const uint32_t idesc = (1u << 4) | ((static_cast<uint32_t>(n) >> 3) << 17) | ((128u >> 4) << 24);
    const uint64_t ad = desc_noswz(a, 128, 256), bd = desc_noswz(b, 128, 256);
    for (int i = 0; i < iters; ++i) {
      if (kind == 0)
        umma_f16(tmem, ad, bd, idesc, i > 0);
      else
        umma_f8(tmem, ad, bd, idesc, i > 0);
    }
    umma_commit(&done_bar);
  }
  __syncwarp();
  mbar_wait(&done_bar, 0, err);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  float v[8];
  tmem_ld8(tmem + (static_cast<uint32_t>(32 * warp) << 16), v);
  sink[blockIdx.x * 128 + tid] = __float_as_uint(v[0]);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem));
  }
}


// fp8 -> f16 conversions: 8 independent cvt.rn.f16x2.e4m3x2 streams per thread
__global__ void __launch_bounds__(256) cvt_kernel(int iters, uint32_t* out) {
  uint32_t x[8], acc = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = 0x38303830u + threadIdx.x * 0x01010101u + j;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t r;
      const uint16_t in = static_cast<uint16_t>(x[j]);
      asm volatile("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
      x[j] = (x[j] & 0xFFFF0000u) | (r & 0x7F7Fu);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) acc ^= x[j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

// tcgen05 kind::f16 M=128 N=16 K=16 into `nacc` independent accumulators in turn
__global__ void __launch_bounds__(128, 1) umma_multi_kernel(int iters, int nacc, int32_t* err, uint32_t* sink) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t done_bar;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < 16384; i += 128) reinterpret_cast<uint32_t*>(smem)[i] = 0x3C003C00u;
  if (tid == 0) {
    mbar_init(&done_bar, 1);
    mbar_fence_init();
  }
  fence_proxy_async();
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(&tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_slot;
  if (tid == 0) {
    const uint32_t a = smem_u32(smem), b = smem_u32(smem + 16384);
    const uint32_t idesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
    const uint64_t ad = desc_noswz(a, 128, 256), bd = desc_noswz(b, 128, 256);
    for (int i = 0; i < iters; ++i) {
      const int c = i % nacc;
      umma_f16(tmem + 16 * c, ad, bd, idesc, i >= nacc);
    }
    umma_commit(&done_bar);
  }
  __syncwarp();
  mbar_wait(&done_bar, 0, err);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  float v[8];
  tmem_ld8(tmem + (static_cast<uint32_t>(32 * warp) << 16), v);
  sink[blockIdx.x * 128 + tid] = __float_as_uint(v[0]);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem));
  }
}

// sf_layout: every operand value 1.0, so D = 32 * 2^(sa-127) * 2^(sb-127).
// sa_words[128][8], sb_words[128][8]: the 32-bit cells written to lane i,
// columns 256..263 (A's scale factors) and 288..295 (B's).
__global__ void __launch_bounds__(128, 1) sf_layout_kernel(const uint32_t* sa_words, const uint32_t* sb_words, int a_sf_id,
                                                    int b_sf_id, float* out, int32_t* err) {
  // large operand buffers of one value each: any reading of the descriptors
  // within them sees 1.0
  __shared__ __align__(1024) uint8_t a[16384];
  __shared__ __align__(1024) uint8_t b[16384];
  __shared__ uint64_t bar;
  __shared__ uint32_t slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < 16384; i += 128) {
    a[i] = 0x38;  // e4m3 1.0
    b[i] = 0x22;  // two e2m1 1.0 (padding bytes too)
  }
  fence_proxy_async();
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = slot;
  const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
  // A scales in columns 256..263, B scales in columns 288..295
  for (int c = 0; c < 8; ++c) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tmem + lane_base + 256 + c),
                 "r"(sa_words[tid * 8 + c])
                 : "memory");
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tmem + lane_base + 288 + c),
                 "r"(sb_words[tid * 8 + c])
                 : "memory");
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (tid == 0) {
    // M = 128, N = 128, K = 32; A e4m3, B e2m1, scales e8m0
    const uint32_t idesc = idesc_mxf8f6f4(kFmtE4m3, kFmtE2m1, 128, 128, a_sf_id, b_sf_id);
    const uint64_t ad = desc_noswz(smem_u32(a), 128, 256), bd = desc_noswz(smem_u32(b), 128, 256);
    umma_mx(tmem, ad, bd, idesc, tmem + 256, tmem + 288, 0);
    umma_commit(&bar);
  }
  __syncwarp();
  mbar_wait(&bar, 0, err);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  for (int c = 0; c < 128; c += 32) {
    float v[32];
    tmem_ld32(tmem + lane_base + c, v);
    for (int i = 0; i < 32; ++i) out[tid * 128 + c + i] = v[i];
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

extern "C" {

int micro_gather(const void* pool, const int32_t* ids, int rows, int pages_per_row, int ring, uint32_t* sink,
                 int32_t* err, cudaStream_t s) {
  const int smem = 4 * ring * 4096 + 4 * ring * 8;
  cudaError_t e;
#define G(R)                                                                                          \
  case R:                                                                                             \
    e = cudaFuncSetAttribute(gather_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);   \
    if (e) return e;                                                                                  \
    gather_kernel<R><<<rows, 128, smem, s>>>(static_cast<const uint8_t*>(pool), ids, pages_per_row, sink, err); \
    break;
  switch (ring) {
    G(2) G(3) G(4) G(6) default : return -1;
  }
  return cudaGetLastError();
}

int micro_stream_ld(const void* pool, int64_t bytes, int ctas, uint32_t* sink, cudaStream_t s) {
  stream_ld_kernel<<<ctas, 256, 0, s>>>(static_cast<const uint4*>(pool), bytes / 16, sink);
  return cudaGetLastError();
}

int micro_chunk(const void* pool, const int32_t* ids, int ctas, int chunks_per_cta, int chunk, int stages,
                uint32_t* sink, int32_t* err, cudaStream_t s) {
  if (chunk % 16 || chunk < 512 || stages < 1) return -1;
  const int smem = stages * chunk + stages * 8;
  if (smem > 227 * 1024) return -1;
  cudaError_t e = cudaFuncSetAttribute(chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e) return e;
  chunk_kernel<<<ctas, 128, smem, s>>>(static_cast<const uint8_t*>(pool), ids, chunks_per_cta, chunk, stages, sink,
                                        err);
  return cudaGetLastError();
}

int micro_tma_ring(const void* pool, int64_t bytes, const int32_t* rows, int ctas, int tiles, int stages, int mode,
                   uint32_t* sink, int32_t* err, cudaStream_t s) {
  if (stages < 1 || stages > 6) return -1;
  CUtensorMap map;
  if (!make_map_u8(&map, pool, static_cast<uint64_t>(bytes / 128))) return -2;
  const int smem = 1024 + stages * 32768 + stages * 8;
  cudaError_t e = cudaFuncSetAttribute(tma_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e) return e;
  tma_ring_kernel<<<ctas, 32, smem, s>>>(map, static_cast<const uint8_t*>(pool), rows, tiles, stages, mode, sink, err);
  return cudaGetLastError();
}

int micro_mma_sync(int ctas, int iters, float* out, int e4m3, cudaStream_t s) {
  if (e4m3)
    mma_sync_e4m3_kernel<<<ctas, 256, 0, s>>>(iters, out);
  else
    mma_sync_kernel<<<ctas, 256, 0, s>>>(iters, out);
  return cudaGetLastError();
}

int micro_umma(int ctas, int iters, int n, int kind, int32_t* err, uint32_t* sink, cudaStream_t s) {
  const int smem = 128 * 1024;
  cudaError_t e = cudaFuncSetAttribute(umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e) return e;
  umma_kernel<<<ctas, 128, smem, s>>>(iters, n, kind, err, sink);
  return cudaGetLastError();
}

int micro_cvt(int ctas, int iters, uint32_t* out, cudaStream_t s) {
  cvt_kernel<<<ctas, 256, 0, s>>>(iters, out);
  return cudaGetLastError();
}

int micro_umma_multi(int ctas, int iters, int nacc, int32_t* err, uint32_t* sink, cudaStream_t s) {
  if (nacc < 1 || nacc > 16) return -1;
  const int smem = 128 * 1024;
  cudaError_t e = cudaFuncSetAttribute(umma_multi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e) return e;
  umma_multi_kernel<<<ctas, 128, smem, s>>>(iters, nacc, err, sink);
  return cudaGetLastError();
}
}

extern "C" int micro_sf_layout(const uint32_t* sa, const uint32_t* sb, int a_id, int b_id, float* out, int32_t* err,
                               cudaStream_t s) {
  sf_layout_kernel<<<1, 128, 0, s>>>(sa, sb, a_id, b_id, out, err);
  return cudaGetLastError();
}
