// common.cuh -- device helpers shared by the sm_103a kernels of libbsp:
// sizes of the cache formats, inline-PTX wrappers for mbarriers, 1-D TMA bulk
// copies, mma.sync / ldmatrix, and conversions of the stored number formats.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bsp.h"

namespace bsp {

// 128-token blocks, 16-token pages, 8 pages per block side, head_dim 128
// (vLLM PR 61889, Validation: K view [.., 8, 16, 16] and V view
// [.., 1, 128, 16]; server command --block-size 128).
constexpr int kBlock = 128;
constexpr int kPage = 16;
constexpr int kPagesPerSide = 8;
constexpr int kDim = 128;
// MXFP4 field: 128 tokens x 64 B e2m1 + 128 x 4 B e8m0 (ROCm/ATOM PR 2962).
constexpr int kMxField = 8704;
constexpr int kMxScaleOff = 8192;
// fp8 index field: 128 x 128 B e4m3 + 128 x 4 B fp32 per-token scale.
constexpr int kFp8IndexField = 16896;
constexpr int kFp8IndexScaleOff = 16384;
constexpr int kBf16IndexField = 32768;

// The longest a kernel waits for one of its own TMA copies before it gives
// up, reports BSP_DEVERR_TIMEOUT and carries on (~1 s of try_wait rounds).
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ void set_err(int32_t* err, int bit) {
  if (err) atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier -----------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// plain arrival (no transaction bytes): completes a phase that no copy fills
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Bounded wait on a phase; returns false (and flags the error) on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* err) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  set_err(err, BSP_DEVERR_TIMEOUT);
  return false;
}
// The same with each round allowed to suspend the thread for up to 1 us
// while the phase is incomplete (the try_wait suspend-time hint; the thread
// resumes as soon as the phase completes), for barriers that many warps of a
// CTA wait on at once: the waiting warps then take fewer issue slots from the
// ones that work.  About the same overall bound as mbar_wait.
constexpr uint32_t kSleepNs = 1000;
constexpr uint32_t kSleepWaitLimit = 1u << 20;
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, int32_t* err) {
  for (uint32_t i = 0; i < kSleepWaitLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSleepNs)
        : "memory");
    if (ok) return true;
  }
  set_err(err, BSP_DEVERR_TIMEOUT);
  return false;
}

// ---- TMA bulk copies (1-D, global -> shared, completion on an mbarrier) ----
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tensor cores (mma.sync) ------------------------------------------------
// D (16x8 f32) += A (16x16, row) * B (16x8, col); fragments as in the PTX ISA.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D (16x8 f32) += A (16x32 e4m3, row) * B (32x8 e4m3, col): a0/a1 rows g and
// g+8 at k 4t..4t+3, a2/a3 the same rows at k 16+4t..; b0 k 4t.., b1 k 16+4t..
// of column g (one byte per element, the lowest k in the low byte).
__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Four 8x(16 B) matrices; lane l supplies the address of row l%8 of matrix
// l/8 and receives 4 bytes of row l/4 of each matrix (bytes 4*(l%4)..+3).
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// ---- conversions ------------------------------------------------------------
// Four e4m3 bytes -> two f16x2 holding each value times 2^-8, exactly: the
// 7 magnitude bits move under the f16 exponent/mantissa fields (the 4-bit
// e4m3 exponent becomes a biased f16 exponent 8 lower, subnormals included).
// lo = (byte0, byte1), hi = (byte2, byte3); the first byte in the low half.
__device__ __forceinline__ void e4m3x4_to_f16x2_scaled(uint32_t w, uint32_t& lo, uint32_t& hi) {
  uint32_t a = __byte_perm(w, 0u, 0x1404);  // byte1 << 24 | byte0 << 8
  uint32_t b = __byte_perm(w, 0u, 0x3424);  // byte3 << 24 | byte2 << 8
  lo = (a & 0x80008000u) | ((a >> 1) & 0x3F803F80u);
  hi = (b & 0x80008000u) | ((b >> 1) & 0x3F803F80u);
}
// Four e4m3 bytes -> two f16x2 with the hardware conversion (exact, no scale).
__device__ __forceinline__ void e4m3x4_to_f16x2_cvt(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l;\n cvt.rn.f16x2.e4m3x2 %1, h;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// Two e2m1 codes in one byte (first element in the low nibble) -> f16x2.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n" : "=r"(r) : "r"(byte));
  return r;
}
// e4m3 byte -> float (exact)
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  uint16_t in = static_cast<uint16_t>(byte & 0xFF);
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFF)));
}
// Two floats -> two e4m3 bytes (round to nearest even, saturating);
// `first` goes to the low byte.
__device__ __forceinline__ uint32_t float2_to_e4m3x2(float first, float second) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
  return r;
}
// Two floats -> one byte of two e2m1 codes (RNE, saturating); `first` in the
// low nibble.
__device__ __forceinline__ uint32_t float2_to_e2m1x2(float first, float second) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}\n"
      : "=r"(r)
      : "f"(second), "f"(first));
  return r & 0xFF;
}
// 2^(b-127) for an e8m0 byte (b = 255 is NaN and never written)
__device__ __forceinline__ float e8m0_to_float(uint32_t b) {
  return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}
// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32: relative error
// near 2^-22, results below 2^-126 flushed to zero, 2^-inf = 0).  For
// softmax weights, which are rounded to f16 or bf16 before they are used.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// max of three floats in one instruction (PTX max.f32 with three sources)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// (a.x * b.x, a.y * b.y), each rounded to nearest as a scalar multiply, in
// one packed instruction
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  uint64_t x, y, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
  float2 o;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
  return o;
}
// largest of 16 values, as a tree of three-input maxima
__device__ __forceinline__ float max16(const float (&x)[16]) {
  const float a = fmax3(x[0], x[1], x[2]), b = fmax3(x[3], x[4], x[5]), c = fmax3(x[6], x[7], x[8]);
  const float d = fmax3(x[9], x[10], x[11]), e = fmax3(x[12], x[13], x[14]);
  return fmax3(fmax3(a, b, c), fmax3(d, e, x[15]), -INFINITY);
}
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// (a, b) -> bf16x2 hi = RN(a, b) and lo = RN(a - hi, b - hi): hi + lo holds
// a and b to about 16 significant bits.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xFFFF0000u));
}
// Two bf16 (bit patterns in the halves of w) -> f16x2 (exact within the f16 range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = w;
  return __half22float2(h);
}

// ---- thread-block clusters ------------------------------------------------
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The same barrier without release: for a CTA that must stay resident until
// its peers have finished reading its shared memory (their loads have
// returned before they arrive), not to publish anything.
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\nbarrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// ---- programmatic dependent launch -----------------------------------------
// Kernels are launched with programmatic stream serialization, so one may
// start while the kernel before it on the stream is still running.  Each
// kernel calls pdl_wait() before its first global-memory access: it returns
// once the previous grid has completed and its writes are visible (at once
// when there is no such grid).  pdl_trigger() lets the next kernel's CTAs be
// scheduled as this grid's CTAs retire.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// generic address of the same shared-memory location in CTA `rank` of the
// cluster; plain loads through it may be scheduled freely (order them after
// the cluster barrier that publishes the data)
template <typename T>
__device__ __forceinline__ const T* cluster_map(const T* local, uint32_t rank) {
  uint64_t out;
  asm("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(local)), "r"(rank));
  return reinterpret_cast<const T*>(out);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

}  // namespace bsp
