/*
 * write.c -- step 1, quantise and scatter new tokens into the caches (test
 * infrastructure; see bsp_oracle.h).
 *
 * [ATOM-2962] commit "... index key": the fused writer stores K, V and the
 * index key "straight onto the pool pages"; the write test of that PR compares
 * the cache with a dequantised oracle.  The slot of a token is
 * block*128 + offset ([MSA-API] metadata builder: the slot mapping the base
 * rebases for the writer); slot -1 skips the token.  QK-norm and RoPE are model
 * math outside this path: the inputs here are the post-RoPE bf16 rows.
 *
 * Per format:
 *  - bf16: the bf16 bits are stored unchanged;
 *  - fp8 K/V: byte = e4m3(x / k_scale) (resp. v_scale) with an IEEE fp32
 *    division and a saturating cast ([vLLM-61889] Details: the "FP8 scale
 *    arguments" are per-tensor k/v scales);
 *  - MXFP4: per 32-element group the e8m0 shared exponent e (codecs.c), then
 *    nibble = e2m1(x * 2^-e) with an exact power-of-two scaling;
 *  - fp8 index key (reading): one fp32 scale s = amax/448 per (token, head),
 *    s = 1 for an all-zero row, byte = e4m3(x / s), both fp32 operations.
 */
#include "bsp_oracle.h"

#include <math.h>
#include <string.h>

static void write_mx_field(uint8_t* field, int t, const float* x /*128*/) {
  for (int g = 0; g < ORC_DIM / 32; ++g) {
    uint8_t sb = orc_mx_scale_byte(x + 32 * g, 32);
    int e = (int)sb - 127;
    field[8192 + t * 4 + g] = sb;
    for (int i = 0; i < 32; i += 2) {
      int d = 32 * g + i;
      uint8_t lo = orc_e2m1_encode(ldexp((double)x[d], -e));
      uint8_t hi = orc_e2m1_encode(ldexp((double)x[d + 1], -e));
      field[t * 64 + d / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

static void write_kv_side(int kv_dtype, int Hkv, uint8_t* kv, int side, int64_t block, int o, int h,
                          const uint16_t* row /*128 bf16*/, float scale) {
  float x[ORC_DIM];
  for (int d = 0; d < ORC_DIM; ++d) x[d] = orc_bf16_decode(row[d]);
  if (kv_dtype == ORC_MXFP4) {
    write_mx_field(kv + orc_mx_field_offset(Hkv, block, side, h), o, x);
    return;
  }
  int64_t page_id = block * 16 + o / ORC_PAGE;
  int t = o % ORC_PAGE;
  for (int d = 0; d < ORC_DIM; ++d) {
    int64_t off = orc_l1_offset(kv_dtype, Hkv, side, page_id, h, t, d);
    if (kv_dtype == ORC_BF16) {
      memcpy(kv + off, &row[d], 2);
    } else {
      float q = x[d] / scale;
      kv[off] = orc_e4m3_encode(q);
    }
  }
}

static void write_index(int idx_dtype, int Hidx, uint8_t* idx, int64_t block, int o, int h,
                        const uint16_t* row) {
  int64_t fb = orc_index_field_bytes(idx_dtype);
  uint8_t* field = idx + block * (int64_t)Hidx * fb + (int64_t)h * fb;
  float x[ORC_DIM];
  for (int d = 0; d < ORC_DIM; ++d) x[d] = orc_bf16_decode(row[d]);
  if (idx_dtype == ORC_BF16) {
    memcpy(field + (int64_t)o * 256, row, 256);
  } else if (idx_dtype == ORC_FP8) {
    float amax = 0.0f;
    for (int d = 0; d < ORC_DIM; ++d)
      if (fabsf(x[d]) > amax) amax = fabsf(x[d]);
    float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int d = 0; d < ORC_DIM; ++d) {
      float q = x[d] / s;
      field[o * 128 + d] = orc_e4m3_encode(q);
    }
    memcpy(field + 16384 + o * 4, &s, 4);
  } else {
    write_mx_field(field, o, x);
  }
}

void orc_kv_page_write(int kv_dtype, int Hkv, uint8_t* kv, float k_scale, float v_scale,
                       int idx_dtype, int Hidx, uint8_t* idx,
                       const uint16_t* k, const uint16_t* v, const uint16_t* idx_k,
                       const int64_t* slot, int T) {
#pragma omp parallel for schedule(static)
  for (int i = 0; i < T; ++i) {
    if (slot[i] < 0) continue;
    int64_t block = slot[i] / ORC_BLOCK;
    int o = (int)(slot[i] % ORC_BLOCK);
    for (int h = 0; h < Hkv; ++h) {
      const uint16_t* kr = k + ((int64_t)i * Hkv + h) * ORC_DIM;
      const uint16_t* vr = v + ((int64_t)i * Hkv + h) * ORC_DIM;
      write_kv_side(kv_dtype, Hkv, kv, 0, block, o, h, kr, k_scale);
      write_kv_side(kv_dtype, Hkv, kv, 1, block, o, h, vr, v_scale);
    }
    if (idx && idx_k) {
      for (int h = 0; h < Hidx; ++h)
        write_index(idx_dtype, Hidx, idx, block, o, h, idx_k + ((int64_t)i * Hidx + h) * ORC_DIM);
    }
  }
}

int orc_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  extern void omp_set_num_threads(int);
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
