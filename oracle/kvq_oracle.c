/*
 * Plain CPU oracle for the quantized paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library may include, link
 * or call this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header or table with the CUDA
 * path.
 *
 * What it computes, and where each rule comes from:
 *
 *  - E4M3 encode/decode ("fn" variant: max 448, no infinities, NaN =
 *    S.1111.111).  The pages only say that values outside the chosen range
 *    clip and that values far inside lose precision ("Per-tensor vs per-head
 *    FP8 KV cache scales", section "Range sharing explains the accuracy
 *    trade"); the encoder below is round-to-nearest-even with saturation to
 *    +-448, written with integer arithmetic on the fp32 bit pattern.
 *  - Scale layouts: per-tensor (one K and one V scale per layer), static
 *    per-head (one K and one V scale per KV head) and dynamic per-token-head
 *    (scale = amax over head_dim / 448, one FP32 scale stored for every
 *    token-head slot, 1.0 when amax is 0) -- "Per-tensor vs per-head FP8 KV
 *    cache scales", sections "Per-tensor vs per-head FP8 KV cache scales" and
 *    "Dynamic per-token-head scales add 3.125 percent".
 *  - Packed INT4 per-token-head: K/V widths halved, two FP32 scales per
 *    token-head ("Per-token-head KV cache scale overhead", section "INT4 makes
 *    the metadata fraction larger"); symmetric, scale = amax / 7.
 *  - Layer skipping keeps a layer's cache in BF16 with no scales ("FP8 KV
 *    cache layer skipping vs per-head scales", section "FP8 KV cache layer
 *    skipping vs per-head scales"); a sliding-window layer retains at most W
 *    positions (same page, section "Layer skipping follows retained-token
 *    footprint").
 *  - Paged blocks of block_size tokens ("Per-token-head KV cache scale
 *    overhead", section "Convert bytes into block capacity").
 *  - Decode attention is the plain definition: softmax over
 *    softmax_scale * <q, K_hat[p]> for retained positions p, weighted sum of
 *    V_hat[p], in float64 on the dequantized cache.
 *
 * Cache layout (shared by contract with the library, not by code): codes are
 * [num_blocks][Hkv][block_size][row_bytes] with row_bytes = 2*D (BF16), D
 * (FP8) or D/2 (INT4); dynamic scales are [num_blocks][Hkv][block_size] fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_FP8_PER_TENSOR = 1, ORC_FP8_PER_HEAD = 2,
       ORC_FP8_PER_TOKEN_HEAD = 3, ORC_INT4_PER_TOKEN_HEAD = 4 };

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits. */
float orc_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* Round sig / 2^shift to the nearest integer, ties to even (shift >= 1). */
static uint32_t rne_shift(uint32_t sig, int shift) {
  if (shift >= 32) return 0;
  uint32_t q = sig >> shift;
  uint32_t rem = sig & ((1u << shift) - 1u);
  uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) q += 1u;
  return q;
}

/* fp32 -> E4M3 code, round to nearest even, saturating finite values and
 * infinities to +-448 (0x7E / 0xFE); NaN -> 0x7F with the input sign. */
uint8_t orc_e4m3_encode(float y) {
  uint32_t u = f32_bits(y);
  uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint8_t)(sign | 0x7Fu);       /* NaN */
  if (a >= 0x43E00000u) return (uint8_t)(sign | 0x7Eu);      /* |y| >= 448 */
  int ef = (int)(a >> 23);                                   /* biased exponent */
  uint32_t sig;
  int e;                                                     /* |y| = sig * 2^(e-23) */
  if (ef == 0) { sig = a & 0x7FFFFFu; e = -126; }            /* fp32 subnormal */
  else { sig = (a & 0x7FFFFFu) | 0x800000u; e = ef - 127; }
  if (e < -6) {
    /* E4M3 subnormal range: code value = n * 2^-9, n = RNE(|y| * 2^9).
     * n == 8 is the smallest normal, whose code is also 8. */
    uint32_t n = rne_shift(sig, 14 - e);                      /* shift >= 21 */
    return (uint8_t)(sign | n);
  }
  /* Normal: |y| = (n/8) * 2^e with n = RNE(sig / 2^20) in [8, 16].  A carry to
   * 16 rolls into the exponent field because code = ((e+7)<<3) + (n-8). */
  uint32_t n = rne_shift(sig, 20);
  return (uint8_t)(sign | (uint32_t)(((e + 7) << 3) + (int)n - 8));
}

/* The encoder over an array (for exhaustive checks). */
void orc_e4m3_encode_array(const float* y, uint8_t* out, long long n) {
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < n; ++i) out[i] = orc_e4m3_encode(y[i]);
}

/* E4M3 code -> value (exact in double).  0x7F / 0xFF are NaN. */
double orc_e4m3_decode(uint8_t c) {
  int s = c >> 7, E = (c >> 3) & 0xF, m = c & 7;
  double v;
  if ((c & 0x7F) == 0x7F) return NAN;
  if (E == 0) v = ldexp((double)m, -9);
  else v = ldexp((double)(8 + m), E - 10);
  return s ? -v : v;
}

/* fp32 -> signed INT4 in [-7, 7]: round to nearest even, then clamp. */
int orc_int4_encode(float y) {
  float r = nearbyintf(y);                       /* default mode: ties to even */
  if (!(r == r)) return 0;
  if (r > 7.0f) r = 7.0f;
  if (r < -7.0f) r = -7.0f;
  return (int)r;
}

static int int4_nibble_value(uint8_t byte, int hi) {
  int v = hi ? (byte >> 4) & 0xF : byte & 0xF;
  return v >= 8 ? v - 16 : v;                    /* two's complement nibble */
}

static int row_bytes_for(int mode, int D) {
  if (mode == ORC_BF16) return 2 * D;
  if (mode == ORC_INT4_PER_TOKEN_HEAD) return D / 2;
  return D;
}

/* Quantize one head vector x[0..D) into `row` (and the scale it used). */
static void quantize_vector(int mode, int D, const uint16_t* x, float static_scale,
                            uint8_t* row, float* scale_out) {
  if (mode == ORC_BF16) { memcpy(row, x, (size_t)2 * D); return; }
  float s;
  if (mode == ORC_FP8_PER_TENSOR || mode == ORC_FP8_PER_HEAD) {
    s = static_scale;
  } else {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
      float a = fabsf(orc_bf16_to_f32(x[d]));
      if (a > amax) amax = a;
    }
    const float qmax = (mode == ORC_INT4_PER_TOKEN_HEAD) ? 7.0f : 448.0f;
    s = (amax == 0.0f) ? 1.0f : amax / qmax;    /* fp32, round to nearest */
    *scale_out = s;
  }
  if (mode == ORC_INT4_PER_TOKEN_HEAD) {
    memset(row, 0, (size_t)D / 2);
    for (int d = 0; d < D; ++d) {
      float y = orc_bf16_to_f32(x[d]) / s;
      int q = orc_int4_encode(y);
      row[d / 2] |= (uint8_t)((q & 0xF) << ((d & 1) ? 4 : 0));
    }
  } else {
    for (int d = 0; d < D; ++d) row[d] = orc_e4m3_encode(orc_bf16_to_f32(x[d]) / s);
  }
}

/* Cache write: every token t with slot_mapping[t] >= 0 is quantized and stored
 * at block slot/bs, offset slot%bs, for every KV head.  Returns 0, or -1 when a
 * slot points past the cache (nothing is written for that token). */
int orc_cache_write(int mode, long long T, int Hkv, int D, int bs, long long num_blocks,
                    const uint16_t* k_new, const uint16_t* v_new, const int64_t* slots,
                    const float* k_scale, const float* v_scale,
                    uint8_t* k_cache, uint8_t* v_cache,
                    float* k_cache_scale, float* v_cache_scale) {
  const int rb = row_bytes_for(mode, D);
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (long long t = 0; t < T; ++t) {
    int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * (long long)bs) { bad |= 1; continue; }
    long long blk = slot / bs, off = slot % bs;
    for (int h = 0; h < Hkv; ++h) {
      size_t cell = ((size_t)blk * Hkv + h) * bs + off;
      const uint16_t* kx = k_new + ((size_t)t * Hkv + h) * D;
      const uint16_t* vx = v_new + ((size_t)t * Hkv + h) * D;
      float ks = 0.f, vs = 0.f, ks_out = 0.f, vs_out = 0.f;
      if (mode == ORC_FP8_PER_TENSOR) { ks = k_scale[0]; vs = v_scale[0]; }
      if (mode == ORC_FP8_PER_HEAD) { ks = k_scale[h]; vs = v_scale[h]; }
      quantize_vector(mode, D, kx, ks, k_cache + cell * rb, &ks_out);
      quantize_vector(mode, D, vx, vs, v_cache + cell * rb, &vs_out);
      if (mode == ORC_FP8_PER_TOKEN_HEAD || mode == ORC_INT4_PER_TOKEN_HEAD) {
        k_cache_scale[cell] = ks_out;
        v_cache_scale[cell] = vs_out;
      }
    }
  }
  return bad ? -1 : 0;
}

/* Static per-head calibration: amax over a sample [T][Hkv][D] per head, divided
 * by qmax in fp32; a head whose sample is all zero gets 1.0. */
void orc_calibrate_per_head(long long T, int Hkv, int D, const uint16_t* x, float qmax,
                            float* scale_out) {
  for (int h = 0; h < Hkv; ++h) {
    float amax = 0.0f;
    for (long long t = 0; t < T; ++t)
      for (int d = 0; d < D; ++d) {
        float a = fabsf(orc_bf16_to_f32(x[((size_t)t * Hkv + h) * D + d]));
        if (a > amax) amax = a;
      }
    scale_out[h] = (amax == 0.0f) ? 1.0f : amax / qmax;
  }
}

/* Dequantized value of element d of the cached row at (blk, h, off). */
static double cached_value(int mode, int Hkv, int D, int bs, const uint8_t* cache,
                           const float* tensor_or_head_scale, const float* slot_scale,
                           long long blk, int h, int off, int d) {
  const int rb = row_bytes_for(mode, D);
  size_t cell = ((size_t)blk * Hkv + h) * bs + off;
  const uint8_t* row = cache + cell * rb;
  switch (mode) {
    case ORC_BF16: {
      uint16_t v; memcpy(&v, row + 2 * d, 2);
      return (double)orc_bf16_to_f32(v);
    }
    case ORC_FP8_PER_TENSOR: return orc_e4m3_decode(row[d]) * (double)tensor_or_head_scale[0];
    case ORC_FP8_PER_HEAD: return orc_e4m3_decode(row[d]) * (double)tensor_or_head_scale[h];
    case ORC_FP8_PER_TOKEN_HEAD: return orc_e4m3_decode(row[d]) * (double)slot_scale[cell];
    default:
      return (double)int4_nibble_value(row[d / 2], d & 1) * (double)slot_scale[cell];
  }
}

/* Paged GQA decode attention in float64 on the dequantized cache, for the
 * listed (sequence, query head) pairs.  Query head hq reads KV head
 * hq / (Hq/Hkv).  Sequence b attends to positions [lo, L) with
 * L = context_lens[b] and lo = max(0, L - window) when window > 0, else 0.
 * out_pairs is [n_pairs][D]; a pair with no retained position gets zeros.
 * Returns 0, or -1 if a block-table entry needed by a position is out of range. */
int orc_decode_pairs(int mode, int Hq, int Hkv, int D, int bs, long long num_blocks,
                     int window, double softmax_scale, const uint16_t* q,
                     const uint8_t* k_cache, const uint8_t* v_cache,
                     const float* k_scale, const float* v_scale,
                     const float* k_cache_scale, const float* v_cache_scale,
                     const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                     int n_pairs, const int32_t* pair_b, const int32_t* pair_h,
                     double* out_pairs) {
  const int G = Hq / Hkv;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int i = 0; i < n_pairs; ++i) {
    const int b = pair_b[i], hq = pair_h[i], g = hq / G;
    const int L = context_lens[b];
    const int lo = (window > 0 && L > window) ? L - window : 0;
    double* o = out_pairs + (size_t)i * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (L <= lo) continue;
    const uint16_t* qv = q + ((size_t)b * Hq + hq) * D;
    double* score = (double*)malloc(sizeof(double) * (size_t)(L - lo));
    double mx = -INFINITY;
    for (int p = lo; p < L; ++p) {
      long long blk = block_table[(size_t)b * max_blocks + p / bs];
      if (blk < 0 || blk >= num_blocks) { bad |= 1; score[p - lo] = -INFINITY; continue; }
      double acc = 0.0;
      for (int d = 0; d < D; ++d)
        acc += (double)orc_bf16_to_f32(qv[d]) *
               cached_value(mode, Hkv, D, bs, k_cache, k_scale, k_cache_scale, blk, g, p % bs, d);
      score[p - lo] = softmax_scale * acc;
      if (score[p - lo] > mx) mx = score[p - lo];
    }
    double denom = 0.0;
    for (int p = lo; p < L; ++p) {
      long long blk = block_table[(size_t)b * max_blocks + p / bs];
      if (blk < 0 || blk >= num_blocks) continue;
      double w = exp(score[p - lo] - mx);
      denom += w;
      for (int d = 0; d < D; ++d)
        o[d] += w * cached_value(mode, Hkv, D, bs, v_cache, v_scale, v_cache_scale, blk, g,
                                 p % bs, d);
    }
    for (int d = 0; d < D; ++d) o[d] /= denom;
    free(score);
  }
  return bad ? -1 : 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
