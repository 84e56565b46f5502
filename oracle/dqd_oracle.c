/*
 * CPU oracle for the memory-bound decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library, its
 * Python binding) may include, link, import or call this file. Only the tests,
 * the package's smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant generator with the CUDA path.
 *
 * Every routine is the plain definition, evaluated in double precision with no
 * blocking, fusion or reordering beyond what the definition states. Where a
 * step decides an integer (an FP8 code), it is taken in the precision the
 * method fixes for it (IEEE binary32, the kernel's precision) and says so.
 *
 * Sources (web pages; the section is named in each routine):
 *   [MTC]  "降低每個 Token 的生成成本" (Making each token cheaper), optiverse-tech.com
 *   [LIF]  "LLM 推理是怎么变快的" (How LLM inference gets fast), random.sdx88.com
 *   [CS10] "第 10 讲：推理" (CS336 lecture 10 notes), semidirectx.com
 *   [ATC]  "AcceptedTokens 阅读笔记" (reading notes on speculative-decoding energy), zhongzhuzhou.org
 *
 * Readings taken where the pages are silent (each is also listed in the design notes):
 *   - INT4 g128: unsigned codes 0..15 with a 4-bit zero point and a bf16 scale
 *     per 128-weight group; deq = bf16_RNE((q - z) * s), one rounding.
 *   - FP8 row-wise: scale = fp32(max|w|) / 448 (IEEE binary32 division),
 *     code = e4m3_RNE_satfinite(fp32(w) / scale); a row of zeros takes scale 1.
 *   - Paged KV layout [block][kv_head][16][d]; GQA groups are contiguous
 *     (kv head = q head / (Hq/Hkv)); the W verify tokens are already in the
 *     cache, query i sits at position ctx - W + i and sees keys 0..ctx-W+i.
 *
 * Builds with any C11 compiler (x86_64 and aarch64); OpenMP is optional.
 * Do not build with -ffast-math: the FP8 quantiser relies on IEEE binary32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* bf16: the upper 16 bits of an IEEE binary32.                              */
/* ------------------------------------------------------------------------ */

static double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

ORC_EXPORT double orc_bf16_to_double(uint16_t h) { return bf16_to_double(h); }

/* Round a real number to the nearest bf16 (8 significant bits, exponent range
 * of binary32), ties to the even significand, overflow to infinity. Written
 * from the format: the quantum of the binade holding |v| is 2^(e-7), with the
 * subnormal quantum 2^-133 below 2^-126. */
ORC_EXPORT uint16_t orc_bf16_round(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  int e2;
  (void)frexp(a, &e2);          /* a = f * 2^e2 with f in [0.5, 1) */
  int lead = e2 - 1;            /* exponent of the leading bit      */
  if (lead < -126) lead = -126; /* subnormal binade                 */
  double quantum = ldexp(1.0, lead - 7);
  double r = nearbyint(a / quantum) * quantum; /* default mode: ties to even */
  if (r >= 0x1p128) return sign | 0x7F80;
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return sign | (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 [MTC, "格式" (Formats)]: 4 exponent bits, 3 mantissa bits, largest */
/* normal 448. Bias 7, subnormals, no infinities, S.1111.111 is NaN.          */
/* ------------------------------------------------------------------------ */

ORC_EXPORT double orc_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? ldexp((double)m, -9)          /* m/8 * 2^-6     */
                        : ldexp((double)(8 + m), e - 10); /* (1+m/8) 2^(e-7) */
  return s ? -mag : mag;
}

/* Round-to-nearest-even onto the finite E4M3 grid, saturating magnitudes at
 * or above 448 to 448 ("satfinite"); NaN stays NaN. Brute force over the 127
 * non-negative finite codes, so that nothing but the grid itself is assumed. */
static double e4m3_grid[0x7F]; /* values of codes 0x00..0x7E */

static void e4m3_grid_init(void) {
  static volatile int done = 0;
  if (done) return;
  for (int c = 0; c <= 0x7E; ++c) e4m3_grid[c] = orc_e4m3_decode((uint8_t)c);
  done = 1;
}

ORC_EXPORT uint8_t orc_e4m3_encode(float v) {
  e4m3_grid_init();
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  int best = 0;
  double best_d = a; /* distance to code 0 (value 0) */
  for (int c = 1; c <= 0x7E; ++c) {
    double d = fabs(e4m3_grid[c] - a);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return sign | (uint8_t)best;
}

/* FP8 row-wise weight quantiser [MTC, "格式" (Formats): values are multiplied
 * by a scale before the cast so that they fit the narrow range]. The scale
 * maps the row's largest magnitude onto 448. Decides integer codes, so it runs
 * in IEEE binary32 like the kernel. W is bf16 [n][k] row-major. */
ORC_EXPORT void orc_quant_fp8_rowwise(const uint16_t* w, int64_t n, int64_t k,
                                      uint8_t* codes, float* scales) {
  e4m3_grid_init();
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    const uint16_t* row = w + r * k;
    float amax = 0.0f;
    for (int64_t j = 0; j < k; ++j) {
      float a = fabsf((float)bf16_to_double(row[j]));
      if (a > amax) amax = a;
    }
    float scale = (amax > 0.0f) ? amax / 448.0f : 1.0f;
    scales[r] = scale;
    for (int64_t j = 0; j < k; ++j) {
      float v = (float)bf16_to_double(row[j]) / scale;
      codes[r * k + j] = orc_e4m3_encode(v);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* INT4 g128 weight-only (W4A16) [MTC, "格式" (Formats): 4-bit integers, one    */
/* scale per group of 128, dequantised to 16-bit before the arithmetic;        */
/* CS10 §5.2 for the scale/zero-point form].                                  */
/* ------------------------------------------------------------------------ */

static uint16_t int4_deq(uint8_t q, uint8_t z, uint16_t s) {
  /* (q - z) * s has at most 12 significant bits: exact in double. */
  return orc_bf16_round((double)((int)q - (int)z) * bf16_to_double(s));
}

/* deq[n][k] (bf16) from codes u8 [n][k] (0..15), scales bf16 [n][k/128],
 * zeros u8 [n][k/128] (0..15). */
ORC_EXPORT void orc_int4_dequant(const uint8_t* codes, const uint16_t* scales,
                                 const uint8_t* zeros, int64_t n, int64_t k,
                                 uint16_t* deq) {
  int64_t groups = k / 128;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r)
    for (int64_t j = 0; j < k; ++j)
      deq[r * k + j] = int4_deq(codes[r * k + j], zeros[r * groups + j / 128],
                                scales[r * groups + j / 128]);
}

/* INT4 asymmetric min/max quantiser [CS10 §5.2: a scale and a zero point map
 * x to an integer grid, x ~ (q - z) * s; "粒度" (granularity): how many values
 * share one scale, finer groups are more accurate at the cost of storing more
 * scales; MTC "格式": INT4 with one scale per group of 128]. The pages' worked
 * example is garbled; the plain min/max reading, per group of gsize weights of
 * one row:
 *   lo = min(0, min w), hi = max(0, max w)     (0 stays on the grid)
 *   s  = bf16_RNE(fp32(fp32(hi - lo) / 15)); a group of zeros takes s = 1;
 *        an s that rounds to 0 becomes the smallest bf16 subnormal
 *   z  = clamp(rint(fp32(-lo / s)), 0, 15)
 *   q  = clamp(rint(fp32(w / s)) + z, 0, 15)   (rint: ties to even)
 * Every step that decides an integer is taken in IEEE binary32, the
 * precision of the kernel. w: bf16 [n][k]; k % gsize == 0. */
ORC_EXPORT void orc_int4_quant(const uint16_t* w, int64_t n, int64_t k, int64_t gsize,
                               uint8_t* codes, uint16_t* scales, uint8_t* zeros) {
  const int64_t G = k / gsize;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t g = 0; g < G; ++g) {
      const uint16_t* wg = w + r * k + g * gsize;
      float lo = 0.0f, hi = 0.0f;
      for (int64_t j = 0; j < gsize; ++j) {
        const float v = (float)bf16_to_double(wg[j]);
        if (v < lo) lo = v;
        if (v > hi) hi = v;
      }
      const float d = hi - lo;
      uint16_t sb = 0x3F80; /* 1.0 */
      if (d > 0.0f) {
        const float s32 = d / 15.0f;
        sb = orc_bf16_round((double)s32);
        if ((sb & 0x7FFF) == 0) sb = 0x0001;
      }
      const float sf = (float)bf16_to_double(sb);
      float zf = rintf(-lo / sf);
      if (zf < 0.0f) zf = 0.0f;
      if (zf > 15.0f) zf = 15.0f;
      for (int64_t j = 0; j < gsize; ++j) {
        const float v = (float)bf16_to_double(wg[j]);
        float q = rintf(v / sf) + zf;
        if (q < 0.0f) q = 0.0f;
        if (q > 15.0f) q = 15.0f;
        codes[r * k + g * gsize + j] = (uint8_t)q;
      }
      scales[r * G + g] = sb;
      zeros[r * G + g] = (uint8_t)zf;
    }
  }
}

/* The packed INT4 g128 layout, as documented in include/dqd.h:
 *   NT = ceil(n/16) row tiles, G = k/128 groups, block b = T*G + g.
 *   Codes: 1024-byte blocks of 256 little-endian 32-bit words. Word
 *   w = 128*h + 4*l + j (h in 0..1, l in 0..31, j in 0..3); i = 4h + j,
 *   c = i/2, e = i%2, r0 = l/4, t = l%4. Nibble v (bits 4v..4v+3) holds the
 *   code of row 16T + r0 + 8*(v&1), column 128g + 32c + 8t + 4e
 *   + 2*((v>>1)&1) + (v>>2). Rows at or beyond n hold 0.
 *   Scales: 32-byte blocks of 8 words; word r0 = bf16 scale of row 16T+r0
 *   (bits 0..15) and of row 16T+r0+8 (bits 16..31).
 *   Zeros: 8-byte blocks; byte r0 = zero of row 16T+r0 (bits 0..3) and of
 *   row 16T+r0+8 (bits 4..7).
 * The two routines below are each other's inverse and are written from that
 * description alone. */
static void int4_layout_position(int64_t T, int64_t g, int w, int v,
                                 int64_t* row, int64_t* col) {
  int h = w / 128, l = (w / 4) % 32, j = w % 4;
  int i = 4 * h + j, c = i / 2, e = i % 2, r0 = l / 4, t = l % 4;
  *row = 16 * T + r0 + 8 * (v & 1);
  *col = 128 * g + 32 * c + 8 * t + 4 * e + 2 * ((v >> 1) & 1) + (v >> 2);
}

ORC_EXPORT void orc_int4_pack(const uint8_t* codes, const uint16_t* scales,
                              const uint8_t* zeros, int64_t n, int64_t k,
                              uint8_t* packed, uint8_t* packed_scales,
                              uint8_t* packed_zeros) {
  int64_t NT = (n + 15) / 16, G = k / 128;
#pragma omp parallel for schedule(static)
  for (int64_t T = 0; T < NT; ++T) {
    for (int64_t g = 0; g < G; ++g) {
      int64_t b = T * G + g;
      for (int w = 0; w < 256; ++w) {
        uint32_t word = 0;
        for (int v = 0; v < 8; ++v) {
          int64_t row, col;
          int4_layout_position(T, g, w, v, &row, &col);
          uint32_t q = (row < n) ? (codes[row * k + col] & 15u) : 0u;
          word |= q << (4 * v);
        }
        for (int byte = 0; byte < 4; ++byte)
          packed[b * 1024 + 4 * w + byte] = (uint8_t)(word >> (8 * byte));
      }
      for (int r0 = 0; r0 < 8; ++r0) {
        int64_t lo = 16 * T + r0, hi = lo + 8;
        uint16_t s_lo = (lo < n) ? scales[lo * G + g] : 0;
        uint16_t s_hi = (hi < n) ? scales[hi * G + g] : 0;
        uint8_t z_lo = (lo < n) ? (zeros[lo * G + g] & 15u) : 0;
        uint8_t z_hi = (hi < n) ? (zeros[hi * G + g] & 15u) : 0;
        uint8_t* sw = packed_scales + b * 32 + 4 * r0;
        sw[0] = (uint8_t)(s_lo & 0xFF);
        sw[1] = (uint8_t)(s_lo >> 8);
        sw[2] = (uint8_t)(s_hi & 0xFF);
        sw[3] = (uint8_t)(s_hi >> 8);
        packed_zeros[b * 8 + r0] = (uint8_t)(z_lo | (z_hi << 4));
      }
    }
  }
}

/* Decoder of the packed layout back to logical codes/scales/zeros. Rows at or
 * beyond n are checked to be zero; returns the number of nonzero padding
 * entries found (0 for a well-formed buffer). */
ORC_EXPORT int64_t orc_int4_unpack(const uint8_t* packed,
                                   const uint8_t* packed_scales,
                                   const uint8_t* packed_zeros, int64_t n,
                                   int64_t k, uint8_t* codes, uint16_t* scales,
                                   uint8_t* zeros) {
  int64_t NT = (n + 15) / 16, G = k / 128, bad = 0;
  for (int64_t T = 0; T < NT; ++T) {
    for (int64_t g = 0; g < G; ++g) {
      int64_t b = T * G + g;
      for (int w = 0; w < 256; ++w) {
        const uint8_t* p = packed + b * 1024 + 4 * w;
        uint32_t word = (uint32_t)p[0] | ((uint32_t)p[1] << 8) |
                        ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
        for (int v = 0; v < 8; ++v) {
          int64_t row, col;
          int4_layout_position(T, g, w, v, &row, &col);
          uint8_t q = (uint8_t)((word >> (4 * v)) & 15u);
          if (row < n)
            codes[row * k + col] = q;
          else
            bad += (q != 0);
        }
      }
      for (int r0 = 0; r0 < 8; ++r0) {
        const uint8_t* sw = packed_scales + b * 32 + 4 * r0;
        uint16_t s_lo = (uint16_t)(sw[0] | (sw[1] << 8));
        uint16_t s_hi = (uint16_t)(sw[2] | (sw[3] << 8));
        uint8_t zb = packed_zeros[b * 8 + r0];
        int64_t lo = 16 * T + r0, hi = lo + 8;
        if (lo < n) {
          scales[lo * G + g] = s_lo;
          zeros[lo * G + g] = zb & 15u;
        } else {
          bad += (s_lo != 0) + ((zb & 15u) != 0);
        }
        if (hi < n) {
          scales[hi * G + g] = s_hi;
          zeros[hi * G + g] = zb >> 4;
        } else {
          bad += (s_hi != 0) + ((zb >> 4) != 0);
        }
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------ */
/* dq_gemm: y = x * deq(W)^T [MTC, "量化省下什麼" (What quantisation saves):      */
/* a quantised matrix times a full-precision vector, weights dequantised on   */
/* the fly, activations not quantised]. x bf16 [m][k], W [n][k], y [m][n].    */
/* ------------------------------------------------------------------------ */

enum { ORC_W_BF16 = 0, ORC_W_FP8_E4M3 = 1, ORC_W_INT4_G128 = 2 };

/* Dequantised weight value of W[r][j] as a real number.
 *   BF16: the weight itself.
 *   FP8:  the E4M3 value; the per-row scale multiplies the whole dot product.
 *   INT4: bf16_RNE((q - z) * s). */
static double weight_value(int wtype, const void* data, const void* scales,
                           const uint8_t* zeros, int64_t k, int64_t r,
                           int64_t j) {
  switch (wtype) {
    case ORC_W_BF16:
      return bf16_to_double(((const uint16_t*)data)[r * k + j]);
    case ORC_W_FP8_E4M3:
      return orc_e4m3_decode(((const uint8_t*)data)[r * k + j]);
    default: {
      int64_t G = k / 128;
      uint8_t q = ((const uint8_t*)data)[r * k + j];
      return bf16_to_double(int4_deq(q, zeros[r * G + j / 128],
                                     ((const uint16_t*)scales)[r * G + j / 128]));
    }
  }
}

/* Computes y[mi][ri] = sum_j x[mi][j] * value(W[rows[ri]][j]) (times the FP8
 * row scale) for the listed rows (all n rows when rows == NULL; then
 * nrows must equal n). y is [m][nrows] double. Returns 0, or -1 on bad
 * arguments. */
ORC_EXPORT int orc_dq_gemm(int wtype, const void* data, const void* scales,
                           const uint8_t* zeros, int64_t n, int64_t k,
                           const uint16_t* x, int64_t m, const int64_t* rows,
                           int64_t nrows, double* y) {
  if (wtype < 0 || wtype > 2 || n < 0 || k < 0 || m < 0 || nrows < 0) return -1;
  if (wtype == ORC_W_INT4_G128 && k % 128 != 0) return -1;
  if (rows == NULL && nrows != n) return -1;
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t ri = 0; ri < nrows; ++ri) {
    int64_t r = rows ? rows[ri] : ri;
    double* wrow = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    for (int64_t j = 0; j < k; ++j)
      wrow[j] = weight_value(wtype, data, scales, zeros, k, r, j);
    double rs = (wtype == ORC_W_FP8_E4M3) ? (double)((const float*)scales)[r] : 1.0;
    for (int64_t mi = 0; mi < m; ++mi) {
      double acc = 0.0;
      for (int64_t j = 0; j < k; ++j) acc += bf16_to_double(x[mi * k + j]) * wrow[j];
      y[mi * nrows + ri] = rs * acc;
    }
    free(wrow);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* GQA decode / verify attention over a paged KV cache.                       */
/*   softmax(q K^T * scale) V for the new tokens' queries against every       */
/*   cached key/value [CS10 §2.2: append the new K,V, then attend; LIF §2.1]; */
/*   K/V read through a block table of 16-token blocks [LIF §3.1, CS10 §7.3]; */
/*   Hq query heads share Hkv KV heads [LIF §2.3]; causal inside the draft    */
/*   block [ATC, Algorithm 1: later candidates cannot affect earlier ones].   */
/* q: bf16 [B][W][Hq][D]; k_pool, v_pool: [blocks][Hkv][16][D] elements;      */
/* block_table: int32 [B][max_blocks]; ctx: int32 [B].                        */
/* Output rows are r = (b*W + i)*Hq + h; out is [nrows][D] double.            */
/* Returns 0, or -1 on bad arguments / a violated precondition.               */
/*                                                                            */
/* KV element formats: KV_BF16 (bf16 bits, read exactly) and KV_FP8 (E4M3     */
/* codes; the element's value is the code's value times one scale per pool,   */
/* k_scale for K and v_scale for V) [LIF §4.2 C: K/V cached as FP8; MTC,      */
/* speculative-decoding exercises: a 1-byte FP8 KV cache whose scale factors  */
/* the pages leave open — one fp32 scale per tensor is the plain reading].    */
/* ------------------------------------------------------------------------ */

enum { KV_BF16 = 0, KV_FP8 = 1 };

static double kv_elem(const void* pool, int fmt, int64_t idx, double scale) {
  if (fmt == KV_FP8) return orc_e4m3_decode(((const uint8_t*)pool)[idx]) * scale;
  return bf16_to_double(((const uint16_t*)pool)[idx]);
}

static int attn_core(const uint16_t* q, const void* k_pool, const void* v_pool, int fmt,
                     double k_scale, double v_scale, const int32_t* block_table,
                     int64_t max_blocks, const int32_t* ctx, int64_t num_blocks, int64_t B,
                     int64_t W, int64_t Hq, int64_t Hkv, int64_t D, double scale,
                     const int64_t* rows, int64_t nrows, double* out) {
  const int64_t BS = 16;
  if (B < 0 || W < 1 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv != 0) return -1;
  if (rows == NULL && nrows != B * W * Hq) return -1;
  for (int64_t b = 0; b < B; ++b)
    if (ctx[b] < W || (ctx[b] + BS - 1) / BS > max_blocks) return -1;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int64_t ri = 0; ri < nrows; ++ri) {
    int64_t r = rows ? rows[ri] : ri;
    int64_t h = r % Hq, i = (r / Hq) % W, b = r / (Hq * W);
    int64_t g = h / (Hq / Hkv);
    int64_t pos = ctx[b] - W + i; /* keys 0..pos are visible */
    int64_t nk = pos + 1;
    double* s = (double*)malloc(sizeof(double) * (size_t)nk);
    const uint16_t* qr = q + r * D;
    double smax = -INFINITY;
    for (int64_t j = 0; j < nk; ++j) {
      int32_t phys = block_table[b * max_blocks + j / BS];
      if (phys < 0 || phys >= num_blocks) { err |= 1; phys = 0; }
      const int64_t kr = ((phys * Hkv + g) * BS + j % BS) * D;
      double dot = 0.0;
      for (int64_t d = 0; d < D; ++d)
        dot += bf16_to_double(qr[d]) * kv_elem(k_pool, fmt, kr + d, k_scale);
      s[j] = scale * dot;
      if (s[j] > smax) smax = s[j];
    }
    double denom = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
      s[j] = exp(s[j] - smax);
      denom += s[j];
    }
    for (int64_t d = 0; d < D; ++d) out[ri * D + d] = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
      int32_t phys = block_table[b * max_blocks + j / BS];
      if (phys < 0 || phys >= num_blocks) phys = 0;
      const int64_t vr = ((phys * Hkv + g) * BS + j % BS) * D;
      double p = s[j] / denom;
      for (int64_t d = 0; d < D; ++d) out[ri * D + d] += p * kv_elem(v_pool, fmt, vr + d, v_scale);
    }
    free(s);
  }
  return err ? -1 : 0;
}

ORC_EXPORT int orc_gqa_decode_attn(const uint16_t* q, const uint16_t* k_pool,
                                   const uint16_t* v_pool,
                                   const int32_t* block_table, int64_t max_blocks,
                                   const int32_t* ctx, int64_t num_blocks,
                                   int64_t B, int64_t W, int64_t Hq, int64_t Hkv,
                                   int64_t D, double scale, const int64_t* rows,
                                   int64_t nrows, double* out) {
  return attn_core(q, k_pool, v_pool, KV_BF16, 1.0, 1.0, block_table, max_blocks, ctx,
                   num_blocks, B, W, Hq, Hkv, D, scale, rows, nrows, out);
}

/* The same attention over an FP8-E4M3 cache: k_pool, v_pool hold one code per
 * element, K = decode(code) * k_scale and V = decode(code) * v_scale. */
ORC_EXPORT int orc_gqa_decode_attn_fp8kv(const uint16_t* q, const uint8_t* k_pool,
                                         const uint8_t* v_pool, double k_scale,
                                         double v_scale, const int32_t* block_table,
                                         int64_t max_blocks, const int32_t* ctx,
                                         int64_t num_blocks, int64_t B, int64_t W,
                                         int64_t Hq, int64_t Hkv, int64_t D, double scale,
                                         const int64_t* rows, int64_t nrows, double* out) {
  return attn_core(q, k_pool, v_pool, KV_FP8, k_scale, v_scale, block_table, max_blocks, ctx,
                   num_blocks, B, W, Hq, Hkv, D, scale, rows, nrows, out);
}

/* ------------------------------------------------------------------------ */
/* RoPE and KV append [CS10 §2.2-2.3: for each new token compute q, k, v,     */
/* rotate q and k at the token's global position (start .. end-1, not from    */
/* 0), append k and v to the cache, then attend]. Rotary embedding in the     */
/* pairwise form: dims (2i, 2i+1) of a head rotate by angle pos * theta_i,    */
/* theta_i = base^(-2i/d), i.e. [x0', x1'] = [x0 c - x1 s, x0 s + x1 c].      */
/* ------------------------------------------------------------------------ */

/* Rotates one head vector x[d] (double) in place at position pos. */
static void rope_head(double* x, int64_t d, double pos, double base) {
  for (int64_t i = 0; i < d / 2; ++i) {
    const double theta = pow(base, -2.0 * (double)i / (double)d);
    const double a = pos * theta, c = cos(a), s = sin(a);
    const double x0 = x[2 * i], x1 = x[2 * i + 1];
    x[2 * i] = x0 * c - x1 * s;
    x[2 * i + 1] = x0 * s + x1 * c;
  }
}

ORC_EXPORT void orc_rope(double* x, int64_t rows, int64_t d, const double* pos, double base) {
  for (int64_t r = 0; r < rows; ++r) rope_head(x + r * d, d, pos[r], base);
}

/* qkv: bf16 [B*W][(Hq + 2*Hkv) * D], token (b, i) in row b*W + i, heads in the
 * order q_0..q_{Hq-1}, k_0..k_{Hkv-1}, v_0..v_{Hkv-1}. Token (b, i) sits at
 * position ctx[b] - W + i. Outputs (double): q_out [B*W][Hq][D] rotated,
 * k_out, v_out [B*W][Hkv][D] (k rotated, v as is), and slot [B*W]: the pool
 * row (phys * Hkv * 16 + pos % 16, to be offset by head * 16) the token's k
 * and v are appended to, or -1 for a position below 0. */
ORC_EXPORT int orc_rope_kv_append(const uint16_t* qkv, int64_t B, int64_t W, int64_t Hq,
                                  int64_t Hkv, int64_t D, double base, const int32_t* ctx,
                                  const int32_t* block_table, int64_t max_blocks,
                                  int64_t num_blocks, double* q_out, double* k_out,
                                  double* v_out, int64_t* slot) {
  if (D % 2 || B < 1 || W < 1) return -1;
  const int64_t width = (Hq + 2 * Hkv) * D;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t i = 0; i < W; ++i) {
      const int64_t row = b * W + i;
      const int64_t pos = (int64_t)ctx[b] - W + i;
      const uint16_t* src = qkv + row * width;
      for (int64_t e = 0; e < Hq * D; ++e) q_out[row * Hq * D + e] = bf16_to_double(src[e]);
      for (int64_t e = 0; e < Hkv * D; ++e) {
        k_out[row * Hkv * D + e] = bf16_to_double(src[Hq * D + e]);
        v_out[row * Hkv * D + e] = bf16_to_double(src[(Hq + Hkv) * D + e]);
      }
      for (int64_t h = 0; h < Hq; ++h) rope_head(q_out + (row * Hq + h) * D, D, (double)pos, base);
      for (int64_t h = 0; h < Hkv; ++h) rope_head(k_out + (row * Hkv + h) * D, D, (double)pos, base);
      if (pos < 0 || pos / 16 >= max_blocks) {
        slot[row] = -1;
      } else {
        int64_t phys = block_table[b * max_blocks + pos / 16];
        if (phys < 0) phys = 0;
        if (phys >= num_blocks) phys = num_blocks - 1;
        slot[row] = phys * Hkv * 16 + pos % 16;
      }
    }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Speculative verify: the step after the target's verify forward.            */
/* ------------------------------------------------------------------------ */

/* Greedy verify and KV-tail invalidation [ATC, Algorithm 1 "贪心验证及状态回退"]:
 * per request, position 0 of the verify block is the round's input token and
 * positions 1..k = w-1 hold the drafts d_1..d_k. t_i = argmax logits[i] (ties:
 * the smallest token id). Compare d_{i+1} with t_i from i = 0, stop at the
 * first mismatch: a = number of leading matches. The round emits the a matched
 * drafts and then the target's token t_a (the correction, or the extra token
 * when every draft matched): out = t_0 .. t_a, count = a + 1. The cache holds
 * the w verify tokens at its end; the k - a rejected drafts' KV becomes
 * invalid: context_lens -= k - a. A draft id outside [0, vocab) never matches.
 * logits: bf16 [b][w][vocab]; draft: int32 [b][w-1]; out: int32 [b][w] gets
 * t_0 .. t_{w-1}, of which the first count are the round's output; count:
 * int32 [b]; ctx: int32 [b] or NULL. */
ORC_EXPORT void orc_spec_verify_greedy(const uint16_t* logits, int64_t B, int64_t W, int64_t V,
                                       const int32_t* draft, int32_t* out, int32_t* count,
                                       int32_t* ctx) {
  for (int64_t b = 0; b < B; ++b) {
    int64_t a = 0;
    for (int64_t i = 0; i < W; ++i) {
      const uint16_t* row = logits + (b * W + i) * V;
      int64_t best = 0;
      double bv = bf16_to_double(row[0]);
      for (int64_t v = 1; v < V; ++v) {
        const double x = bf16_to_double(row[v]);
        if (x > bv) { bv = x; best = v; }
      }
      out[b * W + i] = (int32_t)best;   /* t_i */
      if (i == a && i < W - 1 && draft[b * (W - 1) + i] == best) a = i + 1;
    }
    count[b] = (int32_t)(a + 1);
    if (ctx) ctx[b] -= (int32_t)((W - 1) - a);
  }
}

/* Speculative sampling [CS336 lecture notes §6 "推测采样": draft x accepted with
 * probability min(1, q(x)/p(x)); on the first rejection, one token from
 * norm(max(q - p, 0)) and the rest of the draft is dropped; if all k are
 * accepted, one extra token from the target's position k+1]. The random
 * numbers are inputs: u_accept[b][i] in [0,1) decides draft i (accept iff
 * u * p(x) < q(x), the same test without a division, in binary32 like the
 * kernel), u_sample[b] in [0,1) draws the one sampled token by inverse CDF:
 * the smallest y with sum_{z<=y} r(z) > u * sum_z r(z) (sums in double),
 * r = max(q - p, 0) (binary32 difference) on a rejection, r = q for the extra
 * token. A residual that sums to 0 (possible only through rounding) falls back
 * to q. out = accepted drafts, then the sampled token; count = j + 1 with j
 * the number accepted; ctx -= k - j.
 * p: f32 [b][k][vocab]; q: f32 [b][k+1][vocab]; draft: int32 [b][k]. */
static int64_t orc_inverse_cdf(const float* q, const float* p, int64_t V, double u) {
  double total = 0.0;
  for (int64_t y = 0; y < V; ++y) {
    const float r = p ? fmaxf(q[y] - p[y], 0.0f) : q[y];
    total += (double)r;
  }
  if (p && total <= 0.0) return orc_inverse_cdf(q, NULL, V, u);
  const double thr = u * total;
  double acc = 0.0;
  int64_t last = 0;
  for (int64_t y = 0; y < V; ++y) {
    const float r = p ? fmaxf(q[y] - p[y], 0.0f) : q[y];
    if (r > 0.0f) last = y;
    acc += (double)r;
    if (acc > thr) return y;
  }
  return last; /* u * total rounded up to the total: the last token with mass */
}

ORC_EXPORT void orc_spec_verify_sample(const float* p, const float* q, const int32_t* draft,
                                       const float* u_accept, const float* u_sample,
                                       int64_t B, int64_t K, int64_t V, int32_t* out,
                                       int32_t* count, int32_t* ctx) {
  for (int64_t b = 0; b < B; ++b) {
    int64_t j = 0;
    while (j < K) {
      const int32_t x = draft[b * K + j];
      if (x < 0 || x >= V) break;
      const float px = p[(b * K + j) * V + x], qx = q[(b * (K + 1) + j) * V + x];
      if (!(u_accept[b * K + j] * px < qx)) break;
      out[b * (K + 1) + j] = x;
      ++j;
    }
    const float* qrow = q + (b * (K + 1) + j) * V;
    const float* prow = j < K ? p + (b * K + j) * V : NULL;
    out[b * (K + 1) + j] = (int32_t)orc_inverse_cdf(qrow, prow, V, (double)u_sample[b]);
    count[b] = (int32_t)(j + 1);
    if (ctx) ctx[b] -= (int32_t)(K - j);
  }
}

ORC_EXPORT int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads for the oracle's later parallel loops (n >= 1); a no-op without OpenMP. */
ORC_EXPORT void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Array forms of the scalar codecs, for the Python wrapper. */
ORC_EXPORT void orc_e4m3_decode_n(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(c[i]);
}
ORC_EXPORT void orc_e4m3_encode_n(const float* v, int64_t n, uint8_t* out) {
  e4m3_grid_init();
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}
ORC_EXPORT void orc_bf16_round_n(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_round(v[i]);
}
