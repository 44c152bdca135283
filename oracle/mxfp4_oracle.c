/*
 * mxfp4_oracle.c -- TEST INFRASTRUCTURE ONLY: the plain CPU definition that
 * the CUDA library is checked against. Only the tests, the package smoke
 * check and the benchmark's CPU-baseline leg load it; the product path never
 * does, and no code is shared with the CUDA sources.
 *
 * Sources of the method (cited by page title and section):
 *  [News]  "Block-Scaled MXFP4 With Stochastic Hadamard Rounding Matches BF16
 *          Convergence on 70B Pre-Training" -- para. 1 (E8M0 scale shared by a
 *          block of 32 E2M1 elements), para. 2 (32-element block Hadamard
 *          rotation fused with stochastic rounding before 4-bit packing).
 *  [Cim]   "Pretraining large language models with MXFP4" -- Abstract
 *          (Fprop/Dgrad/Wgrad; deterministic vs randomized Hadamard).
 *  [TIBQ]  "Stable FP4 Training via Transposition-Invariant Block
 *          Quantization" -- "Why FP4 training is the current frontier" (E2M1,
 *          P_i = round(X_i/S), reconstruction P_i*S), "The fix: 2D blocks"
 *          (b x b square blocks, transposition invariance), "Truncation-free
 *          scaling" (scale rounded up to a power of two, nothing clips),
 *          "Stochastic rounding in the backward pass" (E[round(x)] = x).
 *  [Tseng] "Training LLMs with MXFP4" -- Abstract (stochastic rounding with a
 *          random Hadamard transform; MXFP4 GEMMs).
 * Where the pages leave a step open the reading taken is stated at the step.
 *
 * Build: cc -O2 -std=c99 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC
 */
#include "mxfp4_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- E2M1 ---- */

/* E2M1: 1 sign, 2 exponent, 1 mantissa bit [TIBQ, "Why FP4 training is the
 * current frontier"]. Its eight magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6
 * (exponent bias 1, subnormal 0.5); code = sign<<3 | magnitude index. The
 * page's count of "16 magnitudes per sign" is read as 16 codes in total. */
static const double kGrid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

float orc_e2m1_value(int code) {
  double m = kGrid[code & 7];
  return (float)((code & 8) ? -m : m);
}

/* ------------------------------------------------------------- Philox ---- */

/* Philox4x32-10 as published by Salmon et al., "Parallel Random Numbers: As
 * Easy as 1, 2, 3" (SC'11): each round multiplies counter words 0 and 2 by the
 * two round multipliers, mixes the high halves with the other words and the
 * key; the key is bumped by the two Weyl constants between rounds. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Random bits for stochastic rounding. The pages fix no generator; the
 * reading taken: key = (seed low word, seed high word); counter =
 * (i/8 low word, i/8 high word, stream, 0) for source element index i, so one
 * Philox call serves 8 consecutive elements; element i takes 16-bit half
 * (i & 1) of output word ((i >> 1) & 3). */
uint32_t orc_sr_bits(uint64_t seed, uint32_t stream, uint64_t i) {
  uint64_t g = i >> 3;
  uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), stream, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  uint32_t w = out[(i >> 1) & 3];
  return (i & 1) ? (w >> 16) : (w & 0xFFFFu);
}

/* ---------------------------------------------------------------- WHT ---- */

/* fp32 nearest value of 1/sqrt(32); bit pattern 0x3E3504F3. */
static float wht_norm(void) {
  uint32_t u = 0x3E3504F3u;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* In-place unnormalised Walsh-Hadamard butterflies on 32 fp32 values in the
 * order h = 1, 2, 4, 8, 16; each pair (a, b) = (y[i], y[i+h]) with (i & h) == 0
 * becomes (a + b, a - b). The result is the Sylvester-ordered H with
 * H[i][j] = (-1)^popcount(i & j). The pages give neither the ordering nor the
 * normalisation of the "32-element Hadamard blocks" [News, para. 2]; this
 * order is the reading taken, and every fp32 operation is one rounded add. */
static void butterflies(float y[32]) {
  for (int h = 1; h < 32; h <<= 1) {
    for (int i = 0; i < 32; ++i) {
      if (i & h) continue;
      float a = y[i], b = y[i + h];
      y[i] = a + b;
      y[i + h] = a - b;
    }
  }
}

/* Forward: y = c * H * diag(s) * x, with s_i = -1 where bit i of the mask is
 * set (the random-sign transform of [Tseng, Abstract]; mask 0 gives the
 * deterministic rotation of [Cim, Abstract]). Inverse: x = diag(s) * c * H * y.
 * c = fp32(1/sqrt(32)) is applied as one rounded multiply after the last
 * butterfly. */
void orc_wht32(const float in[32], uint32_t sign_mask, int inverse, float out[32]) {
  float y[32];
  const float c = wht_norm();
  for (int i = 0; i < 32; ++i) {
    y[i] = in[i];
    if (!inverse && ((sign_mask >> i) & 1u)) y[i] = -y[i];
  }
  butterflies(y);
  for (int i = 0; i < 32; ++i) {
    y[i] = y[i] * c;
    if (inverse && ((sign_mask >> i) & 1u)) y[i] = -y[i];
  }
  memcpy(out, y, sizeof(y));
}

/* --------------------------------------------------------- E8M0 scale ---- */

/* Shared scale S = 2^e for a block with max-abs M.
 * Floor mode (OCP Microscaling Formats v1.0, the standard [News, para. 1]
 * names): e = floor(log2 M) - emax(E2M1), emax = 2, so M/S lies in [4, 8) and
 * the block max may saturate at 6.
 * Round-up mode [TIBQ, "Truncation-free scaling"]: the scale is rounded up to
 * the next power of two so that no element exceeds the E2M1 bound Q_p = 6:
 * e = ceil(log2(M / 6)), the smallest e with 6 * 2^e >= M.
 * M == 0 gives e = -127. e is clamped to the E8M0 range [-127, 127]; the
 * stored byte is e + 127 (0xFF, the E8M0 NaN, is never produced).
 * Computed with exact fp64 frexp/ldexp. */
int orc_scale_exponent_fmt(float M, int scale_mode, int elem_format) {
  /* exponent and value of the largest element: E2M1 6 = 1.5 * 2^2, E4M3
   * 448 = 1.75 * 2^8, E5M2 57344 = 1.75 * 2^15 */
  const int emax = elem_format == ORC_FORMAT_E4M3 ? 8 : (elem_format == ORC_FORMAT_E5M2 ? 15 : 2);
  const double vmax = elem_format == ORC_FORMAT_E4M3 ? 448.0
                      : (elem_format == ORC_FORMAT_E5M2 ? 57344.0 : 6.0);
  int e;
  if (!(M > 0.0f)) {
    e = -127;
  } else {
    int E2;
    (void)frexp((double)M, &E2);      /* M = m * 2^E2, m in [0.5, 1) */
    int fl = E2 - 1;                  /* floor(log2 M) */
    e = fl - emax;
    if (scale_mode == ORC_SCALE_ROUNDUP) {
      while (ldexp(vmax, e) < (double)M) ++e;      /* smallest e: vmax*2^e >= M */
      while (ldexp(vmax, e - 1) >= (double)M) --e;
    }
  }
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

int orc_scale_exponent(float M, int scale_mode) {
  return orc_scale_exponent_fmt(M, scale_mode, ORC_FORMAT_E2M1);
}

/* -------------------------------------------------------------- E4M3 ---- */
/* MXFP8 element format [TIBQ, "The fix, and its supporting cast": MXFP8 for
 * queries and keys; the OCP Microscaling v1.0 family the News page names]. */
float orc_e4m3_value(int code) {
  const int sgn = (code >> 7) & 1, E = (code >> 3) & 15, m = code & 7;
  double v;
  if (E == 15 && m == 7) return NAN;
  if (E == 0)
    v = ldexp((double)m, -9);                       /* subnormal: m/8 * 2^-6 */
  else
    v = ldexp(1.0 + m / 8.0, E - 7);
  return (float)(sgn ? -v : v);
}

int orc_round_e4m3_rtn(float v) {
  double a = fabs((double)v);
  if (a > 448.0) a = 448.0;                         /* saturate */
  int best = 0;
  double bestd = a;
  for (int k = 1; k < 127; ++k) {                   /* the finite non-negative codes */
    const double d = fabs(a - (double)orc_e4m3_value(k));
    if (d < bestd || (d == bestd && (k % 2) == 0 && (best % 2) != 0)) {
      best = k;
      bestd = d;
    }
  }
  return (signbit(v) ? 0x80 : 0) | best;
}

/* -------------------------------------------------------------- E5M2 ---- */
/* The other OCP FP8 element format of the same MX family: sign, 5 exponent
 * bits (bias 15), 2 mantissa bits; exponent field 31 holds infinities
 * (mantissa 0) and NaNs; subnormals m/4 * 2^-14; largest finite 57344. */
float orc_e5m2_value(int code) {
  const int sgn = (code >> 7) & 1, E = (code >> 2) & 31, m = code & 3;
  double v;
  if (E == 31) v = m ? NAN : INFINITY;
  else if (E == 0) v = ldexp((double)m, -16);
  else v = ldexp(1.0 + m / 4.0, E - 15);
  return (float)(sgn ? -v : v);
}

/* Nearest finite E5M2 code, ties to the even code, saturating at 57344, sign
 * kept: direct search over the 124 finite non-negative codes. */
int orc_round_e5m2_rtn(float v) {
  double a = fabs((double)v);
  if (a > 57344.0) a = 57344.0;
  int best = 0;
  double bestd = a;
  for (int k = 1; k < 124; ++k) {
    const double d = fabs(a - (double)orc_e5m2_value(k));
    if (d < bestd || (d == bestd && (k % 2) == 0 && (best % 2) != 0)) {
      best = k;
      bestd = d;
    }
  }
  return (signbit(v) ? 0x80 : 0) | best;
}

/* NVFP4 block scale [TIBQ, "Why FP4 training is the current frontier": 1x16
 * blocks (NVFP4) whose shared scale S is chosen from the block's max-abs].
 * Readings (the page gives only the block size and that S follows the block
 * max): S is an E4M3 value (the NVFP4 scale format) applied under a
 * per-tensor power-of-two factor 2^k, so the block scale is S * 2^k. The two
 * scale modes carry over from the E8M0 case: round-up ("truncation-free") is
 * the smallest S with 6 * S * 2^k >= M; floor mode, which has no power-of-two
 * meaning for E4M3, is read as the nearest S to M / (6 * 2^k) (ties to the
 * even code; a block max may then exceed 6 S 2^k by up to half an E4M3 step
 * and those elements saturate). Both saturate at 448. Direct search over the
 * 127 finite non-negative codes with exact fp64 arithmetic: M * 2^-k and
 * 6 * S are exact, and below the saturation point so is the distance to the
 * nearest candidates. */
int orc_nv_scale_code(float M, int k, int scale_mode) {
  const double y = ldexp((double)M, -k);
  if (scale_mode == ORC_SCALE_ROUNDUP) {
    for (int c = 0; c < 127; ++c)
      if (6.0 * (double)orc_e4m3_value(c) >= y) return c;
    return 126;
  }
  if (y >= 6.0 * 448.0) return 126;   /* saturate (keeps every distance below exact) */
  int best = 0;
  double bestd = fabs(y);
  for (int c = 1; c < 127; ++c) {
    const double d = fabs(6.0 * (double)orc_e4m3_value(c) - y);
    if (d < bestd || (d == bestd && (c % 2) == 0 && (best % 2) != 0)) {
      best = c;
      bestd = d;
    }
  }
  return best;
}

/* ------------------------------------------------------------ rounding ---- */

/* Round-to-nearest onto the E2M1 grid [TIBQ, "Stochastic rounding in the
 * backward pass", deterministic round-to-nearest]. Readings: magnitudes above
 * 6 saturate to 6; an exact midpoint goes to the even magnitude code (IEEE
 * nearest-even carried to the grid); the sign bit is v's sign bit, so -0 and
 * negative values that round to 0 encode as 0x8. Found by direct search over
 * the 8 grid points with exact fp64 distances. */
int orc_round_rtn(float v) {
  double a = fabs((double)v);
  if (a > 6.0) a = 6.0;
  int best = 0;
  double bestd = fabs(a - kGrid[0]);
  for (int k = 1; k < 8; ++k) {
    double d = fabs(a - kGrid[k]);
    if (d < bestd || (d == bestd && (k % 2) == 0 && (best % 2) != 0)) {
      best = k;
      bestd = d;
    }
  }
  return (signbit(v) ? 8 : 0) | best;
}

/* Stochastic rounding [TIBQ, "Stochastic rounding in the backward pass";
 * Tseng, Abstract]: a = min(|v|, 6) lies in [lo, hi) between adjacent grid
 * points; it goes to hi with probability p = (a - lo)/(hi - lo) so that the
 * expected value is a. Reading for the random source (the pages give none):
 * a 16-bit draw r rounds up iff r / 2^16 < p, i.e. P(up) = ceil(p*2^16)/2^16,
 * unbiased to within (hi - lo) * 2^-16. Grid values are never moved. */
int orc_round_sr(float v, uint32_t r16) {
  double a = fabs((double)v);
  if (a > 6.0) a = 6.0;
  int lo = 0;
  for (int k = 0; k < 8; ++k)
    if (kGrid[k] <= a) lo = k;
  int code = lo;
  if (lo < 7) {
    double p = (a - kGrid[lo]) / (kGrid[lo + 1] - kGrid[lo]);
    if ((double)(r16 & 0xFFFFu) / 65536.0 < p) code = lo + 1;
  }
  return (signbit(v) ? 8 : 0) | code;
}

/* ------------------------------------------------------------ quantize ---- */

static float load_elem(const void* x, int dtype, int64_t ld, int64_t r, int64_t c) {
  if (dtype == ORC_DTYPE_BF16) {
    uint32_t u = (uint32_t)((const uint16_t*)x)[r * ld + c] << 16; /* exact widening */
    float f;
    memcpy(&f, &u, 4);
    return f;
  }
  return ((const float*)x)[r * ld + c];
}

/* Max-abs over the tensor [TIBQ, "Why FP4 training is the current frontier of
 * precision reduction": block scales follow the max-abs; the per-tensor factor
 * of 1x16 blocks follows the tensor's]: plain loop, fp32 compares. */
float orc_tensor_amax(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld) {
  float m = 0.0f;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      const float a = fabsf(load_elem(x, dtype, ld, r, c));
      if (a > m) m = a;
    }
  return m;
}

/* Reading (the pages give no rule for the tensor factor): the smallest k in
 * [-100, 100] with 2688 * 2^k >= amax, by direct search over k with exact
 * fp64 powers of two; 100 if none is large enough; 0 for amax == 0. */
int orc_nv_tensor_exp(float amax) {
  if (amax == 0.0f) return 0;
  for (int k = -100; k <= 100; ++k)
    if (ldexp(2688.0, k) >= (double)amax) return k;
  return 100;
}

/* Quantize output rows [i0, i1) of one orientation. In the row orientation
 * output row i is source row i and position k is source column k; in the
 * column orientation output row i is source column i and k is source row k.
 * Blocks [News, para. 1; TIBQ, "The fix: 2D blocks", "The evidence" Table 4]:
 * 1x32 = 32 consecutive k of one output row; b x b (b = 32 or 64) = the
 * aligned b x b tile of output rows and k, whose one scale is stored on each
 * of its rows for each of its b/32 runs of 32 k. With the rotation on, each
 * 1x32 run along k is rotated first and the block max is taken afterwards. */
static int quantize_orient_nv(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                              const orc_params* p, int col_orient, int64_t i0, int64_t i1,
                              uint8_t* q, uint8_t* s);

static int quantize_orient(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                           const orc_params* p, int col_orient, int64_t i0, int64_t i1,
                           uint8_t* q, uint8_t* s) {
  if (p->block == ORC_BLOCK_1X16)
    return quantize_orient_nv(x, dtype, rows, cols, ld, p, col_orient, i0, i1, q, s);
  if (p->tensor_exp != 0) return -1;   /* the per-tensor factor belongs to NVFP4 */
  const int64_t nout = col_orient ? cols : rows;  /* output rows */
  const int64_t K = col_orient ? rows : cols;     /* quantization axis */
  /* g output rows by bw values of k share one scale */
  const int g = p->block == ORC_BLOCK_64X64 ? 64 : (p->block == ORC_BLOCK_32X32 ? 32 : 1);
  const int bw = p->block == ORC_BLOCK_64X64 ? 64 : 32;
  /* 8-bit elements (MXFP8): E4M3 or E5M2, one byte each */
  const int fp8 = p->elem_format == ORC_FORMAT_E4M3 || p->elem_format == ORC_FORMAT_E5M2;
  if (K % bw != 0 || i0 < 0 || i1 > nout || i0 > i1) return -1;
  if (p->elem_format != ORC_FORMAT_E2M1 && !fp8) return -1;
  if (fp8 && p->rounding != ORC_ROUND_RTN) return -1;   /* nearest only for MXFP8 */
  if (g > 1 && (nout % g != 0 || i0 % g != 0 || i1 % g != 0)) return -1;
  const int64_t nkb = K / 32;
  const int64_t ngroups = (i1 - i0) / g;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
  for (int64_t gi = 0; gi < ngroups; ++gi) {
    const int64_t ib = i0 + gi * g;
    float y[64][64];
    for (int64_t kb0 = 0; kb0 < K / bw && !bad; ++kb0) {
      float M = 0.0f;
      for (int t = 0; t < g; ++t) {
        const int64_t i = ib + t;
        for (int r = 0; r < bw / 32; ++r) {
          float blk[32];
          for (int j = 0; j < 32; ++j) {
            const int64_t k = kb0 * bw + r * 32 + j;
            blk[j] = col_orient ? load_elem(x, dtype, ld, k, i) : load_elem(x, dtype, ld, i, k);
            if (!isfinite(blk[j])) bad = 1; /* inputs must be finite */
          }
          if (p->wht)
            orc_wht32(blk, p->wht_sign_mask, 0, &y[t][r * 32]);
          else
            memcpy(&y[t][r * 32], blk, sizeof(blk));
        }
        for (int j = 0; j < bw; ++j) {
          float a = fabsf(y[t][j]);
          if (a > M) M = a;
        }
      }
      const int e = orc_scale_exponent_fmt(M, p->scale_mode, p->elem_format);
      const float inv_scale = ldexpf(1.0f, -e); /* 2^-e, exact (2^-127 is subnormal) */
      for (int t = 0; t < g; ++t) {
        const int64_t i = ib + t;
        const int64_t orow = i - i0;
        for (int r = 0; r < bw / 32; ++r) s[orow * nkb + kb0 * (bw / 32) + r] = (uint8_t)(e + 127);
        for (int j = 0; j < bw; ++j) {
          const int64_t k = kb0 * bw + j;
          const float v = y[t][j] * inv_scale;
          int code;
          if (fp8) {
            q[orow * K + k] = (uint8_t)(p->elem_format == ORC_FORMAT_E5M2 ? orc_round_e5m2_rtn(v)
                                                                         : orc_round_e4m3_rtn(v));
            continue;
          }
          if (p->rounding == ORC_ROUND_SR) {
            const int64_t src = col_orient ? (k * cols + i) : (i * cols + k);
            code = orc_round_sr(v, orc_sr_bits(p->seed, p->sr_stream, (uint64_t)src));
          } else {
            code = orc_round_rtn(v);
          }
          uint8_t* byte = &q[orow * (K / 2) + k / 2];
          if ((k & 1) == 0)
            *byte = (uint8_t)((*byte & 0xF0u) | (uint8_t)code);   /* even k: low nibble */
          else
            *byte = (uint8_t)((*byte & 0x0Fu) | (uint8_t)(code << 4));
        }
      }
    }
  }
  return bad ? -3 : 0;
}

/* NVFP4: blocks of 16 consecutive k of one output row, each with its E4M3
 * scale S (orc_nv_scale_code) under the factor 2^k. With the rotation on,
 * each 32-run along k is rotated first (the rotation does not depend on the
 * block size), then both of its 16-blocks are scaled. Scaling reading: one
 * fp32 reciprocal of the block scale, r = 1 / (S * 2^k) rounded to nearest,
 * and one rounded fp32 product per element, v = y * r (r = 0 when S = 0, so
 * such a block encodes as signed zeros). Rounding as for MXFP4; the random
 * bits are keyed by the source index as there. */
static int quantize_orient_nv(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                              const orc_params* p, int col_orient, int64_t i0, int64_t i1,
                              uint8_t* q, uint8_t* s) {
  const int64_t nout = col_orient ? cols : rows;
  const int64_t K = col_orient ? rows : cols;
  if (K % 32 != 0 || i0 < 0 || i1 > nout || i0 > i1) return -1;
  if (p->elem_format != ORC_FORMAT_E2M1) return -1;
  if (p->tensor_exp < -100 || p->tensor_exp > 100) return -1;
  const int64_t nkb = K / 16;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
  for (int64_t i = i0; i < i1; ++i) {
    const int64_t orow = i - i0;
    for (int64_t kr = 0; kr < K / 32 && !bad; ++kr) {
      float blk[32], y[32];
      for (int j = 0; j < 32; ++j) {
        const int64_t k = kr * 32 + j;
        blk[j] = col_orient ? load_elem(x, dtype, ld, k, i) : load_elem(x, dtype, ld, i, k);
        if (!isfinite(blk[j])) bad = 1;
      }
      if (p->wht)
        orc_wht32(blk, p->wht_sign_mask, 0, y);
      else
        memcpy(y, blk, sizeof(blk));
      for (int h = 0; h < 2; ++h) {
        float M = 0.0f;
        for (int j = 16 * h; j < 16 * h + 16; ++j)
          if (fabsf(y[j]) > M) M = fabsf(y[j]);
        const int sc = orc_nv_scale_code(M, p->tensor_exp, p->scale_mode);
        s[orow * nkb + 2 * kr + h] = (uint8_t)sc;
        const float S = ldexpf(orc_e4m3_value(sc), p->tensor_exp);   /* exact */
        const float r = S == 0.0f ? 0.0f : 1.0f / S;
        for (int j = 16 * h; j < 16 * h + 16; ++j) {
          const int64_t k = kr * 32 + j;
          const float v = y[j] * r;
          int code;
          if (p->rounding == ORC_ROUND_SR) {
            const int64_t src = col_orient ? (k * cols + i) : (i * cols + k);
            code = orc_round_sr(v, orc_sr_bits(p->seed, p->sr_stream, (uint64_t)src));
          } else {
            code = orc_round_rtn(v);
          }
          uint8_t* byte = &q[orow * (K / 2) + k / 2];
          if ((k & 1) == 0)
            *byte = (uint8_t)((*byte & 0xF0u) | (uint8_t)code);
          else
            *byte = (uint8_t)((*byte & 0x0Fu) | (uint8_t)(code << 4));
        }
      }
    }
  }
  return bad ? -3 : 0;
}

int orc_quantize_rows(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                      const orc_params* p, int64_t r0, int64_t r1, uint8_t* q, uint8_t* s) {
  if (!x || !p || !q || !s || ld < cols) return -1;
  return quantize_orient(x, dtype, rows, cols, ld, p, 0, r0, r1, q, s);
}

int orc_quantize_cols(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                      const orc_params* p, int64_t c0, int64_t c1, uint8_t* q, uint8_t* s) {
  if (!x || !p || !q || !s || ld < cols) return -1;
  return quantize_orient(x, dtype, rows, cols, ld, p, 1, c0, c1, q, s);
}

/* ------------------------------------------------- tensor-core layout ---- */

/* The block-scaled tensor-core operand layout for scale factors (not on the
 * pages; it is the one the CUDA toolkit documents for block-scaled GEMMs):
 * the [rows, nkb] scale matrix is cut into 128-row x 4-column tiles of 512
 * bytes, tiles ordered row-tile-major; inside a tile, scale (r, kb) sits at
 * (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4. */
int64_t orc_mma_scale_offset(int64_t r, int64_t kb, int64_t rows, int64_t nkb) {
  (void)rows;
  const int64_t tile = (r / 128) * (nkb / 4) + kb / 4;
  return tile * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (kb % 4);
}

int orc_scales_to_mma(const uint8_t* s, int64_t rows, int64_t nkb, uint8_t* out) {
  if (rows % 128 != 0 || nkb % 4 != 0) return -1;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t kb = 0; kb < nkb; ++kb)
      out[orc_mma_scale_offset(r, kb, rows, nkb)] = s[r * nkb + kb];
  return 0;
}

/* ---------------------------------------------------------- dequantize ---- */

/* Reconstruction P_i * S [TIBQ, "Why FP4 training is the current frontier"]:
 * value = E2M1(code) * 2^(byte - 127); byte 0xFF (E8M0 NaN) gives NaN. */
static double deq_one(const uint8_t* q, const uint8_t* s, int layout, int64_t rows, int64_t cols,
                      int64_t r, int64_t c) {
  const int64_t nkb = cols / 32;
  const uint8_t byte = q[r * (cols / 2) + c / 2];
  const int code = (c & 1) ? (byte >> 4) : (byte & 0x0F);
  const uint8_t sb = (layout == ORC_LAYOUT_MMA) ? s[orc_mma_scale_offset(r, c / 32, rows, nkb)]
                                                : s[r * nkb + c / 32];
  if (sb == 0xFF) return NAN;
  return ldexp((double)orc_e2m1_value(code), (int)sb - 127);
}

static int deq_check(int layout, int64_t rows, int64_t cols) {
  if (cols % 32 != 0 || rows < 0) return -1;
  if (layout == ORC_LAYOUT_MMA && (rows % 128 != 0 || (cols / 32) % 4 != 0)) return -1;
  return 0;
}

int orc_dequantize_f32(const uint8_t* q, const uint8_t* s, int layout, int64_t rows,
                       int64_t cols, float* out) {
  if (deq_check(layout, rows, cols)) return -1;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] = (float)deq_one(q, s, layout, rows, cols, r, c);
  return 0;
}

int orc_dequantize_f64(const uint8_t* q, const uint8_t* s, int layout, int64_t rows,
                       int64_t cols, double* out) {
  if (deq_check(layout, rows, cols)) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] = deq_one(q, s, layout, rows, cols, r, c);
  return 0;
}

int orc_dequantize_fp8_f64(const uint8_t* q, const uint8_t* s, int layout, int64_t rows,
                           int64_t cols, int elem_format, double* out) {
  if (deq_check(layout, rows, cols)) return -1;
  if (elem_format != ORC_FORMAT_E4M3 && elem_format != ORC_FORMAT_E5M2) return -1;
  const int64_t nkb = cols / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      const uint8_t sb = (layout == ORC_LAYOUT_MMA) ? s[orc_mma_scale_offset(r, c / 32, rows, nkb)]
                                                    : s[r * nkb + c / 32];
      const int code = q[r * cols + c];
      const double v = elem_format == ORC_FORMAT_E5M2 ? (double)orc_e5m2_value(code)
                                                      : (double)orc_e4m3_value(code);
      out[r * cols + c] = sb == 0xFF ? NAN : ldexp(v, (int)sb - 127);
    }
  return 0;
}

int orc_dequantize_e4m3_f64(const uint8_t* q, const uint8_t* s, int layout, int64_t rows,
                            int64_t cols, double* out) {
  return orc_dequantize_fp8_f64(q, s, layout, rows, cols, ORC_FORMAT_E4M3, out);
}

/* NVFP4 reconstruction: E2M1(code) * E4M3(scale) * 2^tensor_exp. */
static double deq_one_nv(const uint8_t* q, const uint8_t* s, int layout, int64_t rows,
                         int64_t cols, int tensor_exp, int64_t r, int64_t c) {
  const int64_t nkb = cols / 16;
  const uint8_t byte = q[r * (cols / 2) + c / 2];
  const int code = (c & 1) ? (byte >> 4) : (byte & 0x0F);
  const uint8_t sb = (layout == ORC_LAYOUT_MMA) ? s[orc_mma_scale_offset(r, c / 16, rows, nkb)]
                                                : s[r * nkb + c / 16];
  return ldexp((double)orc_e2m1_value(code) * (double)orc_e4m3_value(sb), tensor_exp);
}

static int deq_check_nv(int layout, int64_t rows, int64_t cols) {
  if (cols % 32 != 0 || rows < 0) return -1;
  if (layout == ORC_LAYOUT_MMA && (rows % 128 != 0 || (cols / 16) % 4 != 0)) return -1;
  return 0;
}

int orc_dequantize_nv_f64(const uint8_t* q, const uint8_t* s, int layout, int64_t rows,
                          int64_t cols, int tensor_exp, double* out) {
  if (deq_check_nv(layout, rows, cols)) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] = deq_one_nv(q, s, layout, rows, cols, tensor_exp, r, c);
  return 0;
}

/* ------------------------------------------------------------ hadamard ---- */

int orc_hadamard32(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                   uint32_t sign_mask, int inverse, float* y) {
  if (!x || !y || cols % 32 != 0 || ld < cols) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t kb = 0; kb < cols / 32; ++kb) {
      float blk[32], out[32];
      for (int j = 0; j < 32; ++j) blk[j] = load_elem(x, dtype, ld, r, kb * 32 + j);
      orc_wht32(blk, sign_mask, inverse, out);
      for (int j = 0; j < 32; ++j) y[r * cols + kb * 32 + j] = out[j];
    }
  }
  return 0;
}

/* ---------------------------------------------------------------- GEMM ---- */

/* C[m, n] = sum_k deq(A)[m, k] * deq(B)[n, k] summed in fp64 (both operands
 * K-major), for the MXFP4 GEMMs of [Tseng, Abstract] and the Fprop / Dgrad /
 * Wgrad products of [Cim, Abstract]. Brute force over K for listed pairs. */
int orc_gemm_pairs(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb, const uint8_t* sb,
                   int layout, int64_t M, int64_t N, int64_t K, int64_t npairs,
                   const int64_t* ms, const int64_t* ns, double* c, double* abs_sum) {
  if (deq_check(layout, M, K) || deq_check(layout, N, K)) return -1;
  for (int64_t t = 0; t < npairs; ++t) {
    const int64_t m = ms[t], n = ns[t];
    if (m < 0 || m >= M || n < 0 || n >= N) return -2;
    double acc = 0.0, acc_abs = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double prod = deq_one(qa, sa, layout, M, K, m, k) * deq_one(qb, sb, layout, N, K, n, k);
      acc += prod;
      acc_abs += fabs(prod);
    }
    c[t] = acc;
    abs_sum[t] = acc_abs;
  }
  return 0;
}

int orc_gemm_pairs_nv(const uint8_t* qa, const uint8_t* sa, int ka, const uint8_t* qb,
                      const uint8_t* sb, int kb, int layout, int64_t M, int64_t N, int64_t K,
                      int64_t npairs, const int64_t* ms, const int64_t* ns, double* c,
                      double* abs_sum) {
  if (deq_check_nv(layout, M, K) || deq_check_nv(layout, N, K)) return -1;
  for (int64_t t = 0; t < npairs; ++t) {
    const int64_t m = ms[t], n = ns[t];
    if (m < 0 || m >= M || n < 0 || n >= N) return -2;
    double acc = 0.0, acc_abs = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double prod = deq_one_nv(qa, sa, layout, M, K, ka, m, k) *
                          deq_one_nv(qb, sb, layout, N, K, kb, n, k);
      acc += prod;
      acc_abs += fabs(prod);
    }
    c[t] = acc;
    abs_sum[t] = acc_abs;
  }
  return 0;
}
