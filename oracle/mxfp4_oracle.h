/*
 * mxfp4_oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU restatement of the MXFP4 training hot path: 32-point block
 * Walsh-Hadamard rotation, E8M0 block scale, E2M1 rounding (nearest-even or
 * stochastic), nibble packing, dequantization. It exists so that tests, the
 * package smoke check and the benchmark's CPU-baseline leg can check and time
 * the CUDA library against an independent definition. Nothing in the product
 * path may call it, and it shares no code with the CUDA sources.
 *
 * Every floating-point step that the method fixes in IEEE fp32 is done here in
 * fp32 C arithmetic compiled with -ffp-contract=off (no fused multiply-add,
 * no fast-math); decisions that are definitions (nearest grid point, scale
 * exponent) are made by direct search or exact fp64 arithmetic.
 */
#ifndef MXFP4_ORACLE_H
#define MXFP4_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_BLOCK_1X32 = 0, ORC_BLOCK_32X32 = 1, ORC_BLOCK_64X64 = 2, ORC_BLOCK_1X16 = 3 };
enum { ORC_SCALE_FLOOR = 0, ORC_SCALE_ROUNDUP = 1 };
enum { ORC_ROUND_RTN = 0, ORC_ROUND_SR = 1 };
enum { ORC_LAYOUT_ROWMAJOR = 0, ORC_LAYOUT_MMA = 1 };
enum { ORC_DTYPE_BF16 = 0, ORC_DTYPE_F32 = 1 };
enum { ORC_FORMAT_E2M1 = 0, ORC_FORMAT_E4M3 = 1, ORC_FORMAT_E5M2 = 2 };

typedef struct {
  int block;              /* ORC_BLOCK_* */
  int scale_mode;         /* ORC_SCALE_* */
  int rounding;           /* ORC_ROUND_* */
  int scale_layout;       /* ORC_LAYOUT_* (quantize_* write row-major only) */
  int wht;                /* 1: rotate each 32-block along K before scaling */
  uint32_t wht_sign_mask; /* bit i set => sign -1 on element i of a block */
  uint64_t seed;          /* Philox key */
  uint32_t sr_stream;     /* Philox counter word 2 */
  int elem_format;        /* ORC_FORMAT_*: E2M1 (MXFP4), E4M3 or E5M2 (MXFP8, nearest only) */
  int tensor_exp;         /* 1x16 (NVFP4) only: per-tensor factor 2^tensor_exp; else 0 */
} orc_params;

/* E2M1 code (4 bits, bit 3 = sign) -> value. */
float orc_e2m1_value(int code);

/* Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11). */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* 16 random bits for source element index i (row-major index of the input). */
uint32_t orc_sr_bits(uint64_t seed, uint32_t stream, uint64_t i);

/* One 32-point block rotation: forward c*H*diag(s)*x, inverse diag(s)*c*H*y. */
void orc_wht32(const float in[32], uint32_t sign_mask, int inverse, float out[32]);

/* Shared scale exponent e (scale 2^e) for block max-abs M >= 0. */
int orc_scale_exponent(float M, int scale_mode);

/* E2M1 codes for an already-scaled value v. */
int orc_round_rtn(float v);
int orc_round_sr(float v, uint32_t r16);

/* OCP FP8 E4M3 (8 bits: sign, 4 exponent bits with bias 7, 3 mantissa bits;
 * no infinities, S.1111.111 is NaN, largest finite 448): code -> value, and
 * the nearest code to v (ties to the even code, saturating at 448, sign kept). */
float orc_e4m3_value(int code);
int orc_round_e4m3_rtn(float v);

/* OCP FP8 E5M2 (sign, 5 exponent bits with bias 15, 2 mantissa bits;
 * S.11111.00 infinite, S.11111.xx NaN otherwise, largest finite 57344):
 * code -> value, and the nearest finite code to v (ties to the even code,
 * saturating at 57344, sign kept). */
float orc_e5m2_value(int code);
int orc_round_e5m2_rtn(float v);

/* Scale exponent for an element format: floor: floor(log2 M) - emax (emax 2
 * for E2M1, 8 for E4M3, 15 for E5M2); round-up: the smallest e with
 * max * 2^e >= M (max 6, 448 or 57344). orc_scale_exponent is the E2M1 case. */
int orc_scale_exponent_fmt(float M, int scale_mode, int elem_format);

/* NVFP4 block scale: the E4M3 code (0 .. 126) of the scale S of a 1x16 block
 * with max-abs M under the per-tensor factor 2^k. Round-up mode: the smallest
 * E4M3 value S with 6 * S * 2^k >= M (nothing clips; 448 if none is large
 * enough). Floor mode reads as "nearest": the E4M3 value nearest to
 * M / (6 * 2^k), ties to the even code, saturating at 448. */
int orc_nv_scale_code(float M, int k, int scale_mode);

/* Max-abs of x [rows, cols] (leading dim ld, elements): the largest |x[r][c]|,
 * exact in fp32 (a maximum does not depend on the order). 0 when empty. */
float orc_tensor_amax(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld);

/* Per-tensor exponent k of the NVFP4 factor 2^k for a tensor whose max-abs is
 * amax: the smallest integer k with 2688 * 2^k >= amax (2688 = 6 * 448, so the
 * largest block scale amax / (6 * 2^k) fits E4M3's largest value), clamped to
 * [-100, 100]; 0 for amax == 0. */
int orc_nv_tensor_exp(float amax);

/* Row-wise quantization of rows [r0, r1) of x [rows, cols] (leading dim ld,
 * elements), along cols. q: [(r1-r0), cols/2] bytes (E4M3: [(r1-r0), cols]),
 * s: [(r1-r0), cols/32] bytes (1x16 blocks: cols/16 E4M3 codes), both
 * row-major. Returns 0 on success, nonzero
 * on bad arguments. */
int orc_quantize_rows(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                      const orc_params* p, int64_t r0, int64_t r1, uint8_t* q, uint8_t* s);

/* Column-wise quantization (the quantization of x^T along the rows of x) for
 * columns [c0, c1) of x. q: [(c1-c0), rows/2], s: [(c1-c0), rows/32]. Random
 * bits are keyed by the element's index in x as passed. */
int orc_quantize_cols(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                      const orc_params* p, int64_t c0, int64_t c1, uint8_t* q, uint8_t* s);

/* Byte offset of scale (r, kb) in the tensor-core scale layout for a scale
 * matrix of `rows` rows and `nkb` scale columns. */
int64_t orc_mma_scale_offset(int64_t r, int64_t kb, int64_t rows, int64_t nkb);

/* Row-major [rows, nkb] -> tensor-core layout (rows % 128 == 0, nkb % 4 == 0). */
int orc_scales_to_mma(const uint8_t* s, int64_t rows, int64_t nkb, uint8_t* out);

/* Dequantize q [rows, cols/2] with scales s (layout as given) to fp32 / fp64. */
int orc_dequantize_f32(const uint8_t* q, const uint8_t* s, int layout, int64_t rows,
                       int64_t cols, float* out);
int orc_dequantize_f64(const uint8_t* q, const uint8_t* s, int layout, int64_t rows,
                       int64_t cols, double* out);
/* The same for 8-bit codes q [rows, cols] (one byte per element) of
 * elem_format ORC_FORMAT_E4M3 or ORC_FORMAT_E5M2; the E4M3 form kept too. */
int orc_dequantize_fp8_f64(const uint8_t* q, const uint8_t* s, int layout, int64_t rows,
                           int64_t cols, int elem_format, double* out);
int orc_dequantize_e4m3_f64(const uint8_t* q, const uint8_t* s, int layout, int64_t rows,
                            int64_t cols, double* out);

/* The same for NVFP4: q [rows, cols/2] E2M1 codes, s [rows, cols/16] E4M3
 * scale codes (layout as given; the tensor-core layout with cols/16 scale
 * columns), value = E2M1(code) * E4M3(s) * 2^tensor_exp. */
int orc_dequantize_nv_f64(const uint8_t* q, const uint8_t* s, int layout, int64_t rows,
                          int64_t cols, int tensor_exp, double* out);

/* Stand-alone rotation along cols of x; y [rows, cols] fp32 row-major. */
int orc_hadamard32(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                   uint32_t sign_mask, int inverse, float* y);

/* Brute-force fp64 product C[m,n] = sum_k A[m,k]*B[n,k] of dequantized
 * operands for the listed (m, n) pairs; also returns sum_k |A[m,k]*B[n,k]|. */
int orc_gemm_pairs(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb, const uint8_t* sb,
                   int layout, int64_t M, int64_t N, int64_t K, int64_t npairs,
                   const int64_t* ms, const int64_t* ns, double* c, double* abs_sum);

/* orc_gemm_pairs for NVFP4 operands (scales as in orc_dequantize_nv_f64). */
int orc_gemm_pairs_nv(const uint8_t* qa, const uint8_t* sa, int ka, const uint8_t* qb,
                      const uint8_t* sb, int kb, int layout, int64_t M, int64_t N, int64_t K,
                      int64_t npairs, const int64_t* ms, const int64_t* ns, double* c,
                      double* abs_sum);

#ifdef __cplusplus
}
#endif
#endif
