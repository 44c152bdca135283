/*
 * mxfp4.h -- C ABI of the GB300 (sm_103a) MXFP4 training hot path.
 *
 * The library implements the two parts of the hot path that the following
 * pages describe for MXFP4 training:
 *   [News]  "Block-Scaled MXFP4 With Stochastic Hadamard Rounding Matches BF16
 *           Convergence on 70B Pre-Training", paras. 1-2.
 *   [Cim]   "Pretraining large language models with MXFP4", Abstract.
 *   [TIBQ]  "Stable FP4 Training via Transposition-Invariant Block
 *           Quantization", sections "Why FP4 training is the current
 *           frontier of precision reduction", "The aha: transposition
 *           scrambles the blocks", "The fix, and its supporting cast".
 *   [Tseng] "Training LLMs with MXFP4", Abstract.
 *
 * Conventions for every call:
 *  - Pointers named x, y, q_*, s_*, qa, sa, qb, sb, c, out are DEVICE pointers
 *    (cudaMalloc / PyTorch CUDA memory) owned by the caller; params pointers
 *    are HOST pointers read during the call only. The library allocates no
 *    device memory and keeps no per-call state.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Work is enqueued asynchronously on it; the return value reports argument
 *    validation and launch errors only. Calls are thread-safe.
 *  - The first call of an entry point on a device fills per-device caches
 *    (kernel attributes, occupancy). Later calls of mxfp4_quantize,
 *    mxfp4_gemm, mxfp4_gemm_ex, mxfp4_gemm_quantize, nvfp4_gemm, mxfp8_gemm
 *    and mxfp4_tensor_amax with caller-supplied outputs and workspaces enqueue
 *    only kernel launches and asynchronous memsets on the stream, so a
 *    sequence of them can be captured into a CUDA graph and replayed (tested:
 *    the replay gives the eager results bit for bit).
 *  - Tensors are row-major with a leading dimension in elements. Packed E2M1
 *    codes hold two elements per byte: the even index in the low nibble, the
 *    odd index in the high nibble; code = sign << 3 | magnitude index into
 *    {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *  - Scales are E8M0 bytes (value 2^(byte - 127)), one per block of 32
 *    elements along the quantization axis, stored in one of two layouts:
 *      MXFP4_LAYOUT_ROWMAJOR: s[r * (K/32) + kb];
 *      MXFP4_LAYOUT_MMA: the block-scaled tensor-core operand layout: 128-row
 *        x 4-column tiles of 512 bytes, tiles in row-tile-major order, scale
 *        (r, kb) at tile ((r/128) * (K/128) + kb/4), byte
 *        (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4 (needs rows % 128 == 0
 *        and K % 128 == 0). mxfp4_gemm consumes this layout.
 *  - Pointers must be 16-byte aligned and leading dimensions multiples of
 *    8 elements, else MXFP4_ERR_ALIGN.
 */
#ifndef MXFP4_H
#define MXFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MXFP4_OK = 0,
  MXFP4_ERR_INVALID_ARG = 1, /* null pointer, bad enum value */
  MXFP4_ERR_SHAPE = 2,       /* dimension not supported (see each call) */
  MXFP4_ERR_ALIGN = 3,       /* pointer or leading dimension misaligned */
  MXFP4_ERR_UNSUPPORTED = 4, /* device is not sm_103 / sm_100 family */
  MXFP4_ERR_CUDA = 5,        /* CUDA runtime / driver error at launch */
  MXFP4_ERR_TIMEOUT = 6,     /* a bounded device-side wait ran out */
  MXFP4_ERR_BOUNDS = 7       /* a kernel store fell outside its output (only
                                builds with MXFP4_BOUNDS_CHECK detect it) */
} mxfp4_status;

enum { MXFP4_BLOCK_1X32 = 0, MXFP4_BLOCK_32X32 = 1, MXFP4_BLOCK_64X64 = 2, MXFP4_BLOCK_1X16 = 3 };
enum { MXFP4_SCALE_FLOOR = 0, MXFP4_SCALE_ROUNDUP = 1 };
enum { MXFP4_ROUND_RTN = 0, MXFP4_ROUND_SR = 1 };
enum { MXFP4_LAYOUT_ROWMAJOR = 0, MXFP4_LAYOUT_MMA = 1 };
enum { MXFP4_DTYPE_BF16 = 0, MXFP4_DTYPE_F32 = 1 };
/* Element format of the codes: E2M1 (MXFP4, two codes per byte), or MXFP8
 * with one code per byte, E4M3 or E5M2 (the two OCP FP8 formats) [TIBQ, "The
 * fix, and its supporting cast": MXFP8 for queries and keys]. All share the
 * E8M0 block scale and its layouts. */
enum { MXFP4_FORMAT_E2M1 = 0, MXFP4_FORMAT_E4M3 = 1, MXFP4_FORMAT_E5M2 = 2 };

/* Quantization parameters of one output orientation.
 *  block        MXFP4_BLOCK_1X32: 32 consecutive elements along the
 *               quantization axis share a scale [News, para. 1].
 *               MXFP4_BLOCK_32X32: the aligned 32 x 32 tile shares one scale,
 *               written on each of its 32 rows of the scale array [TIBQ,
 *               "The fix, and its supporting cast", 2D blocks].
 *               MXFP4_BLOCK_64X64: the aligned 64 x 64 tile shares one scale,
 *               written on each of its 64 rows for both of its 32-runs [TIBQ,
 *               "The evidence", Table 4 block sizes]; needs rows and K
 *               multiples of 64 (not available in mxfp4_gemm_quantize).
 *               MXFP4_BLOCK_1X16: NVFP4 [TIBQ, "Why FP4 training is the
 *               current frontier of precision reduction": 1 x 16 blocks]: 16
 *               consecutive E2M1 elements share an E4M3 scale S (one byte,
 *               OCP FP8 E4M3, codes 0..126) under the per-tensor factor
 *               2^tensor_exp; the element value is code * S * 2^tensor_exp.
 *               Scale arrays hold K/16 bytes per output row (both layouts;
 *               the tensor-core layout with K/16 scale columns). Elements are
 *               scaled by one fp32 reciprocal per block, r = RN(1 / (S *
 *               2^tensor_exp)) (0 when S = 0), v = RN(y * r). E2M1 elements
 *               only.
 *  scale_mode   MXFP4_SCALE_FLOOR: e = floor(log2 M) - 2 (OCP Microscaling
 *               v1.0; the block max may saturate at 6).
 *               MXFP4_SCALE_ROUNDUP: e = ceil(log2(M / 6)), nothing clips
 *               [TIBQ, "Truncation-free scaling"]. M is the block max-abs
 *               after the optional rotation; M == 0 gives e = -127; e is
 *               clamped to [-127, 127].
 *               With MXFP4_BLOCK_1X16 (E4M3 scale): round-up is the smallest
 *               S with 6 * S * 2^tensor_exp >= M (nothing clips); floor mode
 *               reads as nearest: the S nearest to M / (6 * 2^tensor_exp),
 *               ties to the even code; both saturate at S = 448.
 *  rounding     MXFP4_ROUND_RTN: nearest grid point, ties to the even code,
 *               saturating at 6. MXFP4_ROUND_SR: stochastic rounding [TIBQ,
 *               "Stochastic rounding in the backward pass"; Tseng, Abstract]:
 *               a 16-bit Philox4x32-10 draw r rounds |v| up from lo to hi iff
 *               r / 2^16 < (|v| - lo) / (hi - lo). The draw for source element
 *               i = row * cols + col (index in x as passed, for either
 *               orientation) is 16-bit half (i & 1) of word ((i >> 1) & 3) of
 *               Philox(counter = {i >> 3 (low, high word), sr_stream, 0},
 *               key = {seed low word, seed high word}).
 *  scale_layout MXFP4_LAYOUT_* for the scale array written.
 *  wht          1: before scaling, rotate every run of 32 elements along the
 *               quantization axis by c * H * diag(s) [News, para. 2; Tseng,
 *               Abstract; Cim, Abstract] -- H the 32 x 32 Sylvester Hadamard
 *               matrix, butterflies in the order h = 1, 2, 4, 8, 16 in fp32,
 *               c = fp32(1/sqrt(32)) applied last as one rounded multiply.
 *  wht_sign_mask bit i set => s_i = -1 (0 = the deterministic rotation).
 *  seed, sr_stream  Philox key and counter word 2 (used by MXFP4_ROUND_SR).
 *  elem_format  MXFP4_FORMAT_E2M1, MXFP4_FORMAT_E4M3 or MXFP4_FORMAT_E5M2.
 *  tensor_exp   MXFP4_BLOCK_1X16 only (else it must be 0): the exponent k of
 *               the per-tensor factor 2^k, in [-100, 100]. Choosing
 *               k = ceil(log2(amax / 2688)) for the tensor's max-abs amax keeps
 *               every block scale within E4M3's range.
 * All arithmetic is IEEE fp32 without fused multiply-add or flush-to-zero, so
 * results are bit-reproducible across calls and streams. */
typedef struct {
  int32_t block;
  int32_t scale_mode;
  int32_t rounding;
  int32_t scale_layout;
  int32_t wht;
  uint32_t wht_sign_mask;
  uint64_t seed;
  uint32_t sr_stream;
  uint32_t elem_format; /* MXFP4_FORMAT_E2M1 (0), MXFP4_FORMAT_E4M3 (1) or MXFP4_FORMAT_E5M2 (2) */
  int32_t tensor_exp;   /* MXFP4_BLOCK_1X16: per-tensor factor 2^tensor_exp */
} mxfp4_quant_params;

/* Fused MXFP4 quantizer ([News], paras. 1-2; [TIBQ] P_i = round(X_i / S)).
 *  x      [rows, cols] bf16 or fp32 (x_dtype), leading dimension ld_x >= cols.
 *  row    if non-NULL, quantize along cols:  q_row [rows, cols/2] bytes,
 *         s_row [rows, cols/32] scale bytes (row->scale_layout).
 *  col    if non-NULL, quantize x^T, i.e. along rows, in the same pass [TIBQ,
 *         "The aha: transposition scrambles the blocks"]: q_col [cols, rows/2],
 *         s_col [cols, rows/32]. Stochastic-rounding draws are keyed by the
 *         source index, so 32x32 blocks without rotation stay transposition
 *         invariant under stochastic rounding too.
 *  At least one of row / col must be non-NULL.
 *  Shapes: cols % 32 == 0; rows % 32 == 0 when col != NULL or either
 *  orientation uses 32x32 or 64x64 blocks; MMA scale layout needs the
 *  output's row count % 128 == 0 and its K % 128 == 0; rows * cols < 2^35
 *  (rows * cols / 16 below 2^31). Else MXFP4_ERR_SHAPE.
 *  With MXFP4_BLOCK_1X16 the scale arrays are s_row [rows, cols/16] and
 *  s_col [cols, rows/16].
 *  With elem_format MXFP4_FORMAT_E4M3 or MXFP4_FORMAT_E5M2 the codes take one
 *  byte per element (q_row [rows, cols], q_col [cols, rows]), the scale is
 *  chosen for the format's largest value, 448 for E4M3 and 57344 for E5M2
 *  (floor: floor(log2 M) - 8 or - 15; round-up: the smallest e with
 *  max * 2^e >= M) and the rounding is nearest-even with saturation at that
 *  value (stochastic rounding: MXFP4_ERR_UNSUPPORTED).
 *  Inputs must be finite, and with the rotation on every rotated value must
 *  be finite too (|x| < 2^122 suffices); otherwise the codes are unspecified. */
mxfp4_status mxfp4_quantize(const void* x, int32_t x_dtype, int64_t rows, int64_t cols,
                            int64_t ld_x, const mxfp4_quant_params* row, uint8_t* q_row,
                            uint8_t* s_row, const mxfp4_quant_params* col, uint8_t* q_col,
                            uint8_t* s_col, void* stream);

/* Reconstruction P_i * S ([TIBQ], "Why FP4 training is the current frontier
 * of precision reduction"): out[r, c] = E2M1(code) * 2^(byte - 127) in fp32;
 * scale byte 0xFF (E8M0 NaN) gives NaN.
 *  q [rows, cols/2], s in scale_layout, out [rows, cols] fp32 (dense).
 *  cols % 32 == 0 (MMA layout: rows % 128 == 0, cols % 128 == 0), at most
 *  2^40 elements; else MXFP4_ERR_SHAPE. */
mxfp4_status mxfp4_dequantize(const uint8_t* q, const uint8_t* s, int32_t scale_layout,
                              int64_t rows, int64_t cols, float* out, void* stream);

/* Reconstruction for every format mxfp4_quantize writes, described by the
 * block, elem_format and tensor_exp it was quantized with:
 *  E2M1 with 1x32 / 32x32 / 64x64 blocks: as mxfp4_dequantize;
 *  MXFP4_FORMAT_E4M3 / MXFP4_FORMAT_E5M2 (MXFP8): q [rows, cols] one byte
 *    per element, out = E4M3(byte) or E5M2(byte) times 2^(scale - 127) (E5M2
 *    infinity and NaN bytes decode as such);
 *  MXFP4_BLOCK_1X16 (NVFP4): q [rows, cols/2], s one E4M3 byte per 16
 *    elements ([rows, cols/16] or the tensor-core layout with cols/16 scale
 *    columns), out = E2M1(code) * E4M3(scale) * 2^tensor_exp.
 * Every product is exact in fp32; NaN scale or code bytes give NaN.
 *  Shapes and layouts as mxfp4_dequantize; tensor_exp in [-100, 100] for
 *  1x16 blocks, 0 otherwise (else MXFP4_ERR_INVALID_ARG). */
mxfp4_status mxfp4_dequantize_ex(const uint8_t* q, const uint8_t* s, int32_t scale_layout,
                                 int32_t block, uint32_t elem_format, int32_t tensor_exp,
                                 int64_t rows, int64_t cols, float* out, void* stream);

/* Block-scaled MXFP4 GEMM ([Tseng], Abstract: "MXFP4 GEMMs"; [Cim], Abstract:
 * Fprop, Dgrad and Wgrad all take this form):
 *   C[m, n] = sum_k deqA[m, k] * deqB[n, k]   (fp32 accumulation)
 * with both operands K-major (the "TN" form): qa [M, K/2], qb [N, K/2] packed
 * codes, sa / sb scales in MXFP4_LAYOUT_MMA. C fp32 [M, N] with leading
 * dimension ldc >= N. Fprop Y = X W^T is (A = X row-wise, B = W row-wise);
 * Dgrad dX = dY W is (A = dY row-wise, B = W column-wise); Wgrad dW = dY^T X is
 * (A = dY column-wise, B = X column-wise).
 *  Shapes: M, N and K positive multiples of 128, each at most 2^30. (The
 *  kernels work on 256 x 256 output tiles and 256-deep K steps: a last tile
 *  of 128 columns and a last K step of 128 are computed on zero-filled
 *  operands and only the valid part is stored.)
 *  Runs on tcgen05 tensor cores (sm_103a); returns MXFP4_ERR_UNSUPPORTED on
 *  other devices. */
mxfp4_status mxfp4_gemm(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                        const uint8_t* sb, int64_t M, int64_t N, int64_t K, float* c,
                        int64_t ldc, void* stream);

/* mxfp4_gemm with a choice of output type ([News], para. 2: a bf16 C is what
 * the next layer reads) and an optional workspace:
 *  c_dtype  MXFP4_DTYPE_F32 writes C as mxfp4_gemm does; MXFP4_DTYPE_BF16
 *           writes each fp32 sum rounded to bf16 (nearest-even), c a bf16
 *           [M, N] array with leading dimension ldc (ldc % 8 == 0, c 16-byte
 *           aligned). Other values return MXFP4_ERR_INVALID_ARG.
 *  workspace, workspace_bytes  caller-owned device memory (16-byte aligned;
 *           NULL or too small: not used). With at least
 *           mxfp4_gemm_workspace_size(M, N, K, 32) bytes and M % 256 == 0,
 *           the call first rewrites sa / sb there as replicated scale images
 *           (four copies of each pair of 512-byte scale tiles) so that the
 *           GEMM moves its scales into tensor memory with half as many
 *           copies. The result is bit-identical either way; the workspace
 *           contents are scratch (overwritten, not read back). */
mxfp4_status mxfp4_gemm_ex(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                           const uint8_t* sb, int64_t M, int64_t N, int64_t K, void* c,
                           int32_t c_dtype, int64_t ldc, void* workspace, size_t workspace_bytes,
                           void* stream);

/* mxfp4_gemm for callers that cannot allocate device memory: code that runs
 * where cudaMalloc is off limits: a framework that owns all device memory
 * through its own pool, a host loop with latency bounds that must not wait on
 * the CUDA allocator, a plugin that is handed only its inputs and
 * outputs. The pages have no counterpart: this is a property of the library,
 * not of the method.
 * It runs the scale-image path of mxfp4_gemm_ex with the workspace taken from
 * a static device array of the library, 96 MiB, which every GPU that loads
 * the library holds until the process exits. The call allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *  - The first call on a device looks up that device's address of the array
 *    (cudaGetSymbolAddress, with the device current); make that first call
 *    before any stream capture on the device.
 *  - The array holds the scale images of the last call. Every call rewrites
 *    all of the bytes it reads, so nothing needs clearing, but calls whose
 *    GEMMs overlap on the GPU (different streams, or different host threads
 *    on one device) race on the array and must be serialised by the caller.
 *  - Shapes as mxfp4_gemm. With M % 256 == 0 the images take
 *    mxfp4_gemm_workspace_size(M, N, K, 32) bytes (4 * (M + N) * K / 32 when
 *    N and K are multiples of 256); above 96 MiB the call returns
 *    MXFP4_ERR_SHAPE before touching the device (M % 256 == 128 uses no images).
 *  - C is bit-identical to mxfp4_gemm's. */
mxfp4_status mxfp4_gemm_noalloc(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                                const uint8_t* sb, int64_t M, int64_t N, int64_t K, float* c,
                                int64_t ldc, void* stream);

/* Workspace bytes for mxfp4_gemm_ex (scale_block 32) or nvfp4_gemm
 * (scale_block 16): four times the scale bytes of both operands, with B's N
 * rounded up to a multiple of 256 and (scale_block 32) A's K rounded up to a
 * multiple of 256: 4 * (M * K' + N' * K) / scale_block (4 * (M + N) * K /
 * scale_block when N and K are multiples of 256). 0 for non-positive sizes
 * or another block. */
size_t mxfp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int32_t scale_block);

/* The MXFP8 counterpart of mxfp4_gemm ([TIBQ], "The fix, and its supporting
 * cast": MXFP8 for queries and keys): qa [M, K] and qb [N, K] E4M3 codes
 * (MXFP4_FORMAT_E4M3, one byte per element), sa / sb E8M0 scales per 32
 * elements in MXFP4_LAYOUT_MMA, C [M, N] = sum_k deqA[m, k] deqB[n, k] in fp32,
 * stored as c_dtype (fp32, or bf16 nearest-even) as in mxfp4_gemm_ex.
 *  Shapes as mxfp4_gemm: M, N and K positive multiples of 128, each at most
 *  2^30 (the K step of one-byte codes is 128 deep; a last 128-row or
 *  128-column tile is computed on zero-filled operands and only its valid
 *  part is stored). */
mxfp4_status mxfp8_gemm(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                        const uint8_t* sb, int64_t M, int64_t N, int64_t K, void* c,
                        int32_t c_dtype, int64_t ldc, void* stream);

/* mxfp8_gemm with the element format named: elem_format MXFP4_FORMAT_E4M3
 * (as mxfp8_gemm) or MXFP4_FORMAT_E5M2 (both operands E5M2 codes, as
 * mxfp4_quantize writes them for that format; kind::mxf8f6f4 with E5M2
 * operands); other values MXFP4_ERR_INVALID_ARG. Shapes and C as mxfp8_gemm. */
mxfp4_status mxfp8_gemm_ex(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                           const uint8_t* sb, int64_t M, int64_t N, int64_t K,
                           uint32_t elem_format, void* c, int32_t c_dtype, int64_t ldc,
                           void* stream);

/* Block-scaled NVFP4 GEMM (the 1 x 16 block format of [TIBQ], "Why FP4
 * training is the current frontier of precision reduction"):
 *   C[m, n] = 2^(ka + kb) * sum_k qa[m, k] SA[m, k/16] * qb[n, k] SB[n, k/16]
 * with E2M1 codes qa [M, K/2], qb [N, K/2], E4M3 scales sa / sb in
 * MXFP4_LAYOUT_MMA with K/16 scale columns (as mxfp4_quantize writes them for
 * MXFP4_BLOCK_1X16), ka / kb the operands' tensor_exp. fp32 accumulation; the
 * factor 2^(ka + kb) is applied exactly to the fp32 sums; C stored as c_dtype
 * (fp32, or bf16 nearest-even) with leading dimension ldc. workspace /
 * workspace_bytes as in mxfp4_gemm_ex, sized by
 * mxfp4_gemm_workspace_size(M, N, K, 16) (six copies per K step instead of
 * twelve; bit-identical result).
 *  Shapes as mxfp4_gemm: M, N and K positive multiples of 128, each at most
 *  2^30; |ka + kb| <= 126. */
mxfp4_status nvfp4_gemm(const uint8_t* qa, const uint8_t* sa, int32_t ka, const uint8_t* qb,
                        const uint8_t* sb, int32_t kb, int64_t M, int64_t N, int64_t K, void* c,
                        int32_t c_dtype, int64_t ldc, void* workspace, size_t workspace_bytes,
                        void* stream);

/* The same GEMM with the quantizer fused into its epilogue ([News], para. 2:
 * the rotation and rounding run where the producing GEMM writes its output).
 * C is quantized straight from the accumulator in one or both orientations,
 * exactly as mxfp4_quantize would quantize the fp32 C this call computes
 * (x = C, rows = M, cols = N):
 *  row  if non-NULL, along N: q_row [M, N/2], s_row ([M, N/32] or
 *       MXFP4_LAYOUT_MMA);
 *  col  if non-NULL, C^T along M (the orientation the next layer's Wgrad
 *       consumes): q_col [N, M/2], s_col ([N, M/32] or MXFP4_LAYOUT_MMA).
 * At least one of row / col must be non-NULL. Any block (except 64x64 and
 * 1x16: MXFP4_ERR_UNSUPPORTED), scale mode, rounding, rotation, element
 * format and scale layout mxfp4_quantize accepts; stochastic draws are keyed
 * by the element index m * N + n of C in both orientations. The codes come
 * from the fp32 sums even when C itself is stored as bf16 (c_dtype as in
 * mxfp4_gemm_ex). c may be NULL: then no C is written (c_dtype and ldc are
 * ignored), which saves its HBM traffic. workspace / workspace_bytes as in
 * mxfp4_gemm_ex (used for row-wise-only outputs; same bits either way).
 *  Shapes as mxfp4_gemm. q_row / q_col must be 16-byte aligned. */
mxfp4_status mxfp4_gemm_quantize(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                                 const uint8_t* sb, int64_t M, int64_t N, int64_t K, void* c,
                                 int32_t c_dtype, int64_t ldc, const mxfp4_quant_params* row,
                                 uint8_t* q_row, uint8_t* s_row, const mxfp4_quant_params* col,
                                 uint8_t* q_col, uint8_t* s_col, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Stand-alone 32-point block rotation along cols ([News], para. 2):
 *  forward (inverse == 0): y = c * H * diag(s) * x per 32-block;
 *  inverse (inverse == 1): y = diag(s) * c * H * x.
 *  x [rows, cols] bf16/fp32 with ld_x; y [rows, cols] fp32 dense; cols % 32 == 0
 *  and at most 2^40 elements (else MXFP4_ERR_SHAPE).
 *  The forward rotation is bit-identical to the one mxfp4_quantize fuses. */
mxfp4_status hadamard32(const void* x, int32_t x_dtype, int64_t rows, int64_t cols,
                        int64_t ld_x, uint32_t sign_mask, int32_t inverse, float* y,
                        void* stream);

/* The per-tensor factor of the 1x16 block format ([TIBQ], "Why FP4 training
 * is the current frontier of precision reduction": NVFP4 blocks whose scale
 * follows the block max-abs, under a tensor-wide factor): computed on the
 * device so a training step can carry it to the next step without a host
 * round trip.
 *  x          [rows, cols] bf16 or fp32 (x_dtype), leading dimension ld_x;
 *             cols % 32 == 0, at most 2^40 elements (else MXFP4_ERR_SHAPE);
 *             16-byte aligned with ld_x % 8 == 0 (else MXFP4_ERR_ALIGN).
 *  amax       device pointer to one float (4-byte aligned): receives the
 *             largest |x| (0 for an empty tensor).
 *  tensor_exp device pointer to one int32 or NULL: receives the smallest k
 *             with 2688 * 2^k >= amax (2688 = 6 * 448: the largest block
 *             scale amax / (6 * 2^k) then fits E4M3), clamped to [-100, 100],
 *             0 when amax is 0 -- the tensor_exp mxfp4_quantize takes for
 *             MXFP4_BLOCK_1X16.
 * Enqueued on `stream` (a memset of *amax, the reduction, and a one-thread
 * kernel for tensor_exp). Inputs must be finite. */
mxfp4_status mxfp4_tensor_amax(const void* x, int32_t x_dtype, int64_t rows, int64_t cols,
                               int64_t ld_x, float* amax, int32_t* tensor_exp, void* stream);

/* Human-readable name of a status code (static string). */
const char* mxfp4_status_string(mxfp4_status s);

/* Detail of the last non-OK status returned on the calling thread. */
const char* mxfp4_last_error(void);

/* Reads and clears the device-side error word that bounded waits inside the
 * GEMM kernel set when they run out (MXFP4_OK if none). Synchronizes `stream`
 * first. */
mxfp4_status mxfp4_device_status(void* stream);

/* Diagnostic of the bounds-checking build (the pages have no counterpart).
 * A library built with MXFP4_BOUNDS_CHECK checks every store of its kernels
 * against the extent the call computed for that output (codes, scales, C,
 * rotated or reconstructed values, scale images); a store outside it is
 * skipped and mxfp4_device_status then returns MXFP4_ERR_BOUNDS. This call
 * makes the code and scale extents of later calls on the calling thread
 * `bytes` smaller (0 restores them), so a test can watch the check fire while
 * every store that does happen stays inside its real buffer. The regular
 * library returns MXFP4_ERR_UNSUPPORTED. */
mxfp4_status mxfp4_bounds_check_shrink(int64_t bytes);

/* Diagnostic for the library's own failure reporting (the pages have no
 * counterpart). Enqueues on `stream` a one-thread kernel that waits on a
 * device barrier nothing ever signals; the wait gives up after its limit
 * (about 2 s), records MXFP4_ERR_TIMEOUT in the device error word exactly as
 * a GEMM wait that ran out would, and the kernel returns, leaving the context
 * usable. Returns the launch status; read the outcome with
 * mxfp4_device_status (which also clears it). */
mxfp4_status mxfp4_selftest_wait_timeout(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MXFP4_H */
