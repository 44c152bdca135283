// api.cu -- the extern "C" entry points declared in include/mxfp4.h:
// argument validation, status codes and the thread-local error detail; the
// work itself is enqueued by the launchers in quant.cu and gemm.cu.
#include <cstdarg>
#include <cstdint>
#include <cmath>
#include <cstdio>

#include "../../include/mxfp4.h"
#include "internal.h"

namespace {

thread_local char g_last_error[512] = "";
// Bounds-checking builds: bytes taken off every output extent this thread's
// later calls check against (mxfp4_bounds_check_shrink).
thread_local int64_t g_extent_shrink = 0;

mxfp4_status fail(mxfp4_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mxfp4_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MXFP4_OK;
  return fail(MXFP4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Validates one orientation's parameters and fills the launcher's view.
mxfp4_status check_params(const mxfp4_quant_params* p, uint8_t* q, uint8_t* s, int64_t out_rows,
                          int64_t k, const char* name, mx::OrientArgs* o) {
  if ((!q || !s) && out_rows * k > 0)
    return fail(MXFP4_ERR_INVALID_ARG, "%s: output pointers must be non-NULL", name);
  if (!aligned16(q)) return fail(MXFP4_ERR_ALIGN, "%s: codes pointer not 16-byte aligned", name);
  if (p->block != MXFP4_BLOCK_1X32 && p->block != MXFP4_BLOCK_32X32 &&
      p->block != MXFP4_BLOCK_64X64 && p->block != MXFP4_BLOCK_1X16)
    return fail(MXFP4_ERR_INVALID_ARG, "%s: bad block %d", name, p->block);
  const bool nv = p->block == MXFP4_BLOCK_1X16;
  if (nv && (p->tensor_exp < -100 || p->tensor_exp > 100))
    return fail(MXFP4_ERR_INVALID_ARG, "%s: tensor_exp %d outside [-100, 100]", name, p->tensor_exp);
  if (!nv && p->tensor_exp != 0)
    return fail(MXFP4_ERR_INVALID_ARG, "%s: tensor_exp is for 1x16 (NVFP4) blocks only", name);
  if (nv && p->elem_format != MXFP4_FORMAT_E2M1)
    return fail(MXFP4_ERR_UNSUPPORTED, "%s: 1x16 blocks take E2M1 elements", name);
  if (p->block == MXFP4_BLOCK_64X64 && (out_rows % 64 != 0 || k % 64 != 0))
    return fail(MXFP4_ERR_SHAPE, "%s: 64x64 blocks need rows %% 64 == 0 and K %% 64 == 0 (got %lld x %lld)",
                name, (long long)out_rows, (long long)k);
  if (p->scale_mode != MXFP4_SCALE_FLOOR && p->scale_mode != MXFP4_SCALE_ROUNDUP)
    return fail(MXFP4_ERR_INVALID_ARG, "%s: bad scale_mode %d", name, p->scale_mode);
  if (p->rounding != MXFP4_ROUND_RTN && p->rounding != MXFP4_ROUND_SR)
    return fail(MXFP4_ERR_INVALID_ARG, "%s: bad rounding %d", name, p->rounding);
  if (p->scale_layout != MXFP4_LAYOUT_ROWMAJOR && p->scale_layout != MXFP4_LAYOUT_MMA)
    return fail(MXFP4_ERR_INVALID_ARG, "%s: bad scale_layout %d", name, p->scale_layout);
  if (p->wht != 0 && p->wht != 1) return fail(MXFP4_ERR_INVALID_ARG, "%s: wht must be 0/1", name);
  if (p->elem_format != MXFP4_FORMAT_E2M1 && p->elem_format != MXFP4_FORMAT_E4M3 &&
      p->elem_format != MXFP4_FORMAT_E5M2)
    return fail(MXFP4_ERR_INVALID_ARG, "%s: bad elem_format %u", name, p->elem_format);
  if (p->elem_format != MXFP4_FORMAT_E2M1 && p->rounding == MXFP4_ROUND_SR)
    return fail(MXFP4_ERR_UNSUPPORTED, "%s: stochastic rounding is available for E2M1 only", name);
  if (p->scale_layout == MXFP4_LAYOUT_MMA && (out_rows % 128 != 0 || k % 128 != 0))
    return fail(MXFP4_ERR_SHAPE,
                "%s: tensor-core scale layout needs rows %% 128 == 0 and K %% 128 == 0 (got %lld x %lld)",
                name, (long long)out_rows, (long long)k);
  o->block = nv ? 0 : p->block;
  o->nv = nv;
  o->nv_p2k = nv ? ldexpf(1.0f, p->tensor_exp) : 1.0f;
  o->nv_zmul = nv ? (float)(ldexp(1.0, -p->tensor_exp) / 6.0) : 1.0f;
  o->roundup = p->scale_mode == MXFP4_SCALE_ROUNDUP;
  o->sr = p->rounding == MXFP4_ROUND_SR;
  o->mma_layout = p->scale_layout == MXFP4_LAYOUT_MMA;
  o->wht = p->wht;
  o->e4m3 = p->elem_format == MXFP4_FORMAT_E4M3 || p->elem_format == MXFP4_FORMAT_E5M2;
  o->e5m2 = p->elem_format == MXFP4_FORMAT_E5M2;
  o->sign_mask = p->wht_sign_mask;
  o->seed = p->seed;
  o->stream = p->sr_stream;
  o->q = q;
  o->s = s;
  const int64_t qb = out_rows * (o->e4m3 ? k : k / 2), sb = out_rows * (nv ? k / 16 : k / 32);
  o->q_bytes = (uint64_t)(qb > g_extent_shrink ? qb - g_extent_shrink : 0);
  o->s_bytes = (uint64_t)(sb > g_extent_shrink ? sb - g_extent_shrink : 0);
  mx::prepare_orient(o);
  return MXFP4_OK;
}

// Element counts above 2^40 (2 TB of bf16) cannot be resident on one GPU;
// rejecting them first keeps every size product below int64's range.
constexpr int64_t kMaxElems = (int64_t)1 << 40;

bool too_large(int64_t rows, int64_t cols) { return rows > 0 && cols > kMaxElems / rows; }

mxfp4_status check_input(const void* x, int32_t dtype, int64_t rows, int64_t cols, int64_t ld) {
  if (dtype != MXFP4_DTYPE_BF16 && dtype != MXFP4_DTYPE_F32)
    return fail(MXFP4_ERR_INVALID_ARG, "bad x_dtype %d", dtype);
  if (rows < 0 || cols < 0) return fail(MXFP4_ERR_SHAPE, "negative dimension");
  if (too_large(rows, cols)) return fail(MXFP4_ERR_SHAPE, "tensor too large (more than 2^40 elements)");
  if (!x && rows * cols > 0) return fail(MXFP4_ERR_INVALID_ARG, "x is NULL");
  if (cols % 32 != 0) return fail(MXFP4_ERR_SHAPE, "cols (%lld) must be a multiple of 32", (long long)cols);
  if (ld < cols) return fail(MXFP4_ERR_SHAPE, "ld_x (%lld) < cols (%lld)", (long long)ld, (long long)cols);
  if (!aligned16(x) || ld % 8 != 0)
    return fail(MXFP4_ERR_ALIGN, "x must be 16-byte aligned with ld_x %% 8 == 0");
  return MXFP4_OK;
}

}  // namespace

extern "C" {

const char* mxfp4_status_string(mxfp4_status s) {
  switch (s) {
    case MXFP4_OK: return "MXFP4_OK";
    case MXFP4_ERR_INVALID_ARG: return "MXFP4_ERR_INVALID_ARG";
    case MXFP4_ERR_SHAPE: return "MXFP4_ERR_SHAPE";
    case MXFP4_ERR_ALIGN: return "MXFP4_ERR_ALIGN";
    case MXFP4_ERR_UNSUPPORTED: return "MXFP4_ERR_UNSUPPORTED";
    case MXFP4_ERR_CUDA: return "MXFP4_ERR_CUDA";
    case MXFP4_ERR_TIMEOUT: return "MXFP4_ERR_TIMEOUT";
    case MXFP4_ERR_BOUNDS: return "MXFP4_ERR_BOUNDS";
  }
  return "MXFP4_ERR_UNKNOWN";
}

const char* mxfp4_last_error(void) { return g_last_error; }

mxfp4_status mxfp4_quantize(const void* x, int32_t x_dtype, int64_t rows, int64_t cols,
                            int64_t ld_x, const mxfp4_quant_params* row, uint8_t* q_row,
                            uint8_t* s_row, const mxfp4_quant_params* col, uint8_t* q_col,
                            uint8_t* s_col, void* stream) {
  if (!row && !col) return fail(MXFP4_ERR_INVALID_ARG, "at least one of row / col params is required");
  mxfp4_status st = check_input(x, x_dtype, rows, cols, ld_x);
  if (st) return st;
  // The row kernel counts 16-element units in 32 bits: units < 2^31 plus a
  // grid stride < 2^31 keeps every index it forms below 2^32.
  if (rows > 0 && cols / 16 > (int64_t)0x7FFFFFFF / rows)
    return fail(MXFP4_ERR_SHAPE, "tensor too large: rows * cols / 16 must be below 2^31");
  const bool need_rows32 =
      col || (row && row->block != MXFP4_BLOCK_1X32 && row->block != MXFP4_BLOCK_1X16);
  if (need_rows32 && rows % 32 != 0)
    return fail(MXFP4_ERR_SHAPE, "rows (%lld) must be a multiple of 32 for column-wise or 32x32 output",
                (long long)rows);
  mx::OrientArgs ro{}, co{};
  if (row && (st = check_params(row, q_row, s_row, rows, cols, "row", &ro))) return st;
  if (col && (st = check_params(col, q_col, s_col, cols, rows, "col", &co))) return st;
  return from_cuda(mx::launch_quantize(x, x_dtype == MXFP4_DTYPE_F32, rows, cols, ld_x,
                                       row ? &ro : nullptr, col ? &co : nullptr,
                                       static_cast<cudaStream_t>(stream)),
                   "mxfp4_quantize launch");
}

namespace {
mxfp4_status dequantize_common(const char* name, const uint8_t* q, const uint8_t* s,
                               int32_t scale_layout, int fmt, int32_t tensor_exp, int64_t rows,
                               int64_t cols, float* out, void* stream) {
  if (scale_layout != MXFP4_LAYOUT_ROWMAJOR && scale_layout != MXFP4_LAYOUT_MMA)
    return fail(MXFP4_ERR_INVALID_ARG, "%s: bad scale_layout %d", name, scale_layout);
  if (rows < 0 || cols < 0 || cols % 32 != 0)
    return fail(MXFP4_ERR_SHAPE, "%s: cols (%lld) must be a non-negative multiple of 32", name,
                (long long)cols);
  if (too_large(rows, cols)) return fail(MXFP4_ERR_SHAPE, "%s: tensor too large (more than 2^40 elements)", name);
  if ((!q || !s || !out) && rows * cols > 0) return fail(MXFP4_ERR_INVALID_ARG, "%s: NULL pointer", name);
  if (scale_layout == MXFP4_LAYOUT_MMA && (rows % 128 != 0 || cols % 128 != 0))
    return fail(MXFP4_ERR_SHAPE, "%s: tensor-core scale layout needs rows and cols %% 128 == 0", name);
  if (!aligned16(q) || !aligned16(out))
    return fail(MXFP4_ERR_ALIGN, "%s: q / out must be 16-byte aligned", name);
  return from_cuda(mx::launch_dequantize(q, s, scale_layout == MXFP4_LAYOUT_MMA, rows, cols, fmt,
                                         ldexpf(1.0f, tensor_exp), out,
                                         static_cast<cudaStream_t>(stream)),
                   name);
}
}  // namespace

mxfp4_status mxfp4_dequantize(const uint8_t* q, const uint8_t* s, int32_t scale_layout,
                              int64_t rows, int64_t cols, float* out, void* stream) {
  return dequantize_common("mxfp4_dequantize", q, s, scale_layout, 0, 0, rows, cols, out, stream);
}

mxfp4_status mxfp4_dequantize_ex(const uint8_t* q, const uint8_t* s, int32_t scale_layout,
                                 int32_t block, uint32_t elem_format, int32_t tensor_exp,
                                 int64_t rows, int64_t cols, float* out, void* stream) {
  if (block != MXFP4_BLOCK_1X32 && block != MXFP4_BLOCK_32X32 && block != MXFP4_BLOCK_64X64 &&
      block != MXFP4_BLOCK_1X16)
    return fail(MXFP4_ERR_INVALID_ARG, "mxfp4_dequantize_ex: bad block %d", block);
  if (elem_format != MXFP4_FORMAT_E2M1 && elem_format != MXFP4_FORMAT_E4M3 &&
      elem_format != MXFP4_FORMAT_E5M2)
    return fail(MXFP4_ERR_INVALID_ARG, "mxfp4_dequantize_ex: bad elem_format %u", elem_format);
  const bool nv = block == MXFP4_BLOCK_1X16;
  if (nv && elem_format != MXFP4_FORMAT_E2M1)
    return fail(MXFP4_ERR_UNSUPPORTED, "mxfp4_dequantize_ex: 1x16 blocks take E2M1 elements");
  if (nv ? (tensor_exp < -100 || tensor_exp > 100) : tensor_exp != 0)
    return fail(MXFP4_ERR_INVALID_ARG, "mxfp4_dequantize_ex: bad tensor_exp %d", tensor_exp);
  const int fmt = nv ? 2 : (elem_format == MXFP4_FORMAT_E4M3 ? 1 : (elem_format == MXFP4_FORMAT_E5M2 ? 3 : 0));
  return dequantize_common("mxfp4_dequantize_ex", q, s, scale_layout, fmt, tensor_exp, rows, cols,
                           out, stream);
}

namespace {
// Shape rules of the GEMM entry points (MXFP4, MXFP8, NVFP4).
mxfp4_status gemm_shape(const char* name, int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || M % 128 != 0 || N % 128 != 0 || K % 128 != 0)
    return fail(MXFP4_ERR_SHAPE, "%s needs M, N, K positive multiples of 128 (got %lld, %lld, %lld)",
                name, (long long)M, (long long)N, (long long)K);
  if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30) || (M / 128) * (N / 128) > (1ll << 30))
    return fail(MXFP4_ERR_SHAPE, "%s dimensions too large", name);
  return MXFP4_OK;
}

mxfp4_status gemm_common(const char* name, const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                         const uint8_t* sb, int64_t M, int64_t N, int64_t K, void* c,
                         int32_t c_dtype, int64_t ldc, const mx::OrientArgs* qout,
                         const mx::OrientArgs* qcol, void* ws, size_t ws_bytes, void* stream) {
  if (!qa || !sa || !qb || !sb || (!c && !qout && !qcol))
    return fail(MXFP4_ERR_INVALID_ARG, "%s: NULL pointer", name);
  if (c_dtype != MXFP4_DTYPE_BF16 && c_dtype != MXFP4_DTYPE_F32)
    return fail(MXFP4_ERR_INVALID_ARG, "%s: bad c_dtype %d", name, c_dtype);
  if (mxfp4_status st = gemm_shape(name, M, N, K)) return st;
  if (c && ldc < N) return fail(MXFP4_ERR_SHAPE, "ldc (%lld) < N (%lld)", (long long)ldc, (long long)N);
  if (!aligned16(qa) || !aligned16(qb) || !aligned16(sa) || !aligned16(sb) || !aligned16(c) ||
      (c && ldc % 8 != 0))
    return fail(MXFP4_ERR_ALIGN, "operands must be 16-byte aligned and ldc %% 8 == 0");
  if (ws && !aligned16(ws)) return fail(MXFP4_ERR_ALIGN, "%s: workspace must be 16-byte aligned", name);
  const char* why = "";
  cudaError_t e = mx::launch_gemm(qa, sa, qb, sb, M, N, K, c, c_dtype == MXFP4_DTYPE_BF16, ldc,
                                  qout, qcol, ws, ws_bytes, static_cast<cudaStream_t>(stream), &why);
  if (e == cudaErrorNotSupported) return fail(MXFP4_ERR_UNSUPPORTED, "%s", why);
  if (e == cudaErrorInvalidValue && why[0]) return fail(MXFP4_ERR_ALIGN, "%s", why);
  return from_cuda(e, name);
}
}  // namespace

mxfp4_status mxfp4_gemm(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                        const uint8_t* sb, int64_t M, int64_t N, int64_t K, float* c,
                        int64_t ldc, void* stream) {
  if (!c) return fail(MXFP4_ERR_INVALID_ARG, "NULL pointer");
  return gemm_common("mxfp4_gemm", qa, sa, qb, sb, M, N, K, c, MXFP4_DTYPE_F32, ldc, nullptr,
                     nullptr, nullptr, 0, stream);
}

mxfp4_status mxfp4_gemm_noalloc(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                                const uint8_t* sb, int64_t M, int64_t N, int64_t K, float* c,
                                int64_t ldc, void* stream) {
  if (!c) return fail(MXFP4_ERR_INVALID_ARG, "NULL pointer");
  if (mxfp4_status st = gemm_shape("mxfp4_gemm_noalloc", M, N, K)) return st;
  // Only the CTA-pair kernel (M % 256 == 0) reads scale images; the dimensions
  // are validated above, so the image size cannot overflow.
  if (M % 256 == 0 && mx::workspace_bytes(M, N, K, false) > (int64_t)mx::kStaticScratchBytes)
    return fail(MXFP4_ERR_SHAPE,
                "mxfp4_gemm_noalloc: scale images of %lld x %lld x %lld exceed the static scratch (%zu bytes)",
                (long long)M, (long long)N, (long long)K, mx::kStaticScratchBytes);
  void* ws = nullptr;
  const cudaError_t e = mx::static_scratch(&ws);
  if (e != cudaSuccess) return from_cuda(e, "mxfp4_gemm_noalloc: static scratch");
  return gemm_common("mxfp4_gemm_noalloc", qa, sa, qb, sb, M, N, K, c, MXFP4_DTYPE_F32, ldc, nullptr,
                     nullptr, ws, mx::kStaticScratchBytes, stream);
}

size_t mxfp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int32_t scale_block) {
  if (M <= 0 || N <= 0 || K <= 0 || (scale_block != 32 && scale_block != 16)) return 0;
  return (size_t)mx::workspace_bytes(M, N, K, scale_block == 16);
}

mxfp4_status mxfp4_gemm_ex(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                           const uint8_t* sb, int64_t M, int64_t N, int64_t K, void* c,
                           int32_t c_dtype, int64_t ldc, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (!c) return fail(MXFP4_ERR_INVALID_ARG, "NULL pointer");
  return gemm_common("mxfp4_gemm_ex", qa, sa, qb, sb, M, N, K, c, c_dtype, ldc, nullptr, nullptr,
                     workspace, workspace_bytes, stream);
}

namespace {
mxfp4_status mxfp8_common(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                          const uint8_t* sb, int64_t M, int64_t N, int64_t K, uint32_t elem_format,
                          void* c, int32_t c_dtype, int64_t ldc, void* stream) {
  if (!qa || !sa || !qb || !sb || !c) return fail(MXFP4_ERR_INVALID_ARG, "mxfp8_gemm: NULL pointer");
  if (elem_format != MXFP4_FORMAT_E4M3 && elem_format != MXFP4_FORMAT_E5M2)
    return fail(MXFP4_ERR_INVALID_ARG, "mxfp8_gemm: elem_format %u is not E4M3 or E5M2", elem_format);
  if (c_dtype != MXFP4_DTYPE_BF16 && c_dtype != MXFP4_DTYPE_F32)
    return fail(MXFP4_ERR_INVALID_ARG, "mxfp8_gemm: bad c_dtype %d", c_dtype);
  if (mxfp4_status st = gemm_shape("mxfp8_gemm", M, N, K)) return st;
  if (ldc < N) return fail(MXFP4_ERR_SHAPE, "ldc (%lld) < N (%lld)", (long long)ldc, (long long)N);
  if (!aligned16(qa) || !aligned16(qb) || !aligned16(sa) || !aligned16(sb) || !aligned16(c) || ldc % 8 != 0)
    return fail(MXFP4_ERR_ALIGN, "operands must be 16-byte aligned and ldc %% 8 == 0");
  const char* why = "";
  cudaError_t e = mx::launch_gemm_f8(qa, sa, qb, sb, M, N, K, elem_format == MXFP4_FORMAT_E5M2, c,
                                     c_dtype == MXFP4_DTYPE_BF16, ldc,
                                     static_cast<cudaStream_t>(stream), &why);
  if (e == cudaErrorNotSupported) return fail(MXFP4_ERR_UNSUPPORTED, "%s", why);
  if (e == cudaErrorInvalidValue && why[0]) return fail(MXFP4_ERR_ALIGN, "%s", why);
  return from_cuda(e, "mxfp8_gemm");
}
}  // namespace

mxfp4_status mxfp8_gemm(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                        const uint8_t* sb, int64_t M, int64_t N, int64_t K, void* c,
                        int32_t c_dtype, int64_t ldc, void* stream) {
  return mxfp8_common(qa, sa, qb, sb, M, N, K, MXFP4_FORMAT_E4M3, c, c_dtype, ldc, stream);
}

mxfp4_status mxfp8_gemm_ex(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                           const uint8_t* sb, int64_t M, int64_t N, int64_t K,
                           uint32_t elem_format, void* c, int32_t c_dtype, int64_t ldc,
                           void* stream) {
  return mxfp8_common(qa, sa, qb, sb, M, N, K, elem_format, c, c_dtype, ldc, stream);
}

mxfp4_status nvfp4_gemm(const uint8_t* qa, const uint8_t* sa, int32_t ka, const uint8_t* qb,
                        const uint8_t* sb, int32_t kb, int64_t M, int64_t N, int64_t K, void* c,
                        int32_t c_dtype, int64_t ldc, void* workspace, size_t workspace_bytes,
                        void* stream) {
  if (!qa || !sa || !qb || !sb || !c) return fail(MXFP4_ERR_INVALID_ARG, "nvfp4_gemm: NULL pointer");
  if (c_dtype != MXFP4_DTYPE_BF16 && c_dtype != MXFP4_DTYPE_F32)
    return fail(MXFP4_ERR_INVALID_ARG, "nvfp4_gemm: bad c_dtype %d", c_dtype);
  if (ka < -100 || ka > 100 || kb < -100 || kb > 100 || ka + kb < -126 || ka + kb > 126)
    return fail(MXFP4_ERR_INVALID_ARG, "nvfp4_gemm: tensor exponents %d, %d out of range", ka, kb);
  if (mxfp4_status st = gemm_shape("nvfp4_gemm", M, N, K)) return st;
  if (ldc < N) return fail(MXFP4_ERR_SHAPE, "ldc (%lld) < N (%lld)", (long long)ldc, (long long)N);
  if (!aligned16(qa) || !aligned16(qb) || !aligned16(sa) || !aligned16(sb) || !aligned16(c) || ldc % 8 != 0)
    return fail(MXFP4_ERR_ALIGN, "operands must be 16-byte aligned and ldc %% 8 == 0");
  if (workspace && !aligned16(workspace))
    return fail(MXFP4_ERR_ALIGN, "nvfp4_gemm: workspace must be 16-byte aligned");
  const char* why = "";
  cudaError_t e = mx::launch_gemm_nv(qa, sa, qb, sb, M, N, K, ldexpf(1.0f, ka + kb), c,
                                     c_dtype == MXFP4_DTYPE_BF16, ldc, workspace, workspace_bytes,
                                     static_cast<cudaStream_t>(stream), &why);
  if (e == cudaErrorNotSupported) return fail(MXFP4_ERR_UNSUPPORTED, "%s", why);
  if (e == cudaErrorInvalidValue && why[0]) return fail(MXFP4_ERR_ALIGN, "%s", why);
  return from_cuda(e, "nvfp4_gemm");
}

mxfp4_status mxfp4_gemm_quantize(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                                 const uint8_t* sb, int64_t M, int64_t N, int64_t K, void* c,
                                 int32_t c_dtype, int64_t ldc, const mxfp4_quant_params* row,
                                 uint8_t* q_row, uint8_t* s_row, const mxfp4_quant_params* col,
                                 uint8_t* q_col, uint8_t* s_col, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (!row && !col)
    return fail(MXFP4_ERR_INVALID_ARG, "mxfp4_gemm_quantize: row or col params are required");
  for (const mxfp4_quant_params* p : {row, col}) {
    if (p && p->block == MXFP4_BLOCK_64X64)
      return fail(MXFP4_ERR_UNSUPPORTED,
                  "mxfp4_gemm_quantize: 64x64 blocks span two epilogue warps; quantize C separately");
    if (p && p->block == MXFP4_BLOCK_1X16)
      return fail(MXFP4_ERR_UNSUPPORTED,
                  "mxfp4_gemm_quantize: 1x16 (NVFP4) output is not fused; quantize C separately");
  }
  mx::OrientArgs ro{}, co{};
  if (M > 0 && N > 0) {
    mxfp4_status st;
    if (row && (st = check_params(row, q_row, s_row, M, N, "row", &ro))) return st;
    if (col && (st = check_params(col, q_col, s_col, N, M, "col", &co))) return st;
  }
  return gemm_common("mxfp4_gemm_quantize", qa, sa, qb, sb, M, N, K, c, c_dtype, ldc,
                     row ? &ro : nullptr, col ? &co : nullptr, workspace, workspace_bytes, stream);
}

mxfp4_status hadamard32(const void* x, int32_t x_dtype, int64_t rows, int64_t cols,
                        int64_t ld_x, uint32_t sign_mask, int32_t inverse, float* y,
                        void* stream) {
  mxfp4_status st = check_input(x, x_dtype, rows, cols, ld_x);
  if (st) return st;
  if (!y && rows * cols > 0) return fail(MXFP4_ERR_INVALID_ARG, "y is NULL");
  if (!aligned16(y)) return fail(MXFP4_ERR_ALIGN, "y must be 16-byte aligned");
  if (inverse != 0 && inverse != 1) return fail(MXFP4_ERR_INVALID_ARG, "inverse must be 0/1");
  return from_cuda(mx::launch_hadamard32(x, x_dtype == MXFP4_DTYPE_F32, rows, cols, ld_x, sign_mask,
                                         inverse != 0, y, static_cast<cudaStream_t>(stream)),
                   "hadamard32 launch");
}

mxfp4_status mxfp4_tensor_amax(const void* x, int32_t x_dtype, int64_t rows, int64_t cols,
                               int64_t ld_x, float* amax, int32_t* tensor_exp, void* stream) {
  mxfp4_status st = check_input(x, x_dtype, rows, cols, ld_x);
  if (st) return st;
  if (!amax) return fail(MXFP4_ERR_INVALID_ARG, "mxfp4_tensor_amax: amax is NULL");
  if ((reinterpret_cast<uintptr_t>(amax) & 3u) || (reinterpret_cast<uintptr_t>(tensor_exp) & 3u))
    return fail(MXFP4_ERR_ALIGN, "mxfp4_tensor_amax: amax / tensor_exp must be 4-byte aligned");
  return from_cuda(mx::launch_amax(x, x_dtype == MXFP4_DTYPE_F32, rows, cols, ld_x, amax, tensor_exp,
                                   static_cast<cudaStream_t>(stream)),
                   "mxfp4_tensor_amax launch");
}

mxfp4_status mxfp4_device_status(void* stream) {
  uint32_t err = 0;
  cudaError_t e = mx::read_device_error(static_cast<cudaStream_t>(stream), &err);
  if (e != cudaSuccess) return from_cuda(e, "mxfp4_device_status");
  if (err == MXFP4_ERR_TIMEOUT)
    return fail(MXFP4_ERR_TIMEOUT, "a bounded device-side wait in the GEMM ran out");
  if (err == MXFP4_ERR_BOUNDS)
    return fail(MXFP4_ERR_BOUNDS, "a kernel store fell outside its output (skipped)");
  return err ? fail(static_cast<mxfp4_status>(err), "device error word %u", err) : MXFP4_OK;
}

mxfp4_status mxfp4_bounds_check_shrink(int64_t bytes) {
#ifdef MXFP4_BOUNDS_CHECK
  if (bytes < 0) return fail(MXFP4_ERR_INVALID_ARG, "mxfp4_bounds_check_shrink: negative bytes");
  g_extent_shrink = bytes;
  return MXFP4_OK;
#else
  (void)bytes;
  return fail(MXFP4_ERR_UNSUPPORTED, "mxfp4_bounds_check_shrink: not a bounds-checking build");
#endif
}

mxfp4_status mxfp4_selftest_wait_timeout(void* stream) {
  cudaError_t e = mx::launch_wait_probe(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return from_cuda(e, "mxfp4_selftest_wait_timeout");
  return MXFP4_OK;
}

}  // extern "C"
