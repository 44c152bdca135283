// quant_device.cuh -- per-run quantization steps shared by the quantizer
// kernels and the GEMM epilogue that quantizes its output (sm_103a).
#pragma once
#include <cstdint>

#include "internal.h"
#include "mx_device.cuh"

// Each translation unit that includes this header defines MX_BOUNDS_FAIL()
// (raise its device error word to kErrBounds) first.
#ifndef MX_BOUNDS_FAIL
#error "define MX_BOUNDS_FAIL() before including quant_device.cuh"
#endif

namespace mx {

// Store v at p. Builds with MXFP4_BOUNDS_CHECK first check that the store lies
// inside [base, base + bytes), the extent the boundary computed for the output;
// a store outside it is skipped and raises the device error word.
template <typename T>
__device__ __forceinline__ void put(T* p, const T& v, const void* base, uint64_t bytes) {
#ifdef MXFP4_BOUNDS_CHECK
  const uint8_t* b = static_cast<const uint8_t*>(base);
  const uint8_t* a = reinterpret_cast<const uint8_t*>(p);
  if (a < b || a + sizeof(T) > b + bytes) {
    MX_BOUNDS_FAIL();
    return;
  }
#else
  (void)base;
  (void)bytes;
#endif
  *p = v;
}

__device__ __forceinline__ int64_t scale_offset(const OrientArgs& o, int64_t orow, int64_t kb,
                                                int64_t nkb) {
  return o.mma_layout ? mma_scale_offset(orow, kb, nkb) : orow * nkb + kb;
}

// The quantizer kernels' 32-bit forms of the scale offset, scale stores and
// draws: their size limit (rows * cols / 16 < 2^31) keeps every scale offset
// below 2^31 and every draw counter i / 8 below 2^32, and 32-bit index
// arithmetic measured 2-4 % faster there. The GEMM epilogue, whose C can
// exceed that size, keeps the 64-bit forms (as does the general tile
// variant, which spilled registers with the 32-bit ones).
__device__ __forceinline__ uint32_t scale_offset32(const OrientArgs& o, uint32_t orow, uint32_t kb,
                                                   uint32_t nkb) {
  return o.mma_layout ? (((orow >> 7) * (nkb >> 2) + (kb >> 2)) << 9) + ((orow & 31) << 4) +
                            (((orow >> 5) & 3) << 2) + (kb & 3)
                      : orow * nkb + kb;
}

__device__ __forceinline__ void store_scale32(const OrientArgs& o, uint32_t orow, uint32_t kb,
                                              uint32_t nkb, int e) {
  put(o.s + scale_offset32(o, orow, kb, nkb), (uint8_t)(e + 127), o.s, o.s_bytes);
}

template <bool kNvfp4 = true>
__device__ __forceinline__ void store_run_scales32(const OrientArgs& o, uint32_t orow, uint32_t k0,
                                                   uint32_t K, int e) {
  if (kNvfp4 && o.nv)
    put(reinterpret_cast<uint16_t*>(o.s + scale_offset32(o, orow, k0 >> 4, K >> 4)), (uint16_t)e, o.s,
        o.s_bytes);
  else
    store_scale32(o, orow, k0 >> 5, K >> 5, e);
}

// Draw words for source elements 8 g0 .. 8 g0 + 31 (counter low words g0 ..
// g0 + 3, high words 0).
__device__ __forceinline__ void draws32_g(const PhiloxKeys& k, uint32_t stream, uint32_t g0,
                                          uint32_t (&w)[16]) {
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const U4 a = philox4x32_10(U4{g0 + (uint32_t)h, 0u, stream, 0u}, k);
    w[4 * h] = a.x; w[4 * h + 1] = a.y; w[4 * h + 2] = a.z; w[4 * h + 3] = a.w;
  }
}

// E8M0 scale 2^e of block kb of output row orow (nkb blocks per row).
__device__ __forceinline__ void store_scale(const OrientArgs& o, int64_t orow, int64_t kb,
                                            int64_t nkb, int e) {
  put(o.s + scale_offset(o, orow, kb, nkb), (uint8_t)(e + 127), o.s, o.s_bytes);
}

// The scales of the 32-run at K positions k0 .. k0 + 31 of output row orow as
// scale_run32 returns them: one E8M0 byte, or (NVFP4) the E4M3 codes of its
// two 16-blocks, which are adjacent in both layouts (k0 / 16 is even).
template <bool kNvfp4 = true>
__device__ __forceinline__ void store_run_scales(const OrientArgs& o, int64_t orow, int64_t k0,
                                                 int64_t K, int e) {
  if (kNvfp4 && o.nv)
    put(reinterpret_cast<uint16_t*>(o.s + scale_offset(o, orow, k0 >> 4, K >> 4)), (uint16_t)e, o.s,
        o.s_bytes);
  else
    store_scale(o, orow, k0 >> 5, K >> 5, e);
}

// Draw words for 32 consecutive source elements i0 .. i0 + 31 (i0 % 32 == 0).
__device__ __forceinline__ void draws32(const PhiloxKeys& k, uint32_t stream, uint64_t i0,
                                        uint32_t (&w)[16]) {
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const uint64_t g = (i0 >> 3) + h;
    const U4 a = philox4x32_10(U4{(uint32_t)g, (uint32_t)(g >> 32), stream, 0u}, k);
    w[4 * h] = a.x; w[4 * h + 1] = a.y; w[4 * h + 2] = a.z; w[4 * h + 3] = a.w;
  }
}

// Scale one 32-run whose max-abs is M, in place (and round it stochastically
// when asked; nearest rounding happens in the conversion). Returns e, or for
// NVFP4 (whose two 16-blocks take their own maxima and E4M3 scales) the two
// scale codes, first block in the low byte. kAnyFormat = false compiles the
// E2M1 / E8M0 case only; kNvfp4 = false leaves NVFP4 out. The draws come as
// words (D = uint32_t, two 16-bit draws each) or as draw_floats pairs.
template <bool kAnyFormat = true, bool kNvfp4 = kAnyFormat, typename D = uint32_t>
__device__ __forceinline__ int scale_run32(float2 (&R)[16], const OrientArgs& o, float M,
                                           const D (&w)[16]) {
  if (kNvfp4 && o.nv) {
    const NvScale a = nv_scale(absmax16(&R[0]), o.roundup, o.nv_p2k, o.nv_zmul);
    const NvScale b = nv_scale(absmax16(&R[8]), o.roundup, o.nv_p2k, o.nv_zmul);
    const float2 ra = make_float2(a.rcp, a.rcp), rb = make_float2(b.rcp, b.rcp);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      R[k] = f2mul(R[k], ra);
      R[8 + k] = f2mul(R[8 + k], rb);
    }
    if (o.sr) {
#pragma unroll
      for (int k = 0; k < 16; ++k) R[k] = sr_pair(R[k], w[k]);
    }
    return (int)(a.code | (b.code << 8));
  }
  const int e = scale_exponent(M, o.roundup, kAnyFormat && o.e4m3, kAnyFormat && o.e5m2);
  const float2 is = make_float2(inv_scale(e), inv_scale(e));
#pragma unroll
  for (int k = 0; k < 16; ++k) R[k] = f2mul(R[k], is);
  if (o.sr) {
#pragma unroll
    for (int k = 0; k < 16; ++k) R[k] = sr_pair(R[k], w[k]);
  }
  return e;
}

// Encode a scaled 32-run of output row `orow`, K positions k0 .. k0 + 31, and
// store it: E2M1 two per byte ([rows, K/2]) or E4M3 / E5M2 one per byte ([rows, K]).
template <bool kAnyFormat = true>
__device__ __forceinline__ void store_run32(const OrientArgs& o, int64_t orow, int64_t k0,
                                            int64_t K, const float2 (&R)[16]) {
  // orow and K are below 2^31 for every caller: one widening multiply.
  if (kAnyFormat && o.e4m3) {
    uint4* d = reinterpret_cast<uint4*>(o.q + (uint64_t)(uint32_t)orow * (uint32_t)K + k0);
    put(d, encode16_fp8(&R[0], o.e5m2), o.q, o.q_bytes);
    put(d + 1, encode16_fp8(&R[8], o.e5m2), o.q, o.q_bytes);
  } else {
    put(reinterpret_cast<uint4*>(o.q + (uint64_t)(uint32_t)orow * (uint32_t)(K >> 1) + (k0 >> 1)),
        encode32(R), o.q, o.q_bytes);
  }
}

// Row-wise quantization of 32 consecutive values of output row `row` (columns
// c0 .. c0 + 31 of a [rows, cols] tensor) held by one lane as 16 pairs, as the
// quantizer treats a 32-run: rotate (optional), block max (over the warp's 32
// rows, one per lane, for 32x32 blocks), scale, round, pack, store.
__device__ __forceinline__ void quantize_run32(float2 (&R)[16], int64_t row, int64_t c0, int64_t cols,
                                               const OrientArgs& o) {
  if (o.wht) hadamard32_lane(R, o.sign_mask, o.sgn);
  float M = absmax32(R);
  if (o.block) M = warp_max(M);
  uint32_t w[16];
  if (o.sr) draws32(o.keys, o.stream, (uint64_t)(row * cols + c0), w);
  const int e = scale_run32<true, false>(R, o, M, w);   // no NVFP4 output here
  store_run32(o, row, c0, cols, R);
  store_run_scales<false>(o, row, c0, cols, e);
}

}  // namespace mx
