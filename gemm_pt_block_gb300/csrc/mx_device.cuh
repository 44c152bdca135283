// mx_device.cuh -- per-element MXFP4 arithmetic shared by the quantizer,
// rotation and dequantization kernels (sm_103a).
//
// Every floating-point step uses explicit round-to-nearest intrinsics
// (__fadd_rn / __fsub_rn / __fmul_rn), which the compiler never contracts into
// FMAs, and the library is built without flush-to-zero, so results are the
// IEEE fp32 results the method's definition fixes.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace mx {

// fp32 nearest value of 1/sqrt(32), the rotation's normalisation.
constexpr uint32_t kWhtNormBits = 0x3E3504F3u;

// ---------------------------------------------------------------- Philox ---
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC'11), written from the published round function: words 0 and
// 2 are multiplied by the round multipliers, the high halves are mixed with
// words 1 and 3 and the key, and the key advances by the Weyl increments
// between rounds.
struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox4x32_10(U4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = U4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
  }
  return c;
}

// The 128 random bits that serve source elements 8g .. 8g+7: element 8g + j
// takes 16-bit half (j & 1) of word (j >> 1).
__device__ __forceinline__ U4 sr_group_bits(uint64_t seed, uint32_t stream, uint64_t g) {
  return philox4x32_10(U4{(uint32_t)g, (uint32_t)(g >> 32), stream, 0u}, (uint32_t)seed,
                       (uint32_t)(seed >> 32));
}

__device__ __forceinline__ uint32_t u4_word(const U4& u, int w) {
  return w == 0 ? u.x : w == 1 ? u.y : w == 2 ? u.z : u.w;
}

// ------------------------------------------------------------- rotation ---
// In-register part of the 32-point butterfly for the 16 elements a thread
// holds (block positions half*16 .. half*16+15): stages h = 1, 2, 4, 8, each
// pair (a, b) = (y[i], y[i+h]) becoming (a + b, a - b).
__device__ __forceinline__ void butterfly16(float (&y)[16]) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      const float a = y[i], b = y[i + h];
      y[i] = __fadd_rn(a, b);
      y[i + h] = __fsub_rn(a, b);
    }
  }
}

// Last stage (h = 16) across the lane pair (lane, lane ^ 1) that holds the
// two halves of one block: the lower half becomes a + b, the upper a - b,
// with a from the lower and b from the upper half.
__device__ __forceinline__ void butterfly_pair(float (&y)[16], int half) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float o = __shfl_xor_sync(0xffffffffu, y[i], 1);
    y[i] = half ? __fsub_rn(o, y[i]) : __fadd_rn(y[i], o);
  }
}

// Forward rotation c * H * diag(s) of one 32-block held by a lane pair.
__device__ __forceinline__ void wht_forward(float (&y)[16], int half, uint32_t sign_mask) {
  const uint32_t m = sign_mask >> (half * 16);
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if ((m >> i) & 1u) y[i] = -y[i];
  butterfly16(y);
  butterfly_pair(y, half);
  const float c = __uint_as_float(kWhtNormBits);
#pragma unroll
  for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(y[i], c);
}

// Inverse rotation diag(s) * c * H.
__device__ __forceinline__ void wht_inverse(float (&y)[16], int half, uint32_t sign_mask) {
  butterfly16(y);
  butterfly_pair(y, half);
  const float c = __uint_as_float(kWhtNormBits);
  const uint32_t m = sign_mask >> (half * 16);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    y[i] = __fmul_rn(y[i], c);
    if ((m >> i) & 1u) y[i] = -y[i];
  }
}

// ----------------------------------------------------------------- scale ---
// Shared exponent e for block max-abs M >= 0 from M's bit fields:
//  floor (OCP MX):  e = E - 2, E = unbiased exponent of M;
//  round-up:        e = E - 2 + (fraction(M) > 0x400000), the smallest e with
//                   6 * 2^e >= M (M / 2^(E-2) = 4 (1 + f) exceeds 6 iff f > 1/2);
//  M zero or subnormal: e = -127. Clamped to [-127, 126] (126 is the largest
//  value a finite fp32 M can give).
__device__ __forceinline__ int scale_exponent(float M, bool roundup) {
  const uint32_t b = __float_as_uint(M);
  const int bexp = (int)(b >> 23) & 0xFF;
  int e = bexp - 129 + ((roundup && (b & 0x7FFFFFu) > 0x400000u) ? 1 : 0);
  e = bexp == 0 ? -127 : e;
  return max(-127, min(126, e));
}

// 2^-e as an fp32 (normal for every e in [-127, 126]).
__device__ __forceinline__ float inv_scale(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// -------------------------------------------------------------- rounding ---
// Nearest E2M1 code, ties to the even code, saturating at 6; sign from v.
// Thresholds are the grid midpoints 0.25 0.75 1.25 1.75 2.5 3.5 5; a midpoint
// whose lower neighbour has an even code rounds down (strict >), else up (>=).
__device__ __forceinline__ uint32_t round_rtn(float v) {
  const float a = fabsf(v);
  uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
               (a >= 3.5f) + (a > 5.0f);
  return m | ((__float_as_uint(v) >> 28) & 8u);
}

// Stochastic rounding with a 16-bit draw r: a = min(|v|, 6) in [lo, hi) goes to
// hi iff r < 2^16 * (a - lo) / (hi - lo). Every step is exact in fp32: a - lo
// is exact (lo <= a < 2 lo or lo = 0) and the step is a power of two.
__device__ __forceinline__ uint32_t round_sr(float v, uint32_t r16) {
  const float a = fminf(fabsf(v), 6.0f);
  float lo, inv_step;
  uint32_t c0;
  if (a < 2.0f) {
    const float t = floorf(__fmul_rn(a, 2.0f));
    c0 = (uint32_t)t;
    lo = __fmul_rn(t, 0.5f);
    inv_step = 2.0f;
  } else if (a < 4.0f) {
    const float t = floorf(a);
    c0 = (uint32_t)t + 2u;
    lo = t;
    inv_step = 1.0f;
  } else if (a < 6.0f) {
    c0 = 6u;
    lo = 4.0f;
    inv_step = 0.5f;
  } else {
    c0 = 7u;
    lo = 6.0f;
    inv_step = 0.0f;
  }
  const float p = __fmul_rn(__fsub_rn(a, lo), inv_step);
  const uint32_t up = ((float)r16 < __fmul_rn(p, 65536.0f)) ? 1u : 0u;
  return (c0 + up) | ((__float_as_uint(v) >> 28) & 8u);
}

// ------------------------------------------------------------ layouts ---
// Byte offset of scale (r, kb) in the block-scaled tensor-core layout for a
// scale matrix with nkb scale columns (128 x 4 tiles of 512 bytes).
__device__ __forceinline__ int64_t mma_scale_offset(int64_t r, int64_t kb, int64_t nkb) {
  return (((r >> 7) * (nkb >> 2) + (kb >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) +
         (kb & 3);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// E2M1 magnitude code 0..7 -> value.
__device__ __forceinline__ float e2m1_magnitude(uint32_t m) {
  const float v = __uint_as_float((((m >> 1) + 126u) << 23) | ((m & 1u) << 22));
  return m >= 2u ? v : (m == 1u ? 0.5f : 0.0f);
}

}  // namespace mx
