// mx_device.cuh -- per-element MXFP4 arithmetic shared by the quantizer,
// rotation and dequantization kernels (sm_103a).
//
// Every floating-point step is an explicitly rounded IEEE operation: scalar
// __fadd_rn / __fmul_rn, or the packed two-lane forms add/sub/mul/fma.f32x2,
// which round each lane exactly like the scalar instruction. Nothing is
// contracted into an FMA by the compiler (the one explicit FMA, in stochastic
// rounding, yields an exactly representable value) and the library is built
// without flush-to-zero, so results are the fp32 results the method's
// definition fixes.
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
// words 1 and 3 and the round key. The ten round keys (the key advanced by the
// Weyl increments) are computed once on the host and passed in.
struct U4 {
  uint32_t x, y, z, w;
};

struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};

// Both 32-bit halves of the 64-bit product a * b in one instruction.
__device__ __forceinline__ void mul_wide(uint32_t a, uint32_t b, uint32_t& lo, uint32_t& hi) {
  asm("{.reg .u64 t;\n\tmul.wide.u32 t, %2, %3;\n\tmov.b64 {%0, %1}, t;}"
      : "=r"(lo), "=r"(hi) : "r"(a), "r"(b));
}

__device__ __forceinline__ U4 philox4x32_10(U4 c, const PhiloxKeys& k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint32_t lo0, hi0, lo1, hi1;
    mul_wide(0xD2511F53u, c.x, lo0, hi0);
    mul_wide(0xCD9E8D57u, c.z, lo1, hi1);
    c = U4{hi1 ^ c.y ^ k.k0[r], lo1, hi0 ^ c.w ^ k.k1[r], lo0};
  }
  return c;
}

// Random words for source elements 16 h .. 16 h + 15 (two Philox calls, one
// per 8 elements). Word j of the result holds the draws of elements 2j (low
// 16 bits) and 2j + 1 (high 16 bits).
__device__ __forceinline__ void draws16(const PhiloxKeys& k, uint32_t stream, uint64_t i0,
                                        uint32_t (&w)[8]) {
  const uint64_t g = i0 >> 3;
  const U4 a = philox4x32_10(U4{(uint32_t)g, (uint32_t)(g >> 32), stream, 0u}, k);
  const U4 b = philox4x32_10(U4{(uint32_t)(g + 1), (uint32_t)((g + 1) >> 32), stream, 0u}, k);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// The same for elements 8 g0 .. 8 g0 + 15 when g0 fits in 32 bits.
__device__ __forceinline__ void draws16_g(const PhiloxKeys& k, uint32_t stream, uint32_t g0,
                                          uint32_t (&w)[8]) {
  const U4 a = philox4x32_10(U4{g0, 0u, stream, 0u}, k);
  const U4 b = philox4x32_10(U4{g0 + 1u, 0u, stream, 0u}, k);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// ------------------------------------------------------- packed fp32 ops ---
__device__ __forceinline__ float2 f2add(float2 a, float2 b) {
  float2 r;
  asm("{.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ float2 f2sub(float2 a, float2 b) {
  float2 r;
  asm("{.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ float2 f2mul(float2 a, float2 b) {
  float2 r;
  asm("{.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// a + b rounded toward +infinity, per lane.
__device__ __forceinline__ float2 f2add_rp(float2 a, float2 b) {
  float2 r;
  asm("{.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rp.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// a * b + c with one rounding (to nearest), per lane.
__device__ __forceinline__ float2 f2fma(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mov.b64 c, {%6, %7};\n\tfma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ------------------------------------------------------------- rotation ---
// A lane pair holds one 32-element block, 16 elements per lane as 8 pairs
// R[k] = (y[2k], y[2k+1]) of the lane's local index. Local butterfly stages
// pair local indices (i, i + h), h = 1, 2, 4, 8: h = 1 is within a pair
// (scalar), the others combine whole pairs (packed f32x2).
__device__ __forceinline__ void local_stage(float2 (&R)[8], int h) {
  if (h == 1) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float a = R[k].x, b = R[k].y;
      R[k] = make_float2(__fadd_rn(a, b), __fsub_rn(a, b));
    }
  } else {
    const int hp = h >> 1;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k & hp) continue;
      const float2 a = R[k], b = R[k + hp];
      R[k] = f2add(a, b);
      R[k + hp] = f2sub(a, b);
    }
  }
}

// The stage across the lane pair (lane, lane ^ 1): the lower lane's element
// (a) and the upper lane's element (b) with the same local index become
// a + b (lower) and a - b (upper).
__device__ __forceinline__ void cross_stage(float2 (&R)[8], int upper) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float2 o;
    o.x = __shfl_xor_sync(0xffffffffu, R[k].x, 1);
    o.y = __shfl_xor_sync(0xffffffffu, R[k].y, 1);
    R[k] = upper ? f2sub(o, R[k]) : f2add(R[k], o);
  }
}

__device__ __forceinline__ void scale_all(float2 (&R)[8], float s) {
  const float2 s2 = make_float2(s, s);
#pragma unroll
  for (int k = 0; k < 8; ++k) R[k] = f2mul(R[k], s2);
}

// Butterflies of c * H in the order h = 1, 2, 4, 8, 16 of the block index, for
// a lane holding block elements 16 * upper + local (contiguous halves): the
// four local stages come first, then the cross-lane stage (h = 16).
__device__ __forceinline__ void hadamard_halves(float2 (&R)[8], int upper) {
  local_stage(R, 1);
  local_stage(R, 2);
  local_stage(R, 4);
  local_stage(R, 8);
  cross_stage(R, upper);
  scale_all(R, __uint_as_float(kWhtNormBits));
}

// The same transform for a lane holding block elements 2 * local + upper
// (interleaved): block stage h = 1 is the cross-lane one, block stages
// 2, 4, 8, 16 are local stages 1, 2, 4, 8.
__device__ __forceinline__ void hadamard_interleaved(float2 (&R)[8], int upper) {
  cross_stage(R, upper);
  local_stage(R, 1);
  local_stage(R, 2);
  local_stage(R, 4);
  local_stage(R, 8);
  scale_all(R, __uint_as_float(kWhtNormBits));
}

// Multiply element i by -1 where bit i of m is set (exact sign flips).
__device__ __forceinline__ void apply_signs(float2 (&R)[8], uint32_t m) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    R[k].x = __uint_as_float(__float_as_uint(R[k].x) ^ ((m >> (2 * k)) << 31));
    R[k].y = __uint_as_float(__float_as_uint(R[k].y) ^ ((m >> (2 * k + 1)) << 31));
  }
}

// ------------------------------------------------ whole block in-thread ---
// A lane holding all 32 elements of a block as 16 pairs R[k] = (y[2k], y[2k+1]).
// Butterfly stage h pairs elements (i, i + h): h = 1 within a pair (scalar),
// h = 2, 4, 8, 16 between pairs k and k + h/2 (packed f32x2).
__device__ __forceinline__ void stage32(float2 (&R)[16], int h) {
  if (h == 1) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float a = R[k].x, b = R[k].y;
      R[k] = make_float2(__fadd_rn(a, b), __fsub_rn(a, b));
    }
  } else {
    const int hp = h >> 1;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if (k & hp) continue;
      const float2 a = R[k], b = R[k + hp];
      R[k] = f2add(a, b);
      R[k + hp] = f2sub(a, b);
    }
  }
}

// y = c * H * diag(s) * x for one block held by one lane, butterflies in the
// order h = 1, 2, 4, 8, 16, c applied last. The signs come as the factors
// sgn[i] = s_i = +-1 (kernel parameters, built on the host from the mask), so
// that no per-element bit extraction is needed; sign_mask != 0 says some are -1.
__device__ __forceinline__ void hadamard32_lane(float2 (&R)[16], uint32_t sign_mask,
                                                const float (&sgn)[32]) {
  if (sign_mask) {
    // Stage h = 1 with the signs folded in: (s0 x0 + s1 x1, s0 x0 - s1 x1),
    // each an exact product and one rounded sum (s = +-1).
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float t = __fmul_rn(R[k].y, sgn[2 * k + 1]);
      R[k] = make_float2(__fmaf_rn(R[k].x, sgn[2 * k], t), __fmaf_rn(R[k].x, sgn[2 * k], -t));
    }
  } else {
    stage32(R, 1);
  }
  stage32(R, 2);
  stage32(R, 4);
  stage32(R, 8);
  stage32(R, 16);
  const float2 c = make_float2(__uint_as_float(kWhtNormBits), __uint_as_float(kWhtNormBits));
#pragma unroll
  for (int k = 0; k < 16; ++k) R[k] = f2mul(R[k], c);
}

__device__ __forceinline__ float absmax32(const float2 (&R)[16]) {
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) m = max3(m, fabsf(R[k].x), fabsf(R[k].y));
  return m;
}

// Maximum over the warp in one instruction (exact, like the shuffle tree it
// replaces; the quantizer's maxima are finite and >= 0).
__device__ __forceinline__ float warp_max(float m) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(m));
  return r;
}

// ----------------------------------------------------------------- scale ---
// Shared exponent e for block max-abs M >= 0 from M's bit fields:
//  floor (OCP MX):  e = E - 2, E = unbiased exponent of M;
//  round-up:        e = E - 2 + (fraction(M) > 0x400000), the smallest e with
//                   6 * 2^e >= M (M / 2^(E-2) = 4 (1 + f) exceeds 6 iff f > 1/2);
//  M zero or subnormal: e = -127. Clamped to [-127, 126] (126 is the largest
//  value a finite fp32 M can give).
// For MXFP8 (E4M3 elements, largest 448 = 1.75 * 2^8) the same with 8 in place
// of 2 and the round-up threshold f > 3/4 (fraction > 0x600000); E5M2
// elements (largest 57344 = 1.75 * 2^15) with 15 in place of 2.
__device__ __forceinline__ int scale_exponent(float M, bool roundup, bool fp8 = false,
                                              bool e5m2 = false) {
  const uint32_t b = __float_as_uint(M);
  const int bexp = (int)(b >> 23) & 0xFF;
  // E2M1: emax 2, 6 = 1.5 * 2^2; E4M3: emax 8; E5M2: emax 15 (both 1.75 * 2^emax).
  const uint32_t over = fp8 ? 0x600000u : 0x400000u;
  int e = bexp - (fp8 ? (e5m2 ? 142 : 135) : 129) + ((roundup && (b & 0x7FFFFFu) > over) ? 1 : 0);
  e = bexp == 0 ? -127 : e;
  return max(-127, min(126, e));
}

// 2^-e as an fp32 (normal for every e in [-127, 126]).
__device__ __forceinline__ float inv_scale(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

__device__ __forceinline__ float pair_absmax(const float2 (&R)[8]) {
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) m = max3(m, fabsf(R[k].x), fabsf(R[k].y));
  return fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
}

// -------------------------------------------------------------- rounding ---
// Round-to-nearest, ties to the even code, saturating at 6, sign kept: the
// IEEE conversion to E2M1 (cvt.rn.satfinite), two values per instruction.
// Returns 8 codes packed little-nibble-first (element 0 in bits 0-3).
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                           float v5, float v6, float v7) {
  uint32_t r;
  asm("{.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return r;
}

// MXFP8 elements: OCP FP8 E4M3, nearest-even with saturation at 448 (the IEEE
// conversion cvt.rn.satfinite), sign kept; 4 values -> 4 bytes, element 0 in
// the lowest byte.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
  uint32_t r;
  asm("{.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
  return r;
}

// OCP FP8 E5M2 elements: nearest-even with saturation at 57344 (the IEEE
// conversion cvt.rn.satfinite), sign kept; 4 values -> 4 bytes.
__device__ __forceinline__ uint32_t e5m2x4(float v0, float v1, float v2, float v3) {
  uint32_t r;
  asm("{.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
  return r;
}

// 8 pairs -> 16 E4M3 bytes, or E5M2 bytes when e5m2.
__device__ __forceinline__ uint4 encode16_fp8(const float2* V, bool e5m2) {
  if (e5m2)
    return make_uint4(e5m2x4(V[0].x, V[0].y, V[1].x, V[1].y), e5m2x4(V[2].x, V[2].y, V[3].x, V[3].y),
                      e5m2x4(V[4].x, V[4].y, V[5].x, V[5].y), e5m2x4(V[6].x, V[6].y, V[7].x, V[7].y));
  return make_uint4(e4m3x4(V[0].x, V[0].y, V[1].x, V[1].y), e4m3x4(V[2].x, V[2].y, V[3].x, V[3].y),
                    e4m3x4(V[4].x, V[4].y, V[5].x, V[5].y), e4m3x4(V[6].x, V[6].y, V[7].x, V[7].y));
}

// ------------------------------------------------------ NVFP4 scales ---
// Non-negative E4M3 code c (0 .. 126) -> value, exact: (8 + m) 2^(E - 10) for
// exponent field E > 0, m 2^-9 for E = 0.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t E = c >> 3, m = c & 7u;
  return E ? __uint_as_float(((E + 120u) << 23) | (m << 20)) : __fmul_rn((float)m, 0.001953125f);
}

struct NvScale {
  uint32_t code;  // E4M3 code of S
  float rcp;      // fp32 nearest 1 / (S 2^k), 0 when S = 0
};

// Scale of one 1x16 block with max-abs M under the per-tensor factor 2^k
// (p2k = 2^k; zmul = 2^-k / 6 rounded to fp32). A first guess, the nearest
// E4M3 value to M * zmul (hardware conversion), is within one code of the
// answer; it is then fixed by exact comparisons of M with thresholds that are
// exact in fp32: 6 S 2^k (round-up: the smallest S with 6 S 2^k >= M) or the
// midpoints 3 (S_c + S_c+1) 2^k (nearest, ties to the even code; M >= 2688
// 2^k saturates at 448).
__device__ __forceinline__ NvScale nv_scale(float M, bool roundup, float p2k, float zmul) {
  const float z = __fmul_rn(M, zmul);
  uint32_t c;
  asm("{.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %1;\n\tcvt.u32.u16 %0, t;}"
      : "=r"(c) : "f"(z));
  c &= 0x7Fu;
  if (roundup) {
    if (c < 126u && __fmul_rn(__fmul_rn(6.0f, e4m3_value(c)), p2k) < M)
      ++c;
    else if (c > 0u && __fmul_rn(__fmul_rn(6.0f, e4m3_value(c - 1u)), p2k) >= M)
      --c;
  } else if (M >= __fmul_rn(2688.0f, p2k)) {
    c = 126u;
  } else {
    if (c < 126u) {
      const float t = __fmul_rn(__fmul_rn(3.0f, __fadd_rn(e4m3_value(c), e4m3_value(c + 1u))), p2k);
      if (M > t || (M == t && (c & 1u))) ++c;          // a tie goes to the even code c + 1
    }
    if (c > 0u) {
      const float t = __fmul_rn(__fmul_rn(3.0f, __fadd_rn(e4m3_value(c - 1u), e4m3_value(c))), p2k);
      if (M < t || (M == t && (c & 1u))) --c;          // a tie goes to the even code c - 1
    }
  }
  const float S = __fmul_rn(e4m3_value(c), p2k);
  return NvScale{c, c ? __frcp_rn(S) : 0.0f};
}

// Max-abs of the 16 values one lane holds.
__device__ __forceinline__ float absmax16(const float2* R) {
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) m = max3(m, fabsf(R[k].x), fabsf(R[k].y));
  return m;
}

__device__ __forceinline__ uint4 encode32(const float2 (&V)[16]) {
  return make_uint4(e2m1x8(V[0].x, V[0].y, V[1].x, V[1].y, V[2].x, V[2].y, V[3].x, V[3].y),
                    e2m1x8(V[4].x, V[4].y, V[5].x, V[5].y, V[6].x, V[6].y, V[7].x, V[7].y),
                    e2m1x8(V[8].x, V[8].y, V[9].x, V[9].y, V[10].x, V[10].y, V[11].x, V[11].y),
                    e2m1x8(V[12].x, V[12].y, V[13].x, V[13].y, V[14].x, V[14].y, V[15].x, V[15].y));
}

__device__ __forceinline__ uint2 encode16(const float2 (&V)[8]) {
  return make_uint2(e2m1x8(V[0].x, V[0].y, V[1].x, V[1].y, V[2].x, V[2].y, V[3].x, V[3].y),
                    e2m1x8(V[4].x, V[4].y, V[5].x, V[5].y, V[6].x, V[6].y, V[7].x, V[7].y));
}

// The draws of w as the floats 2^23 + r (element 0's r in the low half).
__device__ __forceinline__ float2 draw_floats(uint32_t w) {
  return make_float2(__uint_as_float(0x4B000000u | (w & 0xFFFFu)),
                     __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7432)));
}

// Stochastic rounding of two scaled values v whose draws r come as
// f = draw_floats(w) (the 16-bit halves of w, element 0 low). With a = |v|
// in [lo, lo + st) on the E2M1
// grid, the value goes up iff r < 2^16 (a - lo) / st, i.e. iff a - lo > th
// with th = r * st * 2^-16; equivalently the result is the smallest multiple
// of st that is >= a - th (lo is a multiple of st, and a - th > lo - st).
// Every step is exact in fp32 (nothing depends on an FMA contraction):
//   st = max(1, 2^E(a)) / 2 (E = unbiased exponent; 1/2 below 1); the grid
//     points of [lo, lo + st] are multiples of st, and values in (6, 8) that
//     reach 8 saturate to 6 in the E2M1 conversion as they round down to 6;
//   -r * 2^-17 is exact, formed as fma(2^23 + r, -2^-17, 64) from f
//     (r has 16 bits);
//   x = a - th, taken with one rounding as fma(2 st, -r * 2^-17, a) (the
//     product is exact: 2 st is a power of two), is exact for a >= 1/2 (both
//     are multiples of ulp(a) within one binade of x) and otherwise has the
//     sign and the ceiling of the exact difference;
//   the ceiling is (x + C, rounded up) - C with C = 3 * 2^22 * st, whose
//     binade (ulp st) holds x + C for every |x| < 8; it is >= +0.
// The rounding works on |v|; v's sign bit is put back on the result (a
// negative value that rounds to zero gives -0). Returns the chosen grid
// values, whose E2M1 conversion is then exact.
__device__ __forceinline__ float2 sr_pair(float2 v, float2 f) {
  const uint32_t b0 = __float_as_uint(v.x), b1 = __float_as_uint(v.y);
  const float2 a = make_float2(fabsf(v.x), fabsf(v.y));
  const float2 st2 = make_float2(fmaxf(__uint_as_float(b0 & 0x7F800000u), 1.0f),
                                 fmaxf(__uint_as_float(b1 & 0x7F800000u), 1.0f));
  const float2 C = f2mul(st2, make_float2(6291456.0f, 6291456.0f));        // 3 * 2^21
  const float2 nr = f2fma(f, make_float2(-7.62939453125e-6f, -7.62939453125e-6f), make_float2(64.0f, 64.0f));
  const float2 x = f2fma(st2, nr, a);
  const float2 q = f2sub(f2add_rp(x, C), C);
  return make_float2(__uint_as_float(__float_as_uint(q.x) | (b0 & 0x80000000u)),
                     __uint_as_float(__float_as_uint(q.y) | (b1 & 0x80000000u)));
}

// The same with the draws as the word w.
__device__ __forceinline__ float2 sr_pair(float2 v, uint32_t w) { return sr_pair(v, draw_floats(w)); }

// SR of 16 scaled values; word k of w holds the draws of pair R[k].
__device__ __forceinline__ void sr16(float2 (&V)[8], const uint32_t (&w)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) V[k] = sr_pair(V[k], w[k]);
}

// ------------------------------------------------------- fast division ---
// Unsigned 32-bit division by a run-time constant d >= 1 (Granlund and
// Montgomery, "Division by Invariant Integers using Multiplication", PLDI'94):
// l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1, n / d = (mulhi(m, n) + n) >> l.
struct FastDiv {
  uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while (l < 32 && (1ull << l) < d) ++l;
  const uint64_t m = (((1ull << 32) * ((1ull << l) - d)) / d) + 1;
  return FastDiv{d, (uint32_t)m, l};
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return (uint32_t)(((uint64_t)__umulhi(f.m, n) + n) >> f.l);
}

// ------------------------------------------------------------ layouts ---
// Byte offset of scale (r, kb) in the block-scaled tensor-core layout for a
// scale matrix with nkb scale columns (128 x 4 tiles of 512 bytes).
__device__ __forceinline__ int64_t mma_scale_offset(int64_t r, int64_t kb, int64_t nkb) {
  return (((r >> 7) * (nkb >> 2) + (kb >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) +
         (kb & 3);
}

// E2M1 magnitude code 0..7 -> value.
__device__ __forceinline__ float e2m1_magnitude(uint32_t m) {
  const float v = __uint_as_float((((m >> 1) + 126u) << 23) | ((m & 1u) << 22));
  return m >= 2u ? v : (m == 1u ? 0.5f : 0.0f);
}

}  // namespace mx
