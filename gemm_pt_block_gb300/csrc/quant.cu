// quant.cu -- the fused MXFP4 quantizer, the stand-alone 32-point rotation and
// dequantization (sm_103a). All three are HBM-bound streaming kernels: 128-bit
// coalesced loads, the rotation's butterflies in registers with one warp
// shuffle stage, Philox4x32-10 draws for stochastic rounding computed once per
// 8 consecutive source elements, packed 64-bit code stores.
//
// Method: "Block-Scaled MXFP4 With Stochastic Hadamard Rounding Matches BF16
// Convergence on 70B Pre-Training" (paras. 1-2: E8M0 scale per 32 E2M1
// elements; block Hadamard rotation fused with stochastic rounding before
// packing); "Stable FP4 Training via Transposition-Invariant Block
// Quantization" ("The fix, and its supporting cast": 2D 32x32 blocks,
// truncation-free scaling, stochastic rounding; "The aha: transposition
// scrambles the blocks": both orientations of one tensor).
#include <cstdint>

#include "internal.h"
#include "mx_device.cuh"

namespace mx {
namespace {

constexpr int kThreads = 256;

// ------------------------------------------------------------ loading ---
// 16 consecutive elements starting at p (16-byte aligned) widened to fp32.
__device__ __forceinline__ void load16(const uint16_t* p, float (&v)[16]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void load16(const float* p, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p) + i);
    v[4 * i] = a.x;
    v[4 * i + 1] = a.y;
    v[4 * i + 2] = a.z;
    v[4 * i + 3] = a.w;
  }
}

// ------------------------------------------------------- quantize core ---
// Max-abs of a lane pair's 32-block.
__device__ __forceinline__ float pair_max(const float (&y)[16]) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(y[i]));
  return fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
}

// Codes of 16 scaled elements, packed little-nibble-first into two words.
// bits[j] holds element j's 16-bit draw when stochastic rounding is on.
__device__ __forceinline__ uint2 encode16(const float (&y)[16], float is, bool sr,
                                          const uint32_t (&bits)[16]) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float v = __fmul_rn(y[j], is);
    const uint32_t code = sr ? round_sr(v, bits[j]) : round_rtn(v);
    if (j < 8)
      lo |= code << (4 * j);
    else
      hi |= code << (4 * (j - 8));
  }
  return make_uint2(lo, hi);
}

// Draws for source elements i0 .. i0+15 (i0 % 16 == 0): two Philox calls.
__device__ __forceinline__ void draws16(uint64_t seed, uint32_t stream, uint64_t i0,
                                        uint32_t (&bits)[16]) {
  const U4 a = sr_group_bits(seed, stream, i0 >> 3);
  const U4 b = sr_group_bits(seed, stream, (i0 >> 3) + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    bits[2 * j] = w[j] & 0xFFFFu;
    bits[2 * j + 1] = w[j] >> 16;
  }
}

__device__ __forceinline__ void store_scale(const OrientArgs& o, int64_t orow, int64_t kb,
                                            int64_t nkb, int e) {
  const int64_t off = o.mma_layout ? mma_scale_offset(orow, kb, nkb) : orow * nkb + kb;
  o.s[off] = (uint8_t)(e + 127);
}

// ------------------------------------------------- row-wise, 1x32 blocks ---
// One thread per 16 consecutive elements of a row; lanes (2k, 2k+1) hold one
// 32-element block. Grid covers rows * cols / 16 threads.
template <typename InT>
__global__ void __launch_bounds__(kThreads)
quant_rows_1x32_kernel(const InT* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                       OrientArgs o) {
  const int64_t halves = cols >> 4;
  const int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const bool valid = t < rows * halves;
  const int64_t r = valid ? t / halves : 0;
  const int64_t c0 = valid ? (t - r * halves) << 4 : 0;
  const int half = threadIdx.x & 1;

  float y[16];
  if (valid) {
    load16(x + r * ld + c0, y);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = 0.0f;
  }
  if (o.wht) wht_forward(y, half, o.sign_mask);
  const float M = pair_max(y);
  const int e = scale_exponent(M, o.roundup);
  uint32_t bits[16];
  if (o.sr) draws16(o.seed, o.stream, (uint64_t)(r * cols + c0), bits);
  const uint2 packed = encode16(y, inv_scale(e), o.sr, bits);
  if (valid) {
    *reinterpret_cast<uint2*>(o.q + r * (cols >> 1) + (c0 >> 1)) = packed;
    if (!half) store_scale(o, r, c0 >> 5, cols >> 5, e);
  }
}

// --------------------------------------- 64 x 64 tiles: both orientations ---
// Used when the column-wise output is requested or a 32x32 block is in play.
// Phase 1 (row-major ownership, thread t: tile row t/4, columns (t%4)*16..+16)
// loads the tile, quantizes the row-wise output, and stages fp32 values (and
// the column orientation's random draws, keyed by source index) in shared
// memory. Phase 2 (column ownership, thread t: tile column (t/2)%64, rows
// (t/128)*32 + (t%2)*16 .. +16) quantizes x^T from shared memory.
template <typename InT>
__global__ void __launch_bounds__(kThreads)
quant_tile_kernel(const InT* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                  OrientArgs orow, OrientArgs ocol, int do_row, int do_col) {
  __shared__ float tile[64][65];
  __shared__ uint16_t tbits[64][66];
  __shared__ float red_r[2][2][4];
  __shared__ float red_c[2][2][2];

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, half = t & 1;
  const int64_t R0 = (int64_t)blockIdx.y * 64, C0 = (int64_t)blockIdx.x * 64;

  // ---- phase 1 ----
  {
    const int lr = t >> 2, lc = (t & 3) * 16;
    const int64_t r = R0 + lr, c = C0 + lc;
    const bool valid = r < rows && c < cols;
    float v[16];
    if (valid) {
      load16(x + r * ld + c, v);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.0f;
    }
    if (do_col) {
#pragma unroll
      for (int i = 0; i < 16; ++i) tile[lr][lc + i] = v[i];
      if (ocol.sr) {
        uint32_t bits[16];
        draws16(ocol.seed, ocol.stream, valid ? (uint64_t)(r * cols + c) : 0ull, bits);
#pragma unroll
        for (int i = 0; i < 16; ++i) tbits[lr][lc + i] = (uint16_t)bits[i];
      }
    }
    if (do_row) {
      if (orow.wht) wht_forward(v, half, orow.sign_mask);
      float M = pair_max(v);
      if (orow.block) {
        // 32x32: max over the 8 rows of this warp (lane bits 2..4), then over
        // the 4 warps of the 32-row group.
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 4));
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 8));
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
        if (lane == 0 || lane == 2) red_r[warp >> 2][lane >> 1][warp & 3] = M;
        __syncthreads();
        const float* rr = red_r[warp >> 2][(t & 3) >> 1];
        M = fmaxf(fmaxf(rr[0], rr[1]), fmaxf(rr[2], rr[3]));
      }
      const int e = scale_exponent(M, orow.roundup);
      uint32_t bits[16];
      if (orow.sr) draws16(orow.seed, orow.stream, (uint64_t)(r * cols + c), bits);
      const uint2 packed = encode16(v, inv_scale(e), orow.sr, bits);
      if (valid) {
        *reinterpret_cast<uint2*>(orow.q + r * (cols >> 1) + (c >> 1)) = packed;
        if (!half) store_scale(orow, r, c >> 5, cols >> 5, e);
      }
    }
  }
  if (!do_col) return;
  __syncthreads();

  // ---- phase 2: the column orientation (quantization along rows) ----
  {
    const int cc = (t >> 1) & 63, rb = t >> 7;
    const int lr0 = rb * 32 + half * 16;
    const int64_t oc = C0 + cc, k0 = R0 + lr0;
    const bool valid = oc < cols && k0 < rows;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = tile[lr0 + i][cc];
    if (ocol.wht) wht_forward(v, half, ocol.sign_mask);
    float M = pair_max(v);
    if (ocol.block) {
      // 32x32: max over the 16 columns of this warp (lane bits 1..4), then
      // over the 2 warps holding the block's 32 columns.
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 4));
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 8));
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
      if (lane == 0) red_c[rb][(warp & 3) >> 1][warp & 1] = M;
      __syncthreads();
      const float* rc = red_c[rb][(warp & 3) >> 1];
      M = fmaxf(rc[0], rc[1]);
    }
    const int e = scale_exponent(M, ocol.roundup);
    uint32_t bits[16];
    if (ocol.sr) {
#pragma unroll
      for (int i = 0; i < 16; ++i) bits[i] = tbits[lr0 + i][cc];
    }
    const uint2 packed = encode16(v, inv_scale(e), ocol.sr, bits);
    if (valid) {
      *reinterpret_cast<uint2*>(ocol.q + oc * (rows >> 1) + (k0 >> 1)) = packed;
      if (!half) store_scale(ocol, oc, k0 >> 5, rows >> 5, e);
    }
  }
}

// ------------------------------------------------------------ rotation ---
template <typename InT>
__global__ void __launch_bounds__(kThreads)
hadamard32_kernel(const InT* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                  uint32_t sign_mask, int inverse, float* __restrict__ y) {
  const int64_t halves = cols >> 4;
  const int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const bool valid = t < rows * halves;
  const int64_t r = valid ? t / halves : 0;
  const int64_t c0 = valid ? (t - r * halves) << 4 : 0;
  const int half = threadIdx.x & 1;
  float v[16];
  if (valid) {
    load16(x + r * ld + c0, v);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
  }
  if (inverse)
    wht_inverse(v, half, sign_mask);
  else
    wht_forward(v, half, sign_mask);
  if (valid) {
    float4* out = reinterpret_cast<float4*>(y + r * cols + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

// ---------------------------------------------------------- dequantize ---
__global__ void __launch_bounds__(kThreads)
dequant_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int mma_layout,
               int64_t rows, int64_t cols, float* __restrict__ out) {
  const int64_t halves = cols >> 4;
  const int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (t >= rows * halves) return;
  const int64_t r = t / halves, c0 = (t - r * halves) << 4;
  const int64_t nkb = cols >> 5;
  const uint2 w = __ldg(reinterpret_cast<const uint2*>(q + r * (cols >> 1) + (c0 >> 1)));
  const int64_t so = mma_layout ? mma_scale_offset(r, c0 >> 5, nkb) : r * nkb + (c0 >> 5);
  const uint32_t sb = __ldg(s + so);
  const float scale = sb == 255u ? __uint_as_float(0x7FC00000u)
                      : sb == 0u ? __uint_as_float(0x00400000u)   // 2^-127 (subnormal)
                                 : __uint_as_float(sb << 23);
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t code = ((j < 8 ? w.x : w.y) >> (4 * (j & 7))) & 0xFu;
    const float m = e2m1_magnitude(code & 7u);
    v[j] = __fmul_rn((code & 8u) ? -m : m, scale);
  }
  float4* o = reinterpret_cast<float4*>(out + r * cols + c0);
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

inline unsigned blocks_for(int64_t threads) { return (unsigned)((threads + kThreads - 1) / kThreads); }

template <typename InT>
cudaError_t quantize_impl(const InT* x, int64_t rows, int64_t cols, int64_t ld,
                          const OrientArgs* row, const OrientArgs* col, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const bool tile = col != nullptr || (row && row->block);
  if (!tile) {
    quant_rows_1x32_kernel<InT><<<blocks_for(rows * (cols >> 4)), kThreads, 0, st>>>(
        x, rows, cols, ld, *row);
  } else {
    OrientArgs dummy{};
    dim3 grid((unsigned)((cols + 63) / 64), (unsigned)((rows + 63) / 64));
    quant_tile_kernel<InT><<<grid, kThreads, 0, st>>>(x, rows, cols, ld, row ? *row : dummy,
                                                      col ? *col : dummy, row != nullptr,
                                                      col != nullptr);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const void* x, bool f32_in, int64_t rows, int64_t cols, int64_t ld,
                            const OrientArgs* row, const OrientArgs* col, cudaStream_t st) {
  return f32_in ? quantize_impl(static_cast<const float*>(x), rows, cols, ld, row, col, st)
                : quantize_impl(static_cast<const uint16_t*>(x), rows, cols, ld, row, col, st);
}

cudaError_t launch_hadamard32(const void* x, bool f32_in, int64_t rows, int64_t cols, int64_t ld,
                              uint32_t sign_mask, bool inverse, float* y, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const unsigned nb = blocks_for(rows * (cols >> 4));
  if (f32_in)
    hadamard32_kernel<float><<<nb, kThreads, 0, st>>>(static_cast<const float*>(x), rows, cols,
                                                      ld, sign_mask, inverse, y);
  else
    hadamard32_kernel<uint16_t><<<nb, kThreads, 0, st>>>(static_cast<const uint16_t*>(x), rows,
                                                         cols, ld, sign_mask, inverse, y);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* q, const uint8_t* s, bool mma_layout, int64_t rows,
                              int64_t cols, float* out, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  dequant_kernel<<<blocks_for(rows * (cols >> 4)), kThreads, 0, st>>>(q, s, mma_layout, rows,
                                                                      cols, out);
  return cudaGetLastError();
}

}  // namespace mx
