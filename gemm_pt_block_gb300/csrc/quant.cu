// quant.cu -- the fused MXFP4 quantizer, the stand-alone 32-point rotation and
// dequantization (sm_103a). All are streaming kernels bound by HBM traffic
// once the per-element instruction count is low: 128-bit coalesced loads,
// the rotation's butterflies in registers (packed f32x2) with one warp-shuffle
// stage, Philox4x32-10 draws for stochastic rounding once per 8 consecutive
// source elements with host-precomputed round keys, and the hardware E2M1
// conversion for nearest-even rounding and for encoding.
//
// Method: "Block-Scaled MXFP4 With Stochastic Hadamard Rounding Matches BF16
// Convergence on 70B Pre-Training" (paras. 1-2: E8M0 scale per 32 E2M1
// elements; block Hadamard rotation fused with stochastic rounding before
// packing); "Stable FP4 Training via Transposition-Invariant Block
// Quantization" ("The fix, and its supporting cast": 2D 32x32 blocks,
// truncation-free scaling, stochastic rounding; "The aha: transposition
// scrambles the blocks": both orientations of one tensor).
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "mx_device.cuh"

namespace mx {
namespace {
__device__ uint32_t g_quant_error;
}  // namespace
}  // namespace mx
#define MX_BOUNDS_FAIL() atomicExch(&::mx::g_quant_error, ::mx::kErrBounds)

#include "quant_device.cuh"
#include "ptx.cuh"
#include "tma_host.h"

namespace mx {

void prepare_orient(OrientArgs* o) {
  uint32_t k0 = (uint32_t)o->seed, k1 = (uint32_t)(o->seed >> 32);
  for (int r = 0; r < 10; ++r) {
    o->keys.k0[r] = k0;
    o->keys.k1[r] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  const uint32_t m = o->wht ? o->sign_mask : 0u;
  for (int i = 0; i < 32; ++i) o->sgn[i] = ((m >> i) & 1u) ? -1.0f : 1.0f;
  for (int u = 0; u < 2; ++u) {
    o->sm_half[u] = (m >> (16 * u)) & 0xFFFFu;
    // Column-orientation lanes hold block elements 4 (j / 2) + 2 u + (j % 2).
    uint32_t inter = 0;
    for (int j = 0; j < 16; ++j) inter |= ((m >> (4 * (j >> 1) + 2 * u + (j & 1))) & 1u) << j;
    o->sm_inter[u] = inter;
    for (int k = 0; k < 8; ++k) {
      const uint32_t b0 = (o->sm_half[u] >> (2 * k)) & 1u, b1 = (o->sm_half[u] >> (2 * k + 1)) & 1u;
      o->xw[u][k] = (b0 << 15) | (b1 << 31);
    }
  }
}

namespace {

constexpr int kThreads = 256;

// ------------------------------------------------------------ loading ---
// The 16 consecutive inputs a lane processes, as loaded (two 128-bit loads of
// bf16, four of fp32), so the next unit can be prefetched into registers while
// the current one is processed.
template <typename InT>
struct Raw;
template <>
struct Raw<uint16_t> {
  uint4 a, b;
};
template <>
struct Raw<float> {
  float4 a, b, c, d;
};

__device__ __forceinline__ void load_raw(const uint16_t* p, Raw<uint16_t>& r) {
  r.a = __ldg(reinterpret_cast<const uint4*>(p));
  r.b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
}

__device__ __forceinline__ void load_raw(const float* p, Raw<float>& r) {
  const float4* q = reinterpret_cast<const float4*>(p);
  r.a = __ldg(q);
  r.b = __ldg(q + 1);
  r.c = __ldg(q + 2);
  r.d = __ldg(q + 3);
}

__device__ __forceinline__ void zero_raw(Raw<uint16_t>& r) { r.a = r.b = make_uint4(0, 0, 0, 0); }
__device__ __forceinline__ void zero_raw(Raw<float>& r) {
  r.a = r.b = r.c = r.d = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

// Widen to fp32 pairs; for bf16 the lane's sign words xw are applied to the
// packed words first (exact sign flips of the rotation's diag(s)).
__device__ __forceinline__ void unpack(const Raw<uint16_t>& r, float2 (&R)[8], const uint32_t* xw,
                                       bool signs) {
  uint32_t w[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
  if (signs) {
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] ^= xw[k];
  }
#pragma unroll
  for (int k = 0; k < 8; ++k)
    R[k] = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
}

__device__ __forceinline__ void unpack(const Raw<float>& r, float2 (&R)[8], const uint32_t*, bool) {
  R[0] = make_float2(r.a.x, r.a.y); R[1] = make_float2(r.a.z, r.a.w);
  R[2] = make_float2(r.b.x, r.b.y); R[3] = make_float2(r.b.z, r.b.w);
  R[4] = make_float2(r.c.x, r.c.y); R[5] = make_float2(r.c.z, r.c.w);
  R[6] = make_float2(r.d.x, r.d.y); R[7] = make_float2(r.d.z, r.d.w);
}

template <typename InT>
__device__ __forceinline__ void load16(const InT* p, float2 (&R)[8]) {
  Raw<InT> r;
  load_raw(p, r);
  unpack(r, R, nullptr, false);
}

template <typename InT>
__device__ __forceinline__ constexpr bool is_bf16() { return sizeof(InT) == 2; }

// Row-orientation processing of the 16 elements a lane holds (block half
// `upper` of a 1x32 run): rotation, block max (optionally reduced further by
// `reduce`), scale, rounding. Returns the packed codes; *e receives the
// exponent. g0 = source index of the first element / 8 (for the random draws).
template <typename InT, typename Reduce>
__device__ __forceinline__ uint2 quantize_halves(float2 (&R)[8], int upper, const OrientArgs& o,
                                                 uint32_t g0, Reduce reduce, int* e_out) {
  if (o.wht) {
    if (!is_bf16<InT>() && o.sm_half[upper]) apply_signs(R, o.sm_half[upper]);
    hadamard_halves(R, upper);
  }
  if (o.nv) {   // NVFP4: the lane's 16 elements are one block with an E4M3 scale
    const NvScale sc = nv_scale(absmax16(R), o.roundup, o.nv_p2k, o.nv_zmul);
    scale_all(R, sc.rcp);
    if (o.sr) {
      uint32_t w[8];
      draws16_g(o.keys, o.stream, g0, w);
      sr16(R, w);
    }
    *e_out = (int)sc.code;
    return encode16(R);
  }
  const float M = reduce(pair_absmax(R));
  const int e = scale_exponent(M, o.roundup, o.e4m3, o.e5m2);
  scale_all(R, inv_scale(e));
  if (o.sr) {
    uint32_t w[8];
    draws16_g(o.keys, o.stream, g0, w);
    sr16(R, w);
  }
  *e_out = e;
  return o.e4m3 ? uint2{0u, 0u} : encode16(R);
}

// ------------------------------------------------- row-wise, 1x32 blocks ---
// A unit is 16 consecutive elements of a row; lanes (2k, 2k+1) hold one
// 32-element block. Persistent grid-stride loop over `total` units (warp-
// uniform trip count, so the pair shuffles always see both lanes), with the
// next unit's input prefetched into registers while the current one is
// processed. The host keeps total < 2^31 and the stride (grid * kThreads)
// below 2^31, so base + stride and u + stride never wrap in 32 bits.
template <typename InT>
__global__ void __launch_bounds__(kThreads)
quant_rows_1x32_kernel(const InT* __restrict__ x, uint32_t total, FastDiv halves, int64_t cols,
                       int64_t ld, const __grid_constant__ OrientArgs o) {
  const int lane = threadIdx.x & 31, upper = threadIdx.x & 1;
  const uint32_t stride = gridDim.x * kThreads;
  const bool signs = o.sm_half[upper] != 0;
  uint32_t base = blockIdx.x * kThreads + (threadIdx.x & ~31u);
  Raw<InT> nxt;
  auto src = [&](uint32_t u) {
    const uint32_t r = fdiv(u, halves);
    return x + (int64_t)r * ld + (int64_t)(u - r * halves.d) * 16;
  };
  if (base + lane < total) load_raw(src(base + lane), nxt); else zero_raw(nxt);
  for (; base < total; base += stride) {
    const uint32_t u = base + lane;
    const bool valid = u < total;
    const Raw<InT> cur = nxt;
    if (u + stride < total) load_raw(src(u + stride), nxt); else zero_raw(nxt);
    const uint32_t r = fdiv(u, halves);
    const int64_t c0 = (int64_t)(u - r * halves.d) * 16;
    float2 R[8];
    unpack(cur, R, o.xw[upper], signs);
    int e;
    // unit u is elements 16 u .. 16 u + 15 of the row-major tensor
    const uint2 packed = quantize_halves<InT>(R, upper, o, u << 1, [](float m) { return m; }, &e);
    if (valid) {
      if (o.e4m3)
        put(reinterpret_cast<uint4*>(o.q + (int64_t)r * cols + c0), encode16_fp8(R, o.e5m2), o.q,
            o.q_bytes);
      else
        put(reinterpret_cast<uint2*>(o.q + (int64_t)r * (cols >> 1) + (c0 >> 1)), packed, o.q,
            o.q_bytes);
      if (o.nv)
        put(o.s + scale_offset32(o, r, (uint32_t)(c0 >> 4), (uint32_t)(cols >> 4)), (uint8_t)e, o.s,
            o.s_bytes);
      else if (!upper)
        store_scale32(o, r, (uint32_t)(c0 >> 5), (uint32_t)(cols >> 5), e);
    }
  }
}

// --------------------------------------- 64 x 64 tiles: both orientations ---
// Used when the column-wise output is requested or a 32x32 block is in play.
// Persistent, warp-specialized CTAs walk the 64x64 tiles of x:
//  * warp 4 (one lane) streams tiles with TMA (cp.async.bulk.tensor, 128-byte
//    swizzle, zero fill past the tensor's edges) into a 3-stage shared ring,
//    guarded by full / empty mbarriers;
//  * warps 0-3 consume. Phase 1: warp w owns the 32 x 32 block (rows 32(w%2) +
//    lane, columns 32(w/2) ..): each lane holds one whole 1x32 run of its row,
//    so the rotation and the 1x32 max are in-thread and the 32x32 max is one
//    warp reduction; it writes the row-wise output (16 bytes per lane) and,
//    for stochastic rounding of the column orientation, the draws keyed by
//    source index (computed once when both orientations share seed and stream).
//    Phase 2: a lane holds a whole column run. With stochastic column
//    rounding warp w owns columns 32(w/2) + lane of rows 32(w%2) .., the same
//    32 x 32 block, so the shared draws it reads are the ones it wrote (a warp
//    barrier, not a CTA one); otherwise columns 32(w%2) + lane of rows
//    32(w/2) .. (the 64 x 64 general variant keeps this mapping and a CTA
//    barrier).
// Bank conflicts: row reads of 8 rows hit 8 different swizzled chunks; column
// reads of 32 lanes read one 64-byte row segment.
constexpr int kTile = 64;
constexpr int kStages = 3;
constexpr int kConsumers = 128;
constexpr int kTileThreads = kConsumers + 32;
constexpr uint32_t kCodeTileBytes = kTile * kTile / 2;   // one orientation's E2M1 codes of a tile
constexpr uint64_t kQuantWaitNs = 2000000000ull;

// Byte offset of element (r, c) in a 64 x 64 tile as TMA lays it out with the
// 128-byte swizzle: 128-byte rows, 16-byte chunk j of row r at chunk j ^ (r % 8).
// fp32 tiles are two 64 x 32 boxes, 8 KB apart.
__device__ __forceinline__ uint32_t tile_off(int r, int c, uint16_t) {
  return (uint32_t)(r * 128 + ((((c >> 3) ^ r) & 7) << 4) + ((c & 7) << 1));
}
__device__ __forceinline__ uint32_t tile_off(int r, int c, float) {
  return (uint32_t)(((c >> 5) << 13) + r * 128 + (((((c & 31) >> 2) ^ r) & 7) << 4) + ((c & 3) << 2));
}

// 32 consecutive elements (c % 32 == 0) of row r of a staged tile.
__device__ __forceinline__ void read_run(const uint8_t* st, int r, int c, float2 (&R)[16], uint16_t) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 q = *reinterpret_cast<const uint4*>(st + tile_off(r, c + 8 * i, uint16_t()));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      R[4 * i + k] = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
  }
}
__device__ __forceinline__ void read_run(const uint8_t* st, int r, int c, float2 (&R)[16], float) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 q = *reinterpret_cast<const float4*>(st + tile_off(r, c + 4 * i, 0.0f));
    R[2 * i] = make_float2(q.x, q.y);
    R[2 * i + 1] = make_float2(q.z, q.w);
  }
}
// Column reads: for rows r0 + 8 j + t (r0 % 8 == 0) of column c the swizzle
// term depends on t only, so a lane keeps eight byte offsets o[t] (row r0 + t)
// and reaches row r0 + 8 j + t at o[t] + 1024 j (an immediate).
__device__ __forceinline__ void col_offsets(int r0, int c, uint32_t (&o)[8], uint16_t) {
#pragma unroll
  for (int t = 0; t < 8; ++t) o[t] = tile_off(r0 + t, c, uint16_t());
}
__device__ __forceinline__ void col_offsets(int r0, int c, uint32_t (&o)[8], float) {
#pragma unroll
  for (int t = 0; t < 8; ++t) o[t] = tile_off(r0 + t, c, 0.0f);
}

// 32 consecutive rows (o from col_offsets for the run's first row) of a column.
__device__ __forceinline__ void read_col(const uint8_t* st, const uint32_t (&o)[8], float2 (&R)[16],
                                         uint16_t) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t a = *reinterpret_cast<const uint16_t*>(st + o[(2 * k) & 7] + 1024 * (k >> 2));
    const uint32_t b = *reinterpret_cast<const uint16_t*>(st + o[(2 * k + 1) & 7] + 1024 * (k >> 2));
    R[k] = make_float2(__uint_as_float(a << 16), __uint_as_float(b << 16));
  }
}
__device__ __forceinline__ void read_col(const uint8_t* st, const uint32_t (&o)[8], float2 (&R)[16],
                                         float) {
#pragma unroll
  for (int k = 0; k < 16; ++k)
    R[k] = make_float2(*reinterpret_cast<const float*>(st + o[(2 * k) & 7] + 1024 * (k >> 2)),
                       *reinterpret_cast<const float*>(st + o[(2 * k + 1) & 7] + 1024 * (k >> 2)));
}

__device__ __forceinline__ bool same_draws(const OrientArgs& a, const OrientArgs& b) {
  return a.sr && b.sr && a.seed == b.seed && a.stream == b.stream;
}

__device__ __forceinline__ void named_sync_consumers() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// 64x64 blocks: each of the four consumer warps holds the max of one 32x32
// quarter of the tile; combine them through shared memory. Every consumer
// warp calls this (it contains a barrier of the four).
__device__ __forceinline__ float tile_max4(float m, float* slots, int warp, int lane) {
  if (lane == 0) slots[warp] = m;
  named_sync_consumers();
  return fmaxf(fmaxf(slots[0], slots[1]), fmaxf(slots[2], slots[3]));
}

// Bounded wait; false on timeout (which also raises the CTA's abort flag and
// the library error word) or when the CTA has already aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t par, uint32_t* abort_flag) {
  if (ptx::mbar_try_wait(bar, par)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (;;) {
    if (ptx::mbar_try_wait_sleep(bar, par, 500000u)) return true;
    {
      if (*reinterpret_cast<volatile uint32_t*>(abort_flag)) return false;
      if (ptx::globaltimer_ns() - t0 > kQuantWaitNs) {
        *reinterpret_cast<volatile uint32_t*>(abort_flag) = 1u;
        atomicExch(&g_quant_error, 6u);  // MXFP4_ERR_TIMEOUT
        return false;
      }
    }
  }
}

// kVar: kLean (1x32 / 32x32 blocks, E2M1 codes), kGeneral (also 64x64 blocks
// and E4M3 codes, any mix of orientations), kNv (both requested orientations
// NVFP4: the lean structure with the 1x16 E4M3-scale step).
enum : int { kLean = 0, kGeneral = 1, kNv = 2 };

// kProf: 0 reads the rounding and rotation flags at run time; 1..3 fix them at
// compile time for a dual-orientation lean or NVFP4 call (both outputs
// requested, no row-wise rotation):
//   1: rows nearest, columns nearest without rotation (weights);
//   2: rows nearest, columns stochastic with rotation (activations);
//   3: rows stochastic, columns stochastic with rotation (output gradients).
// The fixed variants give the compiler straight-line code (the same bits).
template <int kProf>
struct TileProfile {
  static constexpr bool fixed = kProf != 0;
  static constexpr bool row_sr = kProf == 3, row_wht = false;
  static constexpr bool col_sr = kProf >= 2, col_wht = kProf >= 2;
};

template <typename InT, int kVar, int kProf = 0>
__global__ void __launch_bounds__(kTileThreads, kProf == 1 ? 4 : 3)
quant_tile_kernel(const __grid_constant__ CUtensorMap tmx, int64_t rows, int64_t cols,
                  uint32_t ntiles, FastDiv tiles_x, const __grid_constant__ OrientArgs orow,
                  const __grid_constant__ OrientArgs ocol, int do_row, int do_col,
                  const __grid_constant__ CUtensorMap tmqr, const __grid_constant__ CUtensorMap tmqc) {
  constexpr uint32_t kStageBytes = kTile * kTile * sizeof(InT);
  constexpr uint32_t kBitsBytes = kTile * kTile * 2;
  // The nearest-only MXFP4 profile (weights) stages each tile's E2M1 codes in
  // shared memory and writes them with one tensor store per orientation (64
  // rows of 32 bytes: whole sectors) instead of a 16-byte store per lane on a
  // row of its own: W of the 70B layer 0.169 -> 0.140 ms. The stochastic
  // profiles and the NVFP4 weights profile (two scales per 32-run) measured
  // 1-6 % slower with it (the extra barrier and staging cost more than the
  // stores save), so they keep the per-lane stores, as do bounds-checking
  // builds (each store checked).
#ifdef MXFP4_BOUNDS_CHECK
  constexpr bool kTmaCodes = false;
#else
  constexpr bool kTmaCodes = kVar == kLean && kProf == 1;
#endif
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* tbits0 = sm + kStages * kStageBytes;   // two draw buffers, swizzled like bf16 tiles
  uint8_t* stage0 = tbits0 + 2 * kBitsBytes;       // code staging [tile parity][orientation][64][32]
  uint64_t* full = reinterpret_cast<uint64_t*>(stage0 + 4 * kCodeTileBytes);
  uint64_t* empty = full + kStages;
  uint32_t* abort_flag = reinterpret_cast<uint32_t*>(empty + kStages);

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  auto origin = [&](uint32_t tl, int64_t& R0, int64_t& C0) {
    const uint32_t ty = fdiv(tl, tiles_x);
    R0 = (int64_t)ty * kTile;
    C0 = (int64_t)(tl - ty * tiles_x.d) * kTile;
  };

  if (t == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty[s]), kConsumers / 32);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumers / 32) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmx);
      uint32_t j = 0;
      for (uint32_t tl = blockIdx.x; tl < ntiles; tl += gridDim.x, ++j) {
        const int s = (int)(j % kStages);
        if (j >= kStages &&
            !wait_or_abort(ptx::smem_u32(&empty[s]), ((j / kStages) - 1) & 1u, abort_flag))
          break;
        int64_t R0, C0;
        origin(tl, R0, C0);
        const uint32_t bar = ptx::smem_u32(&full[s]);
        const uint32_t dst = ptx::smem_u32(sm + s * kStageBytes);
        ptx::mbar_arrive_expect_tx(bar, kStageBytes);
        ptx::tma_load_2d(dst, &tmx, (int32_t)C0, (int32_t)R0, bar);
        if (sizeof(InT) == 4) ptx::tma_load_2d(dst + 8192, &tmx, (int32_t)C0 + 32, (int32_t)R0, bar);
      }
      // After an abort, wait (bounded) for the loads still in flight.
      if (*reinterpret_cast<volatile uint32_t*>(abort_flag)) {
        for (uint32_t q = (j > kStages ? j - kStages : 0); q < j; ++q) {
          const uint32_t bar = ptx::smem_u32(&full[q % kStages]);
          const uint64_t t0 = ptx::globaltimer_ns();
          while (!ptx::mbar_try_wait(bar, (q / kStages) & 1u))
            if (ptx::globaltimer_ns() - t0 > kQuantWaitNs / 8) break;
        }
      }
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  __shared__ float bmax[2][2][4];   // [tile parity][orientation][warp]: 64x64 maxima
  const bool share = do_row && do_col && same_draws(orow, ocol);
  uint32_t j = 0;
  for (uint32_t tl = blockIdx.x; tl < ntiles; tl += gridDim.x, ++j) {
    const int s = (int)(j % kStages);
    const uint8_t* st = sm + s * kStageBytes;
    uint8_t* tb = tbits0 + (j & 1) * kBitsBytes;
    uint8_t* stg = stage0 + (j & 1) * 2 * kCodeTileBytes;   // row codes, then column codes
    int ok = 0;
    if (lane == 0) ok = wait_or_abort(ptx::smem_u32(&full[s]), (j / kStages) & 1u, abort_flag);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    int64_t R0, C0;
    origin(tl, R0, C0);

    if constexpr (kVar != kGeneral) {
      constexpr bool nv = kVar == kNv;
      using Pf = TileProfile<kProf>;
      const bool drow = Pf::fixed || do_row, dcol = Pf::fixed || do_col;
      const bool rsr = Pf::fixed ? Pf::row_sr : (bool)orow.sr;
      const bool rwht = Pf::fixed ? Pf::row_wht : (bool)orow.wht;
      const bool csr = Pf::fixed ? Pf::col_sr : (bool)ocol.sr;
      const bool cwht = Pf::fixed ? Pf::col_wht : (bool)ocol.wht;
      // ---- phase 1: rows ----
      if (ok) {
        const int rl = 32 * (warp & 1) + lane, cl = 32 * (warp >> 1);
        const int64_t r = R0 + rl, c = C0 + cl;
        const bool valid = r < rows && c < cols;
        float2 R[16];
        read_run(st, rl, cl, R, InT());
        uint32_t w[16];
        if (dcol && csr) {
          draws32_g(ocol.keys, ocol.stream, (uint32_t)r * (uint32_t)(cols >> 3) + (uint32_t)(c >> 3), w);
  #pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(tb + tile_off(rl, cl + 8 * i, uint16_t())) =
                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
        if (drow) {
          if (rwht) hadamard32_lane(R, orow.sign_mask, orow.sgn);
          float M = nv ? 0.0f : absmax32(R);    // NVFP4 takes its two 16-block maxima itself
          if (!nv && orow.block) M = warp_max(M);
          if (rsr && !share) draws32_g(orow.keys, orow.stream, (uint32_t)r * (uint32_t)(cols >> 3) + (uint32_t)(c >> 3), w);
          const int e = scale_run32<false, nv>(R, orow, M, w);
          if constexpr (kTmaCodes) {
            *reinterpret_cast<uint4*>(stg + rl * 32 + (cl >> 5) * 16) = encode32(R);
            if (valid) store_run_scales32<nv>(orow, (uint32_t)r, (uint32_t)c, (uint32_t)cols, e);
          } else if (valid) {
            store_run32<false>(orow, r, c, cols, R);
            store_run_scales32<nv>(orow, (uint32_t)r, (uint32_t)c, (uint32_t)cols, e);
          }
        }
      }

      // ---- phase 2: columns (quantization of x^T along rows) ----
      if (dcol) {
        // With column draws each warp quantizes the same 32x32 block in both
        // phases, so the draws it reads are the ones it wrote in phase 1 (a
        // warp barrier suffices); without them it takes the other block of
        // its column half, measured 1.5 % faster for the weights profile.
        if (csr) __syncwarp();
        if (ok) {
          const int cl = 32 * (csr ? warp >> 1 : warp & 1) + lane, rl = 32 * (csr ? warp & 1 : warp >> 1);
          const int64_t oc = C0 + cl, k0 = R0 + rl;
          const bool valid = oc < cols && k0 < rows;
          float2 R[16];
          uint32_t o[8];
          col_offsets(rl, cl, o, InT());
          read_col(st, o, R, InT());
          if (cwht) hadamard32_lane(R, ocol.sign_mask, ocol.sgn);
          float M = nv ? 0.0f : absmax32(R);
          if (!nv && ocol.block) M = warp_max(M);
          // The draws of column elements (rl + 2k, rl + 2k + 1), each 16-bit
          // draw read straight into its float 2^23 + r.
          float2 F[16];
          if (csr) {
            uint32_t ob[8];   // the draw buffer is laid out like a bf16 tile
            col_offsets(rl, cl, ob, uint16_t());
  #pragma unroll
            for (int k = 0; k < 16; ++k) {
              const uint32_t a = *reinterpret_cast<const uint16_t*>(tb + ob[(2 * k) & 7] + 1024 * (k >> 2));
              const uint32_t b = *reinterpret_cast<const uint16_t*>(tb + ob[(2 * k + 1) & 7] + 1024 * (k >> 2));
              F[k] = make_float2(__uint_as_float(0x4B000000u | a), __uint_as_float(0x4B000000u | b));
            }
          }
          const int e = scale_run32<false, nv>(R, ocol, M, F);
          if constexpr (kTmaCodes) {
            *reinterpret_cast<uint4*>(stg + kCodeTileBytes + cl * 32 + (rl >> 5) * 16) = encode32(R);
            if (valid) store_run_scales32<nv>(ocol, (uint32_t)oc, (uint32_t)k0, (uint32_t)rows, e);
          } else if (valid) {
            store_run32<false>(ocol, oc, k0, rows, R);
            store_run_scales32<nv>(ocol, (uint32_t)oc, (uint32_t)k0, (uint32_t)rows, e);
          }
        }
      }

      if constexpr (kTmaCodes) {
        // Every consumer's staged codes reach the tensor-store (async) proxy;
        // thread 0 first waits until the previous tile's stores have read
        // their staging buffer (the one the next tile writes), then issues
        // this tile's stores. Out-of-range rows and columns of a ragged tile
        // are clipped by the tensor maps.
        ptx::fence_proxy_async();
        if (t == 0) ptx::bulk_wait_read<0>();
        named_sync_consumers();
        if (t == 0 && ok) {
          if (drow) ptx::tma_store_2d(&tmqr, (int32_t)(C0 >> 1), (int32_t)R0, ptx::smem_u32(stg));
          if (dcol)
            ptx::tma_store_2d(&tmqc, (int32_t)(R0 >> 1), (int32_t)C0,
                              ptx::smem_u32(stg + kCodeTileBytes));
          ptx::bulk_commit();
        }
      }
    } else {
      // 64x64 blocks: the block max needs all four consumer warps, so the
      // barriers sit outside the per-warp "ok" branches.
      // ---- phase 1: rows ----
      {
        const int rl = 32 * (warp & 1) + lane, cl = 32 * (warp >> 1);
        const int64_t r = R0 + rl, c = C0 + cl;
        const bool valid = r < rows && c < cols;
        float2 R[16];
        uint32_t w[16];
        float M = 0.0f;
        if (ok) {
          read_run(st, rl, cl, R, InT());
          if (do_col && ocol.sr) {
            draws32(ocol.keys, ocol.stream, (uint64_t)(r * cols + c), w);
  #pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<uint4*>(tb + tile_off(rl, cl + 8 * i, uint16_t())) =
                  make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
          if (do_row) {
            if (orow.wht) hadamard32_lane(R, orow.sign_mask, orow.sgn);
            M = absmax32(R);
            if (orow.block) M = warp_max(M);
          }
        }
        if (do_row && orow.block == 2) M = tile_max4(M, bmax[j & 1][0], warp, lane);
        if (ok && do_row) {
          if (orow.sr && !share) draws32(orow.keys, orow.stream, (uint64_t)(r * cols + c), w);
          const int e = scale_run32(R, orow, M, w);
          if (valid) {
            store_run32(orow, r, c, cols, R);
            store_run_scales(orow, r, c, cols, e);
          }
        }
      }

      // ---- phase 2: columns (quantization of x^T along rows) ----
      if (do_col) {
        if (ocol.sr) named_sync_consumers();   // the draws were written by other warps
        const int cl = 32 * (warp & 1) + lane, rl = 32 * (warp >> 1);
        const int64_t oc = C0 + cl, k0 = R0 + rl;
        const bool valid = oc < cols && k0 < rows;
        float2 R[16];
        float M = 0.0f;
        if (ok) {
          uint32_t o[8];
          col_offsets(rl, cl, o, InT());
          read_col(st, o, R, InT());
          if (ocol.wht) hadamard32_lane(R, ocol.sign_mask, ocol.sgn);
          M = absmax32(R);
          if (ocol.block) M = warp_max(M);
        }
        if (ocol.block == 2) M = tile_max4(M, bmax[j & 1][1], warp, lane);
        if (ok) {
          uint32_t w[16];
          if (ocol.sr) {
            uint32_t ob[8];   // the draw buffer is laid out like a bf16 tile
            col_offsets(rl, cl, ob, uint16_t());
  #pragma unroll
            for (int k = 0; k < 16; ++k) {
              const uint32_t a = *reinterpret_cast<const uint16_t*>(tb + ob[(2 * k) & 7] + 1024 * (k >> 2));
              const uint32_t b = *reinterpret_cast<const uint16_t*>(tb + ob[(2 * k + 1) & 7] + 1024 * (k >> 2));
              w[k] = __byte_perm(a, b, 0x5410);
            }
          }
          const int e = scale_run32(R, ocol, M, w);
          if (valid) {
            store_run32(ocol, oc, k0, rows, R);
            store_run_scales(ocol, oc, k0, rows, e);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&empty[s]));
  }
  if constexpr (kTmaCodes) {
    if (t == 0) ptx::bulk_wait<0>();   // the last stores are complete before the CTA exits
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
  const int upper = threadIdx.x & 1;
  const uint32_t m = (sign_mask >> (16 * upper)) & 0xFFFFu;
  float2 R[8];
  if (valid) {
    load16(x + r * ld + c0, R);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) R[k] = make_float2(0.0f, 0.0f);
  }
  if (!inverse) apply_signs(R, m);
  hadamard_halves(R, upper);
  if (inverse) apply_signs(R, m);
  if (valid) {
    float4* out = reinterpret_cast<float4*>(y + r * cols + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      put(out + i, make_float4(R[2 * i].x, R[2 * i].y, R[2 * i + 1].x, R[2 * i + 1].y), y,
          (uint64_t)(rows * cols) * 4);
  }
}

// ---------------------------------------------------------- dequantize ---
// Full E4M3 byte -> value (sign, NaN for S.1111.111), exact.
__device__ __forceinline__ float e4m3_decode(uint32_t b) {
  const uint32_t mag = b & 0x7Fu;
  const float v = mag == 0x7Fu ? __uint_as_float(0x7FC00000u) : e4m3_value(mag);
  return (b & 0x80u) ? -v : v;
}

// Full E5M2 byte -> value, exact: exponent field 31 is infinity (mantissa 0)
// or NaN; field 0 the subnormals m 2^-16; else (1 + m/4) 2^(E - 15).
__device__ __forceinline__ float e5m2_decode(uint32_t b) {
  const uint32_t E = (b >> 2) & 31u, m = b & 3u;
  float v;
  if (E == 31u)
    v = __uint_as_float(m ? 0x7FC00000u : 0x7F800000u);
  else if (E == 0u)
    v = __fmul_rn((float)m, 1.52587890625e-05f);
  else
    v = __uint_as_float(((E + 112u) << 23) | (m << 21));
  return (b & 0x80u) ? -v : v;
}

// E8M0 byte -> 2^(byte - 127); 0xFF is NaN.
__device__ __forceinline__ float e8m0_decode(uint32_t sb) {
  return sb == 255u ? __uint_as_float(0x7FC00000u)
         : sb == 0u ? __uint_as_float(0x00400000u)   // 2^-127 (subnormal)
                    : __uint_as_float(sb << 23);
}

// One thread per 16 consecutive elements of a row. Every product is exact
// (an E2M1 or E4M3 value times a power of two or an E4M3 scale).
//  kFmt 0: MXFP4 (E2M1 codes, E8M0 scale per 32);
//  kFmt 1: MXFP8 (E4M3 codes, one byte each, E8M0 scale per 32);
//  kFmt 2: NVFP4 (E2M1 codes, E4M3 scale per 16, times p2k = 2^tensor_exp);
//  kFmt 3: MXFP8 with E5M2 codes, one byte each, E8M0 scale per 32.
template <int kFmt>
__global__ void __launch_bounds__(kThreads)
dequant_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int mma_layout,
               int64_t rows, int64_t cols, float p2k, float* __restrict__ out) {
  const int64_t halves = cols >> 4;
  const int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (t >= rows * halves) return;
  const int64_t r = t / halves, c0 = (t - r * halves) << 4;
  const int64_t nkb = kFmt == 2 ? cols >> 4 : cols >> 5;
  const int64_t kb = kFmt == 2 ? c0 >> 4 : c0 >> 5;
  const int64_t so = mma_layout ? mma_scale_offset(r, kb, nkb) : r * nkb + kb;
  const uint32_t sb = __ldg(s + so);
  const float scale = kFmt == 2 ? __fmul_rn(e4m3_decode(sb), p2k) : e8m0_decode(sb);
  float v[16];
  if constexpr (kFmt == 1 || kFmt == 3) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(q + r * cols + c0));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t b = (ws[j >> 2] >> (8 * (j & 3))) & 0xFFu;
      v[j] = __fmul_rn(kFmt == 3 ? e5m2_decode(b) : e4m3_decode(b), scale);
    }
  } else {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(q + r * (cols >> 1) + (c0 >> 1)));
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t code = ((j < 8 ? w.x : w.y) >> (4 * (j & 7))) & 0xFu;
      const float m = e2m1_magnitude(code & 7u);
      v[j] = __fmul_rn((code & 8u) ? -m : m, scale);
    }
  }
  float4* o = reinterpret_cast<float4*>(out + r * cols + c0);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    put(o + i, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]), out,
        (uint64_t)(rows * cols) * 4);
}

// ------------------------------------------------------- tensor max-abs ---
// Max |x| over a [rows, cols] tensor, as the bit pattern of a non-negative
// fp32 (such patterns order like the values), into *amax_bits, which the
// host zeroes first. CTAs stride over rows; a row's 16-byte vectors (8 bf16
// or 4 fp32) are spread over the CTA's threads; warp and CTA maxima, then one
// atomicMax per CTA.
template <typename InT>
__global__ void __launch_bounds__(kThreads)
amax_kernel(const InT* __restrict__ x, int64_t rows, int64_t vecs, int64_t ld,
            uint32_t* __restrict__ amax_bits) {
  uint32_t m = 0;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4* row = reinterpret_cast<const uint4*>(x + r * ld);
    for (int64_t v = threadIdx.x; v < vecs; v += kThreads) {
      const uint4 q = __ldg(row + v);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (sizeof(InT) == 2) {
          m = max(m, max(w[i] & 0x7FFF0000u, (w[i] << 16) & 0x7FFF0000u));
        } else {
          m = max(m, w[i] & 0x7FFFFFFFu);
        }
      }
    }
  }
  m = __reduce_max_sync(0xffffffffu, m);
  __shared__ uint32_t part[kThreads / 32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < kThreads / 32 ? part[threadIdx.x] : 0u;
    m = __reduce_max_sync(0xffffffffu, m);
    if (threadIdx.x == 0 && m) atomicMax(amax_bits, m);
  }
}

// NVFP4 per-tensor exponent from the max-abs: the smallest k with
// 2688 * 2^k >= amax, clamped to [-100, 100], 0 for amax = 0. For a normal
// amax = (1 + f) 2^E: 2688 * 2^(E - 11) = 1.3125 * 2^E covers it iff
// f <= 0.3125 (fraction bits <= 0x280000), else k = E - 10.
__global__ void nv_tensor_exp_kernel(const uint32_t* __restrict__ amax_bits, int32_t* __restrict__ k) {
  const uint32_t b = *amax_bits;
  int32_t e;
  if (b == 0u) {
    e = 0;
  } else if (b < 0x00800000u) {
    e = -100;
  } else {
    const int32_t E = (int32_t)(b >> 23) - 127;
    e = (b & 0x7FFFFFu) <= 0x280000u ? E - 11 : E - 10;
    e = max(-100, min(100, e));
  }
  *k = e;
}

inline unsigned blocks_for(int64_t threads) { return (unsigned)((threads + kThreads - 1) / kThreads); }

// Persistent grids: as many CTAs as can be resident (queried once per device
// and kernel), never more than there are work items.
template <typename K>
unsigned resident_ctas(K kernel, int64_t items, int smem, int threads) {
  struct Entry {
    const void* fn;
    int dev, per_sm, sms;
  };
  static Entry cache[64];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  const void* fn = reinterpret_cast<const void*>(kernel);
  int per_sm = 0, sms = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].fn == fn && cache[i].dev == dev) {
        per_sm = cache[i].per_sm;
        sms = cache[i].sms;
      }
    if (!per_sm) {
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      int n = 0;
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
      per_sm = n > 0 ? n : 1;
      if (used < 64) cache[used++] = Entry{fn, dev, per_sm, sms};
    }
  }
  const int64_t want = (int64_t)per_sm * sms;
  return (unsigned)(items < want ? items : want);
}

// Opts every tile-kernel instantiation of one input type into `smem` bytes of
// dynamic shared memory, once per device.
template <typename InT>
void set_tile_smem_once(int dev, int smem) {
  static bool done[kMaxDevices] = {false};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return;
  const void* kernels[] = {
      reinterpret_cast<const void*>(quant_tile_kernel<InT, kLean>),
      reinterpret_cast<const void*>(quant_tile_kernel<InT, kGeneral>),
      reinterpret_cast<const void*>(quant_tile_kernel<InT, kNv>),
      reinterpret_cast<const void*>(quant_tile_kernel<InT, kLean, 1>),
      reinterpret_cast<const void*>(quant_tile_kernel<InT, kLean, 2>),
      reinterpret_cast<const void*>(quant_tile_kernel<InT, kLean, 3>),
      reinterpret_cast<const void*>(quant_tile_kernel<InT, kNv, 1>),
      reinterpret_cast<const void*>(quant_tile_kernel<InT, kNv, 2>),
      reinterpret_cast<const void*>(quant_tile_kernel<InT, kNv, 3>)};
  for (const void* k : kernels)
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  done[dev] = true;
}

template <typename InT>
cudaError_t quantize_impl(const InT* x, int64_t rows, int64_t cols, int64_t ld,
                          const OrientArgs* row, const OrientArgs* col, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const bool tile = col != nullptr || (row && row->block);
  if (!tile) {
    const int64_t total = rows * (cols >> 4);
    const unsigned grid =
        resident_ctas(quant_rows_1x32_kernel<InT>, (total + kThreads - 1) / kThreads, 0, kThreads);
    if (total >= (1ll << 31) || (int64_t)grid * kThreads >= (1ll << 31)) return cudaErrorInvalidValue;
    (void)cudaGetLastError();  // drop a stale error left by an earlier call
    quant_rows_1x32_kernel<InT><<<grid, kThreads, 0, st>>>(
        x, (uint32_t)total, make_fastdiv((uint32_t)(cols >> 4)), cols, ld, *row);
    return cudaGetLastError();
  }
  CUtensorMap tm;
  const bool bf = sizeof(InT) == 2;
  if (!make_tma_2d(&tm, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                   sizeof(InT), x, rows, cols, ld, kTile, bf ? 64 : 32))
    return cudaErrorInvalidValue;
  constexpr int smem = kStages * kTile * kTile * sizeof(InT) + 2 * kTile * kTile * 2 +
                       4 * kCodeTileBytes + 256 + 1024;
  int dev = 0;
  const cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return de;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  set_tile_smem_once<InT>(dev, smem);
  OrientArgs dummy{};
  const int64_t tx = (cols + kTile - 1) / kTile, ty = (rows + kTile - 1) / kTile;
  // The lean variant covers 1x32 / 32x32 E2M1 outputs, the NVFP4 one outputs
  // that are all 1x16; anything else (64x64 blocks, E4M3 codes, NVFP4 mixed
  // with another block type) takes the general one.
  auto is_lean = [](const OrientArgs* o) { return !o || (o->block != 2 && !o->e4m3 && !o->nv); };
  auto is_nv = [](const OrientArgs* o) { return !o || o->nv; };
  auto kern = (is_lean(row) && is_lean(col)) ? quant_tile_kernel<InT, kLean>
              : (is_nv(row) && is_nv(col))   ? quant_tile_kernel<InT, kNv>
                                             : quant_tile_kernel<InT, kGeneral>;
  // Dual-orientation lean or NVFP4 calls whose rounding / rotation flags match
  // a fixed profile take that profile's kernel.
  const bool lean2 = row && col && is_lean(row) && is_lean(col);
  const bool nv2 = row && col && row->nv && col->nv;
  if ((lean2 || nv2) && !row->wht) {
    const int prof = (!row->sr && !col->sr && !col->wht) ? 1
                     : (!row->sr && col->sr && col->wht) ? 2
                     : (row->sr && col->sr && col->wht)  ? 3 : 0;
    if (prof == 1) kern = lean2 ? quant_tile_kernel<InT, kLean, 1> : quant_tile_kernel<InT, kNv, 1>;
    if (prof == 2) kern = lean2 ? quant_tile_kernel<InT, kLean, 2> : quant_tile_kernel<InT, kNv, 2>;
    if (prof == 3) kern = lean2 ? quant_tile_kernel<InT, kLean, 3> : quant_tile_kernel<InT, kNv, 3>;
  }
  // Tensor maps of the E2M1 code outputs, written by the MXFP4 weights
  // profile's tile stores (64 rows x 32 bytes); unused by the other variants
  // and by bounds-checking builds, which store per lane.
  CUtensorMap tqr{}, tqc{};
#ifndef MXFP4_BOUNDS_CHECK
  if (kern == quant_tile_kernel<InT, kLean, 1>) {
    if (row && !make_byte_store_map(&tqr, row->q, rows, cols / 2, kTile, 32))
      return cudaErrorInvalidValue;
    if (col && !make_byte_store_map(&tqc, col->q, cols, rows / 2, kTile, 32))
      return cudaErrorInvalidValue;
  }
#endif
  const unsigned grid = resident_ctas(kern, tx * ty, smem, kTileThreads);
  (void)cudaGetLastError();  // drop a stale error left by an earlier call
  kern<<<grid, kTileThreads, smem, st>>>(
      tm, rows, cols, (uint32_t)(tx * ty), make_fastdiv((uint32_t)tx), row ? *row : dummy,
      col ? *col : dummy, row != nullptr, col != nullptr, tqr, tqc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const void* x, bool f32_in, int64_t rows, int64_t cols, int64_t ld,
                            const OrientArgs* row, const OrientArgs* col, cudaStream_t st) {
  return f32_in ? quantize_impl(static_cast<const float*>(x), rows, cols, ld, row, col, st)
                : quantize_impl(static_cast<const uint16_t*>(x), rows, cols, ld, row, col, st);
}

cudaError_t launch_amax(const void* x, bool f32_in, int64_t rows, int64_t cols, int64_t ld,
                        float* amax, int32_t* tensor_exp, cudaStream_t st) {
  uint32_t* bits = reinterpret_cast<uint32_t*>(amax);
  cudaError_t e = cudaMemsetAsync(bits, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  (void)cudaGetLastError();  // drop a stale error left by an earlier call
  if (rows > 0 && cols > 0) {
    const int64_t want = rows < (1ll << 31) ? rows : (1ll << 31) - 1;
    if (f32_in) {
      const unsigned grid = resident_ctas(amax_kernel<float>, want, 0, kThreads);
      amax_kernel<float><<<grid, kThreads, 0, st>>>(static_cast<const float*>(x), rows, cols / 4,
                                                    ld, bits);
    } else {
      const unsigned grid = resident_ctas(amax_kernel<uint16_t>, want, 0, kThreads);
      amax_kernel<uint16_t><<<grid, kThreads, 0, st>>>(static_cast<const uint16_t*>(x), rows,
                                                       cols / 8, ld, bits);
    }
  }
  if (tensor_exp) nv_tensor_exp_kernel<<<1, 1, 0, st>>>(bits, tensor_exp);
  return cudaGetLastError();
}

cudaError_t launch_hadamard32(const void* x, bool f32_in, int64_t rows, int64_t cols, int64_t ld,
                              uint32_t sign_mask, bool inverse, float* y, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const unsigned nb = blocks_for(rows * (cols >> 4));
  (void)cudaGetLastError();  // drop a stale error left by an earlier call
  if (f32_in)
    hadamard32_kernel<float><<<nb, kThreads, 0, st>>>(static_cast<const float*>(x), rows, cols,
                                                      ld, sign_mask, inverse, y);
  else
    hadamard32_kernel<uint16_t><<<nb, kThreads, 0, st>>>(static_cast<const uint16_t*>(x), rows,
                                                         cols, ld, sign_mask, inverse, y);
  return cudaGetLastError();
}

cudaError_t read_quant_error(uint32_t* err) {
  cudaError_t e = cudaMemcpyFromSymbol(err, g_quant_error, sizeof(uint32_t));
  if (e == cudaSuccess && *err) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_quant_error, &zero, sizeof(uint32_t));
  }
  return e;
}

cudaError_t launch_dequantize(const uint8_t* q, const uint8_t* s, bool mma_layout, int64_t rows,
                              int64_t cols, int fmt, float p2k, float* out, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  (void)cudaGetLastError();  // drop a stale error left by an earlier call
  const unsigned nb = blocks_for(rows * (cols >> 4));
  if (fmt == 1)
    dequant_kernel<1><<<nb, kThreads, 0, st>>>(q, s, mma_layout, rows, cols, p2k, out);
  else if (fmt == 3)
    dequant_kernel<3><<<nb, kThreads, 0, st>>>(q, s, mma_layout, rows, cols, p2k, out);
  else if (fmt == 2)
    dequant_kernel<2><<<nb, kThreads, 0, st>>>(q, s, mma_layout, rows, cols, p2k, out);
  else
    dequant_kernel<0><<<nb, kThreads, 0, st>>>(q, s, mma_layout, rows, cols, p2k, out);
  return cudaGetLastError();
}

}  // namespace mx
