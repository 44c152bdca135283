// gemm.cu -- block-scaled MXFP4 GEMM on the 5th-generation tensor cores
// (sm_103a: tcgen05.mma kind::mxf4 with E8M0 block scales).
//
//   C[m, n] = sum_k (a[m,k] * 2^(sa[m,k/32]-127)) * (b[n,k] * 2^(sb[n,k/32]-127))
//
// for packed E2M1 operands, both K-major, fp32 accumulation in tensor memory.
// This is the "MXFP4 GEMM" of "Training LLMs with MXFP4" (Abstract) that all
// three training products -- Fprop, Dgrad, Wgrad of "Pretraining large
// language models with MXFP4" (Abstract) -- reduce to.
//
// Design (one CTA per SM, persistent over output tiles):
//  * tile 128 x 256 x 256 (M x N x K), 4-stage shared-memory ring;
//  * warp 0: TMA producer -- 128-byte-swizzled tensor loads of the A and B
//    code tiles, plus bulk copies of the matching 512-byte scale tiles (the
//    scales are stored in the tensor-core scale layout, so each is one
//    contiguous copy);
//  * warp 1: allocates tensor memory, moves each stage's scales into it with
//    tcgen05.cp, and issues 4 tcgen05.mma (K = 64 each) per stage from one
//    thread; tcgen05.commit releases the stage and, after the last k-block,
//    hands the accumulator to the epilogue;
//  * warps 2..9: epilogue -- drain the 128 x 256 fp32 accumulator from tensor
//    memory into registers, release it so the next tile's MMAs can start, then
//    store to global memory.
// The CTA-pair kernel below (cta_group::2, 256 x 256 tiles) is the one used
// whenever M % 256 == 0; it also serves the MXFP8 (kind::mxf8f6f4, E4M3
// operands) and NVFP4 (kind::mxf4nvf4, E4M3 scales per 16) GEMMs. Epilogues
// store C as fp32 or bf16 and can quantize it row-wise on the way out.
// Every mbarrier wait is bounded (about 2 s): on expiry the CTA sets the
// library's device error word, stops issuing work, and still frees its tensor
// memory before exiting.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace mx {
namespace {
__device__ uint32_t g_gemm_error;
}  // namespace
}  // namespace mx
#define MX_BOUNDS_FAIL() atomicExch(&::mx::g_gemm_error, ::mx::kErrBounds)

#include "quant_device.cuh"
#include "tma_host.h"

namespace mx {
namespace {

constexpr int BM = 128, BN = 256, BK = 256;
constexpr int BKB = BK / 2;                    // bytes of packed codes per row per stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BKB;              // 16 KB
constexpr int B_BYTES = BN * BKB;              // 32 KB
constexpr int SFA_BYTES = BM * (BK / 32);      // 1 KB: two 512-byte scale tiles
constexpr int SFB_BYTES = BN * (BK / 32);      // 2 KB: four 512-byte scale tiles
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 64 + NUM_EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;                // 256 fp32 columns
constexpr uint32_t SFA_COL = 256;              // 2 k-chunks x 4 columns
constexpr uint32_t SFB_COL = 264;              // 2 k-chunks x 8 columns
constexpr int CTL_BYTES = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + CTL_BYTES + 1024;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// Tile raster: a group of G consecutive M-tiles sweeps all N-tiles before the
// next group starts, so a group's A rows (G * 128 * K/2 bytes) stay in L2 while
// B streams through once per group. G is chosen on the host so that this
// footprint is about 24 MB (measured on the 70B-layer GEMMs against 12, 48 and
// 96 MB: 0.5-2 % faster than 48 MB on each).
constexpr int64_t kGroupBytes = 24ll << 20;

static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle alignment");

// Barriers and flags of one CTA; S = pipeline depth of the kernel using it.
template <int S>
struct CtlT {
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
};
using Ctl = CtlT<STAGES>;
static_assert(sizeof(Ctl) <= CTL_BYTES, "control block");

// Instruction descriptor, kind::mxf4 block-scaled: E2M1 A and B (format 1 at
// bits 7-9 and 10-12), both K-major, N >> 3 at bits 17-22, E8M0 scales (bit
// 23), M >> 4 at bits 24-28, scale-factor byte selectors for B (bits 4-5) and
// A (bits 29-30).
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id) {
  return (sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) |
         ((uint32_t)(BM >> 4) << 24) | (sf_id << 29);
}

// Bounded wait; after kWaitLimitNs in total the CTA aborts. With `sleep` each
// try_wait may suspend the thread until the phase completes (used by the
// epilogue, whose waits are off the critical path); the producer and MMA
// threads poll, which wakes them with the least latency.
template <int S>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, CtlT<S>* ctl,
                                         bool sleep = false) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (sleep ? ptx::mbar_try_wait_sleep(bar, parity, 200000u) : ptx::mbar_try_wait(bar, parity))
      return true;
    if (sleep || (i & 63u) == 0) {
      if (*reinterpret_cast<volatile uint32_t*>(&ctl->abort)) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
        *reinterpret_cast<volatile uint32_t*>(&ctl->abort) = 1u;
        atomicExch(&g_gemm_error, 6u);  // MXFP4_ERR_TIMEOUT
        return false;
      }
    }
  }
}

// Bounded wait used only while shutting down after an abort.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs / 8) return;
}

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group_m, int& mb,
                                            int& nb) {
  const int per_group = group_m * num_n;
  const int g = tile / per_group;
  const int first_m = g * group_m;
  const int gm = min(group_m, num_m - first_m);
  const int w = tile - g * per_group;
  mb = first_m + w % gm;
  nb = w / gm;
}

// Two fp32 bit patterns to a bf16 pair (nearest-even), lo in the low half.
__device__ __forceinline__ uint32_t bf16x2(uint32_t lo, uint32_t hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Lanes 2i and 2i + 1 of a warp hold rows r and r + 1 (r even). For one
// 32-byte segment of both rows (byte offset seg of each row), lo and hi are
// this lane's two 16-byte halves of its own row's segment. The pair swaps
// halves (the even lane passes its row's upper half, the odd lane its lower
// half) so that each of the two stores writes a whole 32-byte sector of one
// row: first row r (even lane bytes 0-15, odd lane 16-31), then row r + 1.
// A warp store then fills 16 sectors instead of half-filling 32.
// (cbase, cbytes: C's extent, checked in bounds-checking builds.)
__device__ __forceinline__ void store_row_pair(uint8_t* rowa, uint8_t* rowb, int64_t seg, uint4 lo,
                                               uint4 hi, int odd, const void* cbase, uint64_t cbytes) {
  uint4 g;
  g.x = __shfl_xor_sync(0xffffffffu, odd ? lo.x : hi.x, 1);
  g.y = __shfl_xor_sync(0xffffffffu, odd ? lo.y : hi.y, 1);
  g.z = __shfl_xor_sync(0xffffffffu, odd ? lo.z : hi.z, 1);
  g.w = __shfl_xor_sync(0xffffffffu, odd ? lo.w : hi.w, 1);
  put(reinterpret_cast<uint4*>(rowa + seg + 16 * odd), odd ? g : lo, cbase, cbytes);
  put(reinterpret_cast<uint4*>(rowb + seg + 16 * odd), odd ? hi : g, cbase, cbytes);
}

// One epilogue thread's results: 128 consecutive fp32 values of row `row`
// (columns c0 .. c0 + 127); lane l of the warp holds row r + l of the warp's
// 32 rows (r a multiple of 32). They are stored to C when C is given (fp32,
// or bf16 rounded to nearest-even when c_bf16; adjacent lanes pair up so that
// every store fills whole sectors), and with kQ (and a row-wise output
// requested) they are also quantized row-wise (four 32-runs) from the fp32
// values, exactly as the quantizer would quantize that row of an fp32 C. All
// 32 lanes of the warp take part.
template <bool kQ>
__device__ __forceinline__ void epilogue_out(const uint32_t (&r0)[64], const uint32_t (&r1)[64],
                                             void* C, int c_bf16, int64_t ldc, int64_t row,
                                             int64_t c0, int64_t N, const OrientArgs& qo,
                                             uint64_t c_bytes) {
  if (!kQ || C != nullptr) {
    const int odd = threadIdx.x & 1;
    const int64_t esz = c_bf16 ? 2 : 4;
    uint8_t* rowa = reinterpret_cast<uint8_t*>(C) + ((row - odd) * ldc + c0) * esz;
    uint8_t* rowb = rowa + ldc * esz;
    if (c_bf16) {
      // 16 bf16 values (32 bytes) per segment: columns 16 m .. 16 m + 15.
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint32_t* r = m < 4 ? r0 : r1;
        const int o = (m & 3) * 16;
        const uint4 lo = make_uint4(bf16x2(r[o], r[o + 1]), bf16x2(r[o + 2], r[o + 3]),
                                    bf16x2(r[o + 4], r[o + 5]), bf16x2(r[o + 6], r[o + 7]));
        const uint4 hi = make_uint4(bf16x2(r[o + 8], r[o + 9]), bf16x2(r[o + 10], r[o + 11]),
                                    bf16x2(r[o + 12], r[o + 13]), bf16x2(r[o + 14], r[o + 15]));
        store_row_pair(rowa, rowb, 32 * m, lo, hi, odd, C, c_bytes);
      }
    } else {
      // 8 fp32 values (32 bytes) per segment: columns 8 m .. 8 m + 7.
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const uint32_t* r = m < 8 ? r0 : r1;
        const int o = (m & 7) * 8;
        store_row_pair(rowa, rowb, 32 * m, make_uint4(r[o], r[o + 1], r[o + 2], r[o + 3]),
                       make_uint4(r[o + 4], r[o + 5], r[o + 6], r[o + 7]), odd, C, c_bytes);
      }
    }
  }
  if (kQ && qo.q != nullptr) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float2 R[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int i = (b & 1) * 32 + 2 * k;
        R[k] = b < 2 ? make_float2(__uint_as_float(r0[i]), __uint_as_float(r0[i + 1]))
                     : make_float2(__uint_as_float(r1[i]), __uint_as_float(r1[i + 1]));
      }
      quantize_run32(R, row, c0 + 32 * b, N, qo);
    }
  }
}

// Column-wise quantization of one 32 x 32 chunk of an epilogue warp's block of
// C (rows row0 .. row0 + 31, lane l holding row row0 + l and, in v, its
// values at columns n0 .. n0 + 31): the quantization of C^T along M, whose
// output row n is column n of C and whose 32-runs run along m. The chunk goes
// through the warp's shared buffers -- the values (tb, 32 x 33 floats) and,
// for stochastic rounding, the draws keyed by source index m * N + n (db,
// 32 x 17 words, a row's 32 16-bit draws packed as the quantizer packs them)
// -- so that lane l then holds column n0 + l; that run is quantized as the
// quantizer's column pass does (rotation, block max over the 32 lanes for
// 32x32 blocks, scale, rounding, packing) and stored at q[n0 + l, row0 / 2 ..].
__device__ __forceinline__ void col_chunk(const float2 (&v)[16], float* tb, uint32_t* db, int lane,
                                          int64_t row0, int64_t n0, int64_t M, int64_t N,
                                          const OrientArgs& qc) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    tb[lane * 33 + 2 * k] = v[k].x;
    tb[lane * 33 + 2 * k + 1] = v[k].y;
  }
  if (qc.sr) {
    uint32_t w[16];
    draws32(qc.keys, qc.stream, (uint64_t)((row0 + lane) * N + n0), w);
#pragma unroll
    for (int k = 0; k < 16; ++k) db[lane * 17 + k] = w[k];
  }
  __syncwarp();
  float2 R[16];
#pragma unroll
  for (int k = 0; k < 16; ++k)
    R[k] = make_float2(tb[(2 * k) * 33 + lane], tb[(2 * k + 1) * 33 + lane]);
  uint32_t w[16];
  if (qc.sr) {
    const int sh = 16 * (lane & 1);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t d0 = (db[(2 * k) * 17 + (lane >> 1)] >> sh) & 0xFFFFu;
      const uint32_t d1 = (db[(2 * k + 1) * 17 + (lane >> 1)] >> sh) & 0xFFFFu;
      w[k] = d0 | (d1 << 16);
    }
  }
  __syncwarp();   // the buffers are rewritten by the next chunk
  const int64_t n = n0 + lane;
  if (qc.wht) hadamard32_lane(R, qc.sign_mask, qc.sgn);
  float Mx = absmax32(R);
  if (qc.block) Mx = warp_max(Mx);
  const int e = scale_run32<true, false>(R, qc, Mx, w);
  store_run32(qc, n, row0, M, R);
  store_run_scales<false>(qc, n, row0, M, e);
}

// The epilogue with both orientations: C stored as in epilogue_out, then per
// 32-column chunk the row-wise run (if qo.q) and the column-wise chunk (if
// qc.q), so each chunk's registers die as the loop moves on.
__device__ __forceinline__ void epilogue_rowcol(const uint32_t (&r0)[64], const uint32_t (&r1)[64],
                                                void* C, int c_bf16, int64_t ldc, int64_t row,
                                                int64_t c0, int64_t M, int64_t N,
                                                const OrientArgs& qo, const OrientArgs& qc,
                                                float* tb, uint32_t* db, int lane, uint64_t c_bytes) {
  if (C != nullptr) {
    const OrientArgs none{};
    epilogue_out<false>(r0, r1, C, c_bf16, ldc, row, c0, N, none, c_bytes);
  }
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    float2 v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int i = (b & 1) * 32 + 2 * k;
      v[k] = b < 2 ? make_float2(__uint_as_float(r0[i]), __uint_as_float(r0[i + 1]))
                   : make_float2(__uint_as_float(r1[i]), __uint_as_float(r1[i + 1]));
    }
    if (qo.q != nullptr) {
      float2 R[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) R[k] = v[k];
      quantize_run32(R, row, c0 + 32 * b, N, qo);
    }
    if (qc.q != nullptr) col_chunk(v, tb, db, lane, row - lane, c0 + 32 * b, M, N, qc);
  }
}

template <bool kQ>
__global__ void __launch_bounds__(THREADS, 1)
mxf4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const uint8_t* __restrict__ sa, const uint8_t* __restrict__ sb,
                 void* __restrict__ C, int c_bf16, int64_t ldc, int M, int N, int K, int group_m,
                 const __grid_constant__ OrientArgs qo) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // N and K are multiples of 128: the last N tile may hold only 128 valid
  // columns (B rows past N arrive zero-filled, their scales are not loaded and
  // those columns are not stored) and the last K step only 128 valid K (its
  // second half of the codes arrives zero-filled, its scale tiles are not
  // loaded and its last two MMAs are not issued).
  const int num_m = M / BM, num_n = (N + BN - 1) / BN, num_k = (K + BK - 1) / BK;
  const int num_tiles = num_m * num_n;
  const int64_t ktiles = K / 128;  // 512-byte scale tiles per 128-row band
  const int64_t nbands = N / 128;  // 128-row bands of B
  const bool k_half = (K % BK) != 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&ctl->full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&ctl->empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&ctl->acc_full), 1);
    ptx::mbar_init(ptx::smem_u32(&ctl->acc_empty), NUM_EPI_WARPS);
    ptx::mbar_init(ptx::smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // per-stage bit masks of the last issue
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, num_m, num_n, group_m, mb, nb);
        for (int kb = 0; kb < num_k; ++kb) {
          const uint32_t empty = ptx::smem_u32(&ctl->empty[stage]);
          const uint32_t full = ptx::smem_u32(&ctl->full[stage]);
          if (!(ok = wait_bar(empty, phase ^ 1u, ctl))) break;
          const uint32_t st = ptx::smem_u32(smem + stage * STAGE_BYTES);
          // A half K step (the last one when K % 256 == 128) takes one scale
          // tile per band; a half N tile one band of B scales.
          const uint32_t sf_bytes = (k_half && kb == num_k - 1) ? 512u : 1024u;
          const int b_bands = 2 * nb + 1 < nbands ? 2 : 1;
          ptx::mbar_arrive_expect_tx(full, A_BYTES + B_BYTES + sf_bytes * (1 + b_bands));
          ptx::tma_load_2d(st, &tmA, kb * BKB, mb * BM, full);
          ptx::tma_load_2d(st + A_BYTES, &tmB, kb * BKB, nb * BN, full);
          ptx::bulk_load(st + A_BYTES + B_BYTES, sa + ((int64_t)mb * ktiles + 2 * kb) * 512,
                         sf_bytes, full);
          for (int t = 0; t < b_bands; ++t)
            ptx::bulk_load(st + A_BYTES + B_BYTES + SFA_BYTES + t * 1024,
                           sb + ((int64_t)(2 * nb + t) * ktiles + 2 * kb) * 512, sf_bytes, full);
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // After an abort, wait (bounded) for the last load issued into each
      // stage to land before the CTA's shared memory is released.
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
          if ((issued >> s) & 1u) drain_wait(ptx::smem_u32(&ctl->full[s]), (issued_parity >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        if (!(ok = wait_bar(ptx::smem_u32(&ctl->acc_empty), acc_phase ^ 1u, ctl))) break;
        ptx::tc_fence_after();
        // One K step with kMmas MMAs of K = 64: four, or two for a last,
        // 128-deep step. The full steps run in a loop of their own and the
        // half step after it, so the hot loop has no branch between MMAs
        // (one there measurably slows the issue).
        auto kstep = [&](int kb, auto nmma) -> bool {
          [[maybe_unused]] constexpr int kMmas = decltype(nmma)::value;
          if (!(ok = wait_bar(ptx::smem_u32(&ctl->full[stage]), phase, ctl))) return false;
          ptx::tc_fence_after();
          const uint32_t st = ptx::smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sfa_s = st + A_BYTES + B_BYTES;
          const uint32_t sfb_s = sfa_s + SFA_BYTES;
          // Scales to tensor memory: each 512-byte tile (128 rows x 4 scale
          // columns) fills 4 columns; row r's scales land in column r / 32.
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            ptx::tc_cp_32x128b_warpx4(tmem + SFA_COL + 4 * c,
                                      ptx::smem_desc(sfa_s + c * 512, 0, 128, 0));
#pragma unroll
            for (int t = 0; t < 2; ++t)
              ptx::tc_cp_32x128b_warpx4(tmem + SFB_COL + 8 * c + 4 * t,
                                        ptx::smem_desc(sfb_s + t * 1024 + c * 512, 0, 128, 0));
          }
#pragma unroll
          for (int k = 0; k < kMmas; ++k) {
            const uint64_t ad = ptx::smem_desc(st + k * 32, 16, 1024, 2);
            const uint64_t bd = ptx::smem_desc(st + A_BYTES + k * 32, 16, 1024, 2);
            ptx::mma_mxf4(tmem + ACC_COL, ad, bd, make_idesc((k & 1) * 2),
                          tmem + SFA_COL + 4 * (k >> 1), tmem + SFB_COL + 8 * (k >> 1),
                          (kb | k) != 0);
          }
          ptx::tc_commit(ptx::smem_u32(&ctl->empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          return true;
        };
        const int num_kf = k_half ? num_k - 1 : num_k;
        for (int kb = 0; kb < num_kf; ++kb)
          if (!kstep(kb, std::integral_constant<int, 4>{})) break;
        if (ok && k_half) kstep(num_kf, std::integral_constant<int, 2>{});
        if (!ok) break;
        ptx::tc_commit(ptx::smem_u32(&ctl->acc_full));
        acc_phase ^= 1u;
      }
      // No MMA may still be reading shared or tensor memory at teardown.
      ptx::tc_commit(ptx::smem_u32(&ctl->drain));
      drain_wait(ptx::smem_u32(&ctl->drain), 0);
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;            // tensor-memory lane quarter this warp may access
    const int h = (warp - 2) >> 2;     // column half of the 256-wide tile
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int mb, nb;
      tile_coords(tile, num_m, num_n, group_m, mb, nb);
      // One lane waits; its result is broadcast so the warp stays converged
      // for the .sync.aligned tensor-memory loads.
      int ok = 0;
      if (lane == 0) ok = wait_bar(ptx::smem_u32(&ctl->acc_full), acc_phase, ctl, true);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      ptx::tc_fence_after();
      uint32_t r0[64], r1[64];
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + ACC_COL + h * 128;
      ptx::tmem_ld_32x32b_x64(taddr, r0);
      ptx::tmem_ld_32x32b_x64(taddr + 64, r1);
      ptx::tc_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&ctl->acc_empty));
      acc_phase ^= 1u;
      const int64_t row = (int64_t)mb * BM + q * 32 + lane;
      const int64_t col0 = (int64_t)nb * BN + h * 128;
      if (col0 < N)
        epilogue_out<kQ>(r0, r1, C, c_bf16, ldc, row, col0, N, qo,
                         ((uint64_t)(M - 1) * ldc + N) * (c_bf16 ? 2u : 4u));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ============================================================ CTA pairs ===
// The same GEMM on CTA pairs (a cluster of 2, tcgen05 cta_group::2): a pair
// computes a 256 x 256 output tile. CTA r loads rows 128 r .. of the pair's A
// rows and rows 128 r .. of its B rows, so each SM stages 128 + 128 rows per
// K-step instead of 128 + 256; the leader (rank 0) issues M = 256 MMAs that
// read both CTAs' shared memory, and each CTA's tensor memory receives its
// 128 x 256 fp32 accumulator. Scales: each CTA stages its own 128 rows of A
// scales and all 256 rows of B scales (tensor-memory columns as in the 1-CTA
// kernel); the leader copies them to tensor memory with tcgen05.cp.cta_group::2.
// All loads of a stage (both CTAs) are counted on the leader's full barrier;
// the leader's commits are multicast to both CTAs' empty / accumulator-full
// barriers; both CTAs' epilogues arrive on the leader's accumulator-empty
// barrier.
namespace pair {
constexpr int BM = 128;                        // rows of A per CTA
constexpr int BNP = 256;                       // N of the pair tile
constexpr int BNH = 128;                       // rows of B per CTA
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BKB;              // 16 KB
constexpr int B_BYTES = BNH * BKB;             // 16 KB
constexpr int SFA_BYTES = BM * (BK / 32);      // 1 KB
constexpr int SFB_BYTES = BNP * (BK / 32);     // 2 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr uint32_t TX_BYTES = 2 * STAGE_BYTES; // both CTAs' loads land on the leader's barrier
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + CTL_BYTES + 1024;
static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle alignment");
using Ctl = CtlT<STAGES>;
static_assert(sizeof(Ctl) <= CTL_BYTES, "control block");
// NVFP4 stages: the same codes plus four scale tiles of A and eight of B.
constexpr int NV_STAGES = 5;
constexpr int NV_STAGE_BYTES = A_BYTES + B_BYTES + 4 * 512 + 8 * 512;   // 38 KB
constexpr int NV_SMEM_BYTES = NV_STAGES * NV_STAGE_BYTES + CTL_BYTES + 1024;
constexpr uint32_t SFB_COL_NV = SFA_COL + 16;   // A: 4 tiles x 4 columns, B: 4 x 8
static_assert(NV_STAGE_BYTES % 1024 == 0 && NV_STAGES <= STAGES, "NVFP4 ring");
static_assert(SFB_COL_NV + 32 <= TMEM_COLS, "NVFP4 scale columns");
enum : int { kMxf4 = 0, kMxf8 = 1, kNvf4 = 2, kMxf8e5 = 3 };
// Column-wise epilogue quantization: per epilogue warp a 32 x 33 fp32 value
// buffer and a 32 x 17 word draw buffer, after five stages.
constexpr int QC_STAGES = 5;
constexpr int kXposeBytes = 32 * 33 * 4 + 32 * 17 * 4;     // 6400
constexpr int QC_SMEM_BYTES = QC_STAGES * STAGE_BYTES + CTL_BYTES + NUM_EPI_WARPS * kXposeBytes + 1024;
static_assert(QC_SMEM_BYTES <= 227 * 1024, "column-wise epilogue buffers");
// Scale-image variants (kImg): the scales arrive as 4 KB images built by
// scale_images_kernel -- two 512-byte tiles, interleaved by 8-row group and
// replicated four times -- and each image goes to tensor memory with one
// 128x256b copy (8 columns, the same layout the 32x128b.warpx4 copies of two
// tiles give). MXFP4: one image of A and two of B per stage (three copies
// instead of six), five 44 KB stages; NVFP4: two of A and four of B (six
// instead of twelve), four 56 KB stages.
constexpr int IMG_BYTES = 4096;
constexpr int MXI_STAGES = 5;
constexpr int MXI_STAGE_BYTES = A_BYTES + B_BYTES + 3 * IMG_BYTES;
constexpr int MXI_SMEM_BYTES = MXI_STAGES * MXI_STAGE_BYTES + CTL_BYTES + 1024;
constexpr int NVI_STAGES = 4;
constexpr int NVI_STAGE_BYTES = A_BYTES + B_BYTES + 6 * IMG_BYTES;
constexpr int NVI_SMEM_BYTES = NVI_STAGES * NVI_STAGE_BYTES + CTL_BYTES + 1024;
static_assert(MXI_SMEM_BYTES <= 227 * 1024 && NVI_SMEM_BYTES <= 227 * 1024, "image stages");
static_assert(MXI_STAGE_BYTES % 1024 == 0 && NVI_STAGE_BYTES % 1024 == 0, "image stage alignment");
static_assert(NVI_STAGES <= STAGES && MXI_STAGES <= STAGES, "control block depth");

// kind::mxf4nvf4 with E2M1 A and B (type code 1), K-major, UE4M3 scales (bit
// 23 clear), scale_vec::4X (both scale-factor selectors 0).
__device__ __forceinline__ uint32_t make_idesc_nv() {
  return (1u << 7) | (1u << 10) | ((uint32_t)(BNP >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
}

// kF8: kind::mxf8f6f4 with E4M3 operands (type code 0), or E5M2 operands
// (type code 1) with kE5, instead of kind::mxf4's E2M1 (type code 1).
template <bool kF8 = false, bool kE5 = false>
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id) {
  const uint32_t t = kF8 ? (kE5 ? 1u : 0u) : 1u;
  return (sf_id << 4) | (t << 7) | (t << 10) | ((uint32_t)(BNP >> 3) << 17) | (1u << 23) |
         ((uint32_t)(256 >> 4) << 24) | (sf_id << 29);
}

// kKind selects the operand format:
//  kMxf4: E2M1 codes with E8M0 scales per 32 (kind::mxf4, scale_vec::2X): a
//    stage row is 256 elements of K, two 512-byte scale tiles of A and two per
//    128-row band of B; MMA k reads bytes 2 (k % 2) .. of each row's word;
//  kMxf8: E4M3 codes, one byte per element, so a 128-byte stage row is 128
//    elements of K (4 MMAs of K = 32), with one 512-byte scale tile of A and
//    one per 128-row band of B per stage; MMA k reads byte k of the word;
//  kNvf4: E2M1 codes with E4M3 scales per 16 (kind::mxf4nvf4, scale_vec::4X):
//    each 512-byte scale tile covers one MMA's K = 64, so a stage brings four
//    tiles of A and four per band of B (twelve scale copies), and each MMA
//    reads a whole word; the fp32 sums are multiplied by alpha (the operands'
//    power-of-two tensor factors) in the epilogue. Five stages of 38 KB.
//
// kQ: 0 plain; 1 C also quantized row-wise (qo); 2 row-wise (qo, if qo.q) and
// column-wise (qc) -- five stages, the rest of shared memory holding each
// epilogue warp's transposition buffers (kXposeBytes).
template <int kQ, int kKind = kMxf4, bool kImg = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
mxf4_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                      void* __restrict__ C, int c_bf16, int64_t ldc, int M, int N, int K, int group_m,
                      float alpha, const __grid_constant__ OrientArgs qo,
                      const __grid_constant__ OrientArgs qc) {
  constexpr bool kF8 = kKind == kMxf8 || kKind == kMxf8e5, kNv = kKind == kNvf4;
  static_assert(!kImg || (kQ != 2 && !kF8), "scale images serve the MXFP4 / NVFP4 GEMMs "
                                             "without the column-wise epilogue");
  constexpr int kAImgs = kNv ? 2 : 1, kBImgs = kNv ? 4 : 2;   // images per stage
  constexpr int kStages = kImg ? (kNv ? NVI_STAGES : MXI_STAGES)
                               : (kNv ? NV_STAGES : (kQ == 2 ? QC_STAGES : STAGES));
  constexpr int kStageBytes = kImg ? (kNv ? NVI_STAGE_BYTES : MXI_STAGE_BYTES)
                                   : (kNv ? NV_STAGE_BYTES : STAGE_BYTES);
  constexpr int kSfaBytes = kImg ? kAImgs * IMG_BYTES : (kNv ? 4 * 512 : SFA_BYTES);
  constexpr uint32_t kSfbCol = kNv ? SFB_COL_NV : SFB_COL;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  // M, N and K are multiples of 128: a last M tile with 128 valid rows (CTA
  // 1's A rows and scales arrive zero-filled and its epilogue stores nothing),
  // a last N tile with 128 valid columns (CTA 1's B rows and scale band arrive
  // zero-filled; those columns are not stored) and, for E2M1 operands, a last
  // K step with 128 valid K (the rest arrives zero-filled and its last two
  // MMAs are not issued; an FP8 K step is 128 deep).
  const int num_m = (M + 2 * BM - 1) / (2 * BM), num_n = (N + BNP - 1) / BNP;
  const int num_k = kF8 ? K / (BK / 2) : (K + BK - 1) / BK;
  const bool k_half = !kF8 && (K % BK) != 0;
  const int num_tiles = num_m * num_n;
  const int pair_id = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
  constexpr uint32_t kTx = kF8 ? 2u * (A_BYTES + B_BYTES + 512 + 1024)
                               : ((kNv || kImg) ? 2u * kStageBytes : TX_BYTES);
  // 512-byte scale tiles per 128-row band (image path): K/128, or K/64 for NVFP4
  const int ntiles = kNv ? K / 64 : K / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&ctl->full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&ctl->empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&ctl->acc_full), 1);
    ptx::mbar_init(ptx::smem_u32(&ctl->acc_empty), 2 * NUM_EPI_WARPS);
    ptx::mbar_init(ptx::smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB);
    ptx::prefetch_tensormap(&tmSA);
    ptx::prefetch_tensormap(&tmSB);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&ctl->tmem_base), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();        // both CTAs' barriers initialised before any remote signal
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued_rounds = 0;
      bool ok = true;
      for (int tile = pair_id; ok && tile < num_tiles; tile += num_pairs) {
        int mb, nb;
        tile_coords(tile, num_m, num_n, group_m, mb, nb);
        const int a_row = mb * 2 * BM + (int)rank * BM;
        const int b_row = nb * BNP + (int)rank * BNH;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!(ok = wait_bar(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, ctl))) break;
          const uint32_t full_local = ptx::smem_u32(&ctl->full[stage]);
          const uint32_t full_leader = ptx::mapa(full_local, 0);
          if (leader) ptx::mbar_arrive_expect_tx(full_local, kTx);
          const uint32_t st = ptx::smem_u32(smem + stage * kStageBytes);
          const int kt = kF8 ? kb : (kNv ? 4 * kb : 2 * kb);   // first scale tile of the stage
          ptx::tma_load_2d_pair(st, &tmA, kb * BKB, a_row, full_leader);
          ptx::tma_load_2d_pair(st + A_BYTES, &tmB, kb * BKB, b_row, full_leader);
          if constexpr (kImg) {
            // A images: band * ceil(ntiles / 2) + tile pair; B images: band pair *
            // ntiles + tile.
            ptx::tma_load_3d_pair(st + A_BYTES + B_BYTES, &tmSA, 0, 0,
                                  (a_row / 128) * ((ntiles + 1) / 2) + kAImgs * kb, full_leader);
            ptx::tma_load_3d_pair(st + A_BYTES + B_BYTES + kSfaBytes, &tmSB, 0, 0,
                                  nb * ntiles + kBImgs * kb, full_leader);
          } else {
            ptx::tma_load_3d_pair(st + A_BYTES + B_BYTES, &tmSA, 0, kt, a_row / 128, full_leader);
            ptx::tma_load_3d_pair(st + A_BYTES + B_BYTES + kSfaBytes, &tmSB, 0, kt, nb * 2,
                                  full_leader);
          }
          ++issued_rounds;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Wait until the leader's commits have released every stage this CTA
      // filled, so no remote arrive targets this CTA after it exits.
      for (int s = 0; s < kStages; ++s) {
        const uint32_t n = issued_rounds / kStages + ((uint32_t)s < issued_rounds % kStages ? 1u : 0u);
        if (n) drain_wait(ptx::smem_u32(&ctl->empty[s]), (n - 1) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (leader && lane == 0) {
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = pair_id; ok && tile < num_tiles; tile += num_pairs) {
        const int num_kf = k_half ? num_k - 1 : num_k;
        // With scale images, the first K step's copies go to tensor memory
        // before the accumulator is free: they write only the scale columns,
        // which the previous tile's MMAs (issued earlier by this thread, so
        // executed first) have finished reading, and so overlap the epilogue's
        // drain instead of delaying the first MMA.
        int kb_begin = 0;
        if constexpr (kImg && kKind == kMxf4) {
          if (!(ok = wait_bar(ptx::smem_u32(&ctl->full[stage]), phase, ctl))) break;
          ptx::tc_fence_after();
          const uint32_t st = ptx::smem_u32(smem + stage * kStageBytes);
          const uint32_t sfa_s = st + A_BYTES + B_BYTES;
          ptx::tc_cp_pair_128x256b(tmem + SFA_COL, ptx::smem_desc(sfa_s, 128, 256, 0));
#pragma unroll
          for (int i = 0; i < 2; ++i)
            ptx::tc_cp_pair_128x256b(tmem + kSfbCol + 8 * i,
                                     ptx::smem_desc(sfa_s + IMG_BYTES + i * IMG_BYTES, 128, 256, 0));
          if (!(ok = wait_bar(ptx::smem_u32(&ctl->acc_empty), acc_phase ^ 1u, ctl))) break;
          ptx::tc_fence_after();
          auto mma0 = [&](int k) {
            const uint64_t ad = ptx::smem_desc(st + k * 32, 16, 1024, 2);
            const uint64_t bd = ptx::smem_desc(st + A_BYTES + k * 32, 16, 1024, 2);
            ptx::mma_mxf4_pair(tmem + ACC_COL, ad, bd, make_idesc((k & 1) * 2),
                               tmem + SFA_COL + 4 * (k >> 1), tmem + SFB_COL + 8 * (k >> 1), k != 0);
          };
          if (num_kf > 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) mma0(k);
          } else {
#pragma unroll
            for (int k = 0; k < 2; ++k) mma0(k);
          }
          ptx::tc_commit_pair_multicast(ptx::smem_u32(&ctl->empty[stage]), 0x3);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          kb_begin = 1;
        } else {
          if (!(ok = wait_bar(ptx::smem_u32(&ctl->acc_empty), acc_phase ^ 1u, ctl))) break;
          ptx::tc_fence_after();
        }
        // One K step; kMmas (MXFP4 only) is four, or two for a last, 128-deep
        // step. The full steps run in a loop of their own and the half step
        // after it, so the hot loop has no branch between MMAs (one there
        // measurably slows the issue).
        auto kstep = [&](int kb, auto nmma) -> bool {
          [[maybe_unused]] constexpr int kMmas = decltype(nmma)::value;
          if (!(ok = wait_bar(ptx::smem_u32(&ctl->full[stage]), phase, ctl))) return false;
          ptx::tc_fence_after();
          const uint32_t st = ptx::smem_u32(smem + stage * kStageBytes);
          const uint32_t sfa_s = st + A_BYTES + B_BYTES;
          const uint32_t sfb_s = sfa_s + kSfaBytes;
          if constexpr (kImg) {
            // A image i (tiles 2i, 2i + 1) to SFA_COL + 8 i; B image i (both
            // bands of tile i) to the B columns + 8 i: the columns the narrow
            // copies below would fill.
#pragma unroll
            for (int i = 0; i < kAImgs; ++i)
              ptx::tc_cp_pair_128x256b(tmem + SFA_COL + 8 * i,
                                       ptx::smem_desc(sfa_s + i * IMG_BYTES, 128, 256, 0));
#pragma unroll
            for (int i = 0; i < kBImgs; ++i)
              ptx::tc_cp_pair_128x256b(tmem + kSfbCol + 8 * i,
                                       ptx::smem_desc(sfb_s + i * IMG_BYTES, 128, 256, 0));
          }
          if constexpr (kNv) {
            // Four K tiles, one per MMA: A's tile k to SFA_COL + 4 k, B's band t
            // of tile k to kSfbCol + 8 k + 4 t; each MMA reads whole words.
#pragma unroll
            for (int k = 0; k < kMmas && !kImg; ++k) {
              ptx::tc_cp_pair_32x128b_warpx4(tmem + SFA_COL + 4 * k,
                                             ptx::smem_desc(sfa_s + k * 512, 0, 128, 0));
#pragma unroll
              for (int t = 0; t < 2; ++t)
                ptx::tc_cp_pair_32x128b_warpx4(tmem + kSfbCol + 8 * k + 4 * t,
                                               ptx::smem_desc(sfb_s + t * 2048 + k * 512, 0, 128, 0));
            }
#pragma unroll
            for (int k = 0; k < kMmas; ++k) {
              const uint64_t ad = ptx::smem_desc(st + k * 32, 16, 1024, 2);
              const uint64_t bd = ptx::smem_desc(st + A_BYTES + k * 32, 16, 1024, 2);
              ptx::mma_nvf4_pair(tmem + ACC_COL, ad, bd, make_idesc_nv(), tmem + SFA_COL + 4 * k,
                                 tmem + kSfbCol + 8 * k, (kb | k) != 0);
            }
          } else if constexpr (kF8) {
            // One K tile: A's tile to SFA_COL, B's bands to SFB_COL + 4 t; MMA k
            // reads byte k of each row's word.
            ptx::tc_cp_pair_32x128b_warpx4(tmem + SFA_COL, ptx::smem_desc(sfa_s, 0, 128, 0));
#pragma unroll
            for (int t = 0; t < 2; ++t)
              ptx::tc_cp_pair_32x128b_warpx4(tmem + SFB_COL + 4 * t,
                                             ptx::smem_desc(sfb_s + t * 512, 0, 128, 0));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = ptx::smem_desc(st + k * 32, 16, 1024, 2);
              const uint64_t bd = ptx::smem_desc(st + A_BYTES + k * 32, 16, 1024, 2);
              ptx::mma_mxf8_pair(tmem + ACC_COL, ad, bd, make_idesc<true, kKind == kMxf8e5>(k), tmem + SFA_COL,
                                 tmem + SFB_COL, (kb | k) != 0);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 2 && !kImg; ++c) {
              ptx::tc_cp_pair_32x128b_warpx4(tmem + SFA_COL + 4 * c,
                                             ptx::smem_desc(sfa_s + c * 512, 0, 128, 0));
#pragma unroll
              for (int t = 0; t < 2; ++t)
                ptx::tc_cp_pair_32x128b_warpx4(tmem + SFB_COL + 8 * c + 4 * t,
                                               ptx::smem_desc(sfb_s + t * 1024 + c * 512, 0, 128, 0));
            }
#pragma unroll
            for (int k = 0; k < kMmas; ++k) {
              const uint64_t ad = ptx::smem_desc(st + k * 32, 16, 1024, 2);
              const uint64_t bd = ptx::smem_desc(st + A_BYTES + k * 32, 16, 1024, 2);
              ptx::mma_mxf4_pair(tmem + ACC_COL, ad, bd, make_idesc((k & 1) * 2),
                                 tmem + SFA_COL + 4 * (k >> 1), tmem + SFB_COL + 8 * (k >> 1),
                                 (kb | k) != 0);
            }
          }
          ptx::tc_commit_pair_multicast(ptx::smem_u32(&ctl->empty[stage]), 0x3);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          return true;
        };
        for (int kb = kb_begin; kb < num_kf; ++kb)
          if (!kstep(kb, std::integral_constant<int, 4>{})) break;
        if (ok && k_half && num_kf >= kb_begin) kstep(num_kf, std::integral_constant<int, 2>{});
        if (!ok) break;
        ptx::tc_commit_pair_multicast(ptx::smem_u32(&ctl->acc_full), 0x3);
        acc_phase ^= 1u;
      }
      ptx::tc_commit_pair_multicast(ptx::smem_u32(&ctl->drain), 0x1);
      drain_wait(ptx::smem_u32(&ctl->drain), 0);
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const uint32_t acc_empty_leader = ptx::mapa(ptx::smem_u32(&ctl->acc_empty), 0);
    uint32_t acc_phase = 0;
    for (int tile = pair_id; tile < num_tiles; tile += num_pairs) {
      int mb, nb;
      tile_coords(tile, num_m, num_n, group_m, mb, nb);
      int ok = 0;
      if (lane == 0) ok = wait_bar(ptx::smem_u32(&ctl->acc_full), acc_phase, ctl, true);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      ptx::tc_fence_after();
      uint32_t r0[64], r1[64];
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + ACC_COL + h * 128;
      ptx::tmem_ld_32x32b_x64(taddr, r0);
      ptx::tmem_ld_32x32b_x64(taddr + 64, r1);
      ptx::tc_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(acc_empty_leader);
      acc_phase ^= 1u;
      if ((int64_t)mb * 2 * BM + rank * BM >= M) continue;   // the empty half of a last M tile
      const int64_t row = (int64_t)mb * 2 * BM + rank * BM + q * 32 + lane;
      if constexpr (kNv) {   // exact: alpha is a power of two
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          r0[i] = __float_as_uint(__fmul_rn(__uint_as_float(r0[i]), alpha));
          r1[i] = __float_as_uint(__fmul_rn(__uint_as_float(r1[i]), alpha));
        }
      }
      const int64_t col0 = (int64_t)nb * BNP + h * 128;
      if (col0 >= N) continue;          // the empty half of a last, 128-wide N tile
      if constexpr (kQ == 2) {
        uint8_t* xb = smem + kStages * kStageBytes + CTL_BYTES + (warp - 2) * kXposeBytes;
        epilogue_rowcol(r0, r1, C, c_bf16, ldc, row, col0, M, N, qo, qc,
                        reinterpret_cast<float*>(xb), reinterpret_cast<uint32_t*>(xb + 4224), lane,
                        ((uint64_t)(M - 1) * ldc + N) * (c_bf16 ? 2u : 4u));
      } else {
        epilogue_out<kQ != 0>(r0, r1, C, c_bf16, ldc, row, col0, N, qo,
                              ((uint64_t)(M - 1) * ldc + N) * (c_bf16 ? 2u : 4u));
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();        // the leader's MMAs and the peer's epilogue are both done
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}
}  // namespace pair

// ---------------------------------------------------------------- host ---
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return tma_encode_fn(); }

bool make_code_map(CUtensorMap* m, const uint8_t* base, int64_t rows, int64_t kbytes,
                   uint32_t box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)kbytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kbytes};
  const cuuint32_t box[2] = {(cuuint32_t)BKB, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale array in the tensor-core layout as a 3-D tensor of 32-bit words:
// [rows/128 bands][K/tile_k tiles][128 words (512 bytes)] (a tile covers 128
// elements of K with a scale per 32, 64 with a scale per 16); a box covers
// `ktiles` tiles (one K stage) of `bands` consecutive bands.
bool make_scale_map(CUtensorMap* m, const uint8_t* base, int64_t rows, int64_t K, uint32_t bands,
                    uint32_t ktiles = 2, int64_t tile_k = 128) {
  const cuuint64_t dims[3] = {128, (cuuint64_t)(K / tile_k), (cuuint64_t)(rows / 128)};
  const cuuint64_t strides[2] = {512, (cuuint64_t)(K / tile_k) * 512};
  const cuuint32_t box[3] = {128, ktiles, bands};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale images as a 3-D tensor of 32-bit words {256, 4, n images} (4 KB
// each); a box covers `imgs` consecutive images.
bool make_image_map(CUtensorMap* m, const uint8_t* base, int64_t nimg, uint32_t imgs) {
  const cuuint64_t dims[3] = {256, 4, (cuuint64_t)nimg};
  const cuuint64_t strides[2] = {1024, 4096};
  const cuuint32_t box[3] = {256, 4, imgs};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale images for the kImg kernels, built from the standard tensor-core scale
// layout (512-byte tile (band, tile) at (band * ntiles + tile) * 512). An image
// is 4 KB: four identical 1 KB replicas, each [row group g (4)][chunk c (2)]
// [row j (8)][16 bytes], chunk c's bytes for row 8 g + j being that row's 16
// bytes in the chunk's tile -- the 128-row x 32-byte matrix a 128x256b copy
// reads, row r of which carries tile row r % 32. A-role images pair two
// consecutive tiles of one band (index band * ceil(ntiles / 2) + tile / 2);
// B-role images pair two bands at one tile (index band pair * ntiles + tile).
// A pair member past the last tile (odd ntiles) or the last band (odd band
// count of B) is written as zeros. One thread copies one 16-byte piece.
__global__ void __launch_bounds__(256)
scale_images_kernel(const uint8_t* __restrict__ sa, uint8_t* __restrict__ ia, int64_t na,
                    const uint8_t* __restrict__ sb, uint8_t* __restrict__ ib, int64_t nb,
                    int64_t ntiles, int64_t b_bands, uint64_t ws_bytes) {
  int64_t t = (int64_t)blockIdx.x * 256 + threadIdx.x;
  const bool bside = t >= na;
  if (bside) t -= na;
  if (bside && t >= nb) return;
  const int64_t img = t >> 8;
  const int w = (int)(t & 255), g = (w >> 4) & 3, c = (w >> 3) & 1, j = w & 7;
  int64_t tile;
  bool valid;
  if (!bside) {
    const int64_t per = (ntiles + 1) / 2, band = img / per, k = 2 * (img - band * per) + c;
    tile = band * ntiles + k;
    valid = k < ntiles;
  } else {
    const int64_t q = img / ntiles, band = 2 * q + c;
    tile = band * ntiles + (img - q * ntiles);
    valid = band < b_bands;
  }
  const uint4 v = valid ? __ldg(reinterpret_cast<const uint4*>((bside ? sb : sa) + tile * 512 + (8 * g + j) * 16))
                        : make_uint4(0u, 0u, 0u, 0u);
  put(reinterpret_cast<uint4*>((bside ? ib : ia) + t * 16), v, ia, ws_bytes);
}

// 512-byte scale tiles per 128-row band: K/128 (MXFP4), K/64 (NVFP4).
int64_t scale_tiles(int64_t K, bool nv) { return nv ? K / 64 : K / 128; }
// Image counts: A, (M / 128) bands x ceil(tiles / 2); B, ceil(N / 256) band pairs x tiles.
int64_t a_images(int64_t M, int64_t K, bool nv) { return (M / 128) * ((scale_tiles(K, nv) + 1) / 2); }
int64_t b_images(int64_t N, int64_t K, bool nv) { return ((N + 255) / 256) * scale_tiles(K, nv); }
constexpr int64_t kImageBytes = 4096;

// The image path needs image indices (TMA coordinates) and the pre-pass grid
// within 32 bits.
bool images_fit(int64_t M, int64_t N, int64_t K, bool nv) {
  const int64_t pieces = (a_images(M, K, nv) + b_images(N, K, nv)) * (kImageBytes / 16);
  return a_images(M, K, nv) < (1ll << 31) && b_images(N, K, nv) < (1ll << 31) &&
         (pieces + 255) / 256 < (1ll << 31);
}

// Builds A's and B's images in ws (A first) and encodes their tensor maps.
bool prepare_images(const uint8_t* sa, int64_t M, const uint8_t* sb, int64_t N, int64_t K, bool nv,
                    uint8_t* ws, size_t ws_bytes, CUtensorMap* tsa, CUtensorMap* tsb,
                    cudaStream_t st) {
  const int64_t ai = a_images(M, K, nv), bi = b_images(N, K, nv);
  uint8_t* ia = ws;
  uint8_t* ib = ws + ai * kImageBytes;
  if (!make_image_map(tsa, ia, ai, nv ? 2 : 1) || !make_image_map(tsb, ib, bi, nv ? 4 : 2))
    return false;
  const int64_t na = ai * (kImageBytes / 16), nb = bi * (kImageBytes / 16);
  scale_images_kernel<<<(unsigned)((na + nb + 255) / 256), 256, 0, st>>>(sa, ia, na, sb, ib, nb,
                                                                          scale_tiles(K, nv), N / 128,
                                                                          (uint64_t)ws_bytes);
  return true;
}

struct DevInfo {
  int sms = 0;
  int major = 0;
  bool attr_set = false;
};

DevInfo& dev_info(int dev) {
  static DevInfo info[kMaxDevices];
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  DevInfo& d = info[dev];
  if (!d.attr_set) {
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    if (d.major == 10) {
      cudaFuncSetAttribute(mxf4_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM_BYTES);
      cudaFuncSetAttribute(mxf4_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM_BYTES);
      cudaFuncSetAttribute(pair::mxf4_gemm_pair_kernel<0>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, pair::SMEM_BYTES);
      cudaFuncSetAttribute(pair::mxf4_gemm_pair_kernel<1>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, pair::SMEM_BYTES);
      cudaFuncSetAttribute(pair::mxf4_gemm_pair_kernel<2>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, pair::QC_SMEM_BYTES);
      cudaFuncSetAttribute(pair::mxf4_gemm_pair_kernel<0, pair::kMxf8>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, pair::SMEM_BYTES);
      cudaFuncSetAttribute(pair::mxf4_gemm_pair_kernel<0, pair::kMxf8e5>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, pair::SMEM_BYTES);
      cudaFuncSetAttribute(pair::mxf4_gemm_pair_kernel<0, pair::kNvf4>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, pair::NV_SMEM_BYTES);
      cudaFuncSetAttribute(pair::mxf4_gemm_pair_kernel<0, pair::kMxf4, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, pair::MXI_SMEM_BYTES);
      cudaFuncSetAttribute(pair::mxf4_gemm_pair_kernel<1, pair::kMxf4, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, pair::MXI_SMEM_BYTES);
      cudaFuncSetAttribute(pair::mxf4_gemm_pair_kernel<0, pair::kNvf4, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, pair::NVI_SMEM_BYTES);
    }
    d.attr_set = true;
  }
  return d;
}

}  // namespace

int64_t workspace_bytes(int64_t M, int64_t N, int64_t K, bool nv) {
  return (a_images(M, K, nv) + b_images(N, K, nv)) * kImageBytes;
}

// The library's own scratch for mxfp4_gemm_noalloc: a static device array (one
// per device context, no run-time allocation), its address looked up once per
// device.
__device__ __align__(256) uint8_t g_gemm_scratch[kStaticScratchBytes];

cudaError_t static_scratch(void** p) {
  static void* addr[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    e = cudaGetSymbolAddress(&addr[dev], g_gemm_scratch);
    if (e != cudaSuccess) return e;
  }
  *p = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_gemm(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                        const uint8_t* sb, int64_t M, int64_t N, int64_t K, void* c,
                        bool c_bf16, int64_t ldc, const OrientArgs* qout, const OrientArgs* qcol,
                        void* ws, size_t ws_bytes, cudaStream_t st, const char** why) {
  const OrientArgs none{};
  const OrientArgs& qo = qout ? *qout : none;
  const OrientArgs& qc = qcol ? *qcol : none;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DevInfo& d = dev_info(dev);
  if (d.major != 10) {
    *why = "tcgen05 block-scaled MMA needs an sm_100-family (GB300 sm_103) device";
    return cudaErrorNotSupported;
  }
  if (!encode_fn()) {
    *why = "driver entry point cuTensorMapEncodeTiled not available";
    return cudaErrorNotSupported;
  }
  ensure_context();
  CUtensorMap ta, tb;
  if (M % 256 == 0 || qcol) {
    // CTA pairs: 256 x 256 tiles (the column-wise epilogue runs only there; a
    // last M tile of 128 rows leaves CTA 1 of its pair without output). The
    // 1-CTA kernel below takes the other shapes with M % 256 == 128.
    CUtensorMap tsa, tsb;
    const bool img = ws != nullptr && !qcol && images_fit(M, N, K, false) &&
                     ws_bytes >= (size_t)workspace_bytes(M, N, K, false);
    (void)cudaGetLastError();  // drop a stale error left by an earlier call
    if (!make_code_map(&ta, qa, M, K / 2, pair::BM) || !make_code_map(&tb, qb, N, K / 2, pair::BNH) ||
        !(img ? prepare_images(sa, M, sb, N, K, false, static_cast<uint8_t*>(ws), ws_bytes, &tsa, &tsb, st)
              : (make_scale_map(&tsa, sa, M, K, 1) && make_scale_map(&tsb, sb, N, K, 2)))) {
      *why = "cuTensorMapEncodeTiled rejected the operand layout";
      return cudaErrorInvalidValue;
    }
    const int num_tiles = (int)(((M + 255) / 256) * ((N + pair::BNP - 1) / pair::BNP));
    const int pairs = d.sms / 2;
    const int grid = 2 * (num_tiles < pairs ? num_tiles : pairs);
    int64_t gm = kGroupBytes / (256 * (K / 2));
    gm = gm < 4 ? 4 : (gm > 32 ? 32 : gm);
    if (img && qout)
      pair::mxf4_gemm_pair_kernel<1, pair::kMxf4, true><<<grid, THREADS, pair::MXI_SMEM_BYTES, st>>>(
          ta, tb, tsa, tsb, c, (int)c_bf16, ldc, (int)M, (int)N, (int)K, (int)gm, 1.0f, qo, none);
    else if (img)
      pair::mxf4_gemm_pair_kernel<0, pair::kMxf4, true><<<grid, THREADS, pair::MXI_SMEM_BYTES, st>>>(
          ta, tb, tsa, tsb, c, (int)c_bf16, ldc, (int)M, (int)N, (int)K, (int)gm, 1.0f, qo, none);
    else if (qcol)
      pair::mxf4_gemm_pair_kernel<2><<<grid, THREADS, pair::QC_SMEM_BYTES, st>>>(
          ta, tb, tsa, tsb, c, (int)c_bf16, ldc, (int)M, (int)N, (int)K, (int)gm, 1.0f, qo, qc);
    else if (qout)
      pair::mxf4_gemm_pair_kernel<1><<<grid, THREADS, pair::SMEM_BYTES, st>>>(
          ta, tb, tsa, tsb, c, (int)c_bf16, ldc, (int)M, (int)N, (int)K, (int)gm, 1.0f, qo, none);
    else
      pair::mxf4_gemm_pair_kernel<0><<<grid, THREADS, pair::SMEM_BYTES, st>>>(
          ta, tb, tsa, tsb, c, (int)c_bf16, ldc, (int)M, (int)N, (int)K, (int)gm, 1.0f, qo, none);
    return cudaGetLastError();
  }
  if (!make_code_map(&ta, qa, M, K / 2, BM) || !make_code_map(&tb, qb, N, K / 2, BN)) {
    *why = "cuTensorMapEncodeTiled rejected the operand layout";
    return cudaErrorInvalidValue;
  }
  const int num_tiles = (int)((M / BM) * ((N + BN - 1) / BN));
  const int grid = num_tiles < d.sms ? num_tiles : d.sms;
  int64_t gm = kGroupBytes / (BM * (K / 2));
  gm = gm < 8 ? 8 : (gm > 64 ? 64 : gm);
  (void)cudaGetLastError();  // drop a stale error left by an earlier call
  if (qout)
    mxf4_gemm_kernel<true><<<grid, THREADS, SMEM_BYTES, st>>>(ta, tb, sa, sb, c, (int)c_bf16, ldc, (int)M,
                                                             (int)N, (int)K, (int)gm, qo);
  else
    mxf4_gemm_kernel<false><<<grid, THREADS, SMEM_BYTES, st>>>(ta, tb, sa, sb, c, (int)c_bf16, ldc, (int)M,
                                                              (int)N, (int)K, (int)gm, qo);
  return cudaGetLastError();
}

namespace {
// Self-test of the bounded waits: the one waiting thread waits on an mbarrier
// that nothing ever completes; after the wait limit it raises the error word
// (MXFP4_ERR_TIMEOUT) and returns, as a GEMM wait that ran out would.
__global__ void wait_timeout_probe_kernel() {
  __shared__ CtlT<1> ctl;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&ctl.full[0]), 1);
    ctl.abort = 0;
    ptx::fence_mbar_init();
    (void)wait_bar(ptx::smem_u32(&ctl.full[0]), 0u, &ctl);
  }
}
}  // namespace

cudaError_t launch_wait_probe(cudaStream_t st) {
  (void)cudaGetLastError();  // drop a stale error left by an earlier call
  wait_timeout_probe_kernel<<<1, 32, 0, st>>>();
  return cudaGetLastError();
}

cudaError_t launch_gemm_f8(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                           const uint8_t* sb, int64_t M, int64_t N, int64_t K, bool e5m2, void* c,
                           bool c_bf16, int64_t ldc, cudaStream_t st, const char** why) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DevInfo& d = dev_info(dev);
  if (d.major != 10) {
    *why = "tcgen05 block-scaled MMA needs an sm_100-family (GB300 sm_103) device";
    return cudaErrorNotSupported;
  }
  if (!encode_fn()) {
    *why = "driver entry point cuTensorMapEncodeTiled not available";
    return cudaErrorNotSupported;
  }
  ensure_context();
  CUtensorMap ta, tb, tsa, tsb;
  if (!make_code_map(&ta, qa, M, K, pair::BM) || !make_code_map(&tb, qb, N, K, pair::BNH) ||
      !make_scale_map(&tsa, sa, M, K, 1, 1) || !make_scale_map(&tsb, sb, N, K, 2, 1)) {
    *why = "cuTensorMapEncodeTiled rejected the operand layout";
    return cudaErrorInvalidValue;
  }
  const int num_tiles = (int)(((M + 255) / 256) * ((N + pair::BNP - 1) / pair::BNP));
  const int pairs = d.sms / 2;
  const int grid = 2 * (num_tiles < pairs ? num_tiles : pairs);
  int64_t gm = kGroupBytes / (256 * K);
  gm = gm < 4 ? 4 : (gm > 32 ? 32 : gm);
  const OrientArgs none{};
  (void)cudaGetLastError();  // drop a stale error left by an earlier call
  if (e5m2)
    pair::mxf4_gemm_pair_kernel<0, pair::kMxf8e5><<<grid, THREADS, pair::SMEM_BYTES, st>>>(
        ta, tb, tsa, tsb, c, (int)c_bf16, ldc, (int)M, (int)N, (int)K, (int)gm, 1.0f, none, none);
  else
    pair::mxf4_gemm_pair_kernel<0, pair::kMxf8><<<grid, THREADS, pair::SMEM_BYTES, st>>>(
        ta, tb, tsa, tsb, c, (int)c_bf16, ldc, (int)M, (int)N, (int)K, (int)gm, 1.0f, none, none);
  return cudaGetLastError();
}

cudaError_t launch_gemm_nv(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                           const uint8_t* sb, int64_t M, int64_t N, int64_t K, float alpha,
                           void* c, bool c_bf16, int64_t ldc, void* ws, size_t ws_bytes,
                           cudaStream_t st, const char** why) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DevInfo& d = dev_info(dev);
  if (d.major != 10) {
    *why = "tcgen05 block-scaled MMA needs an sm_100-family (GB300 sm_103) device";
    return cudaErrorNotSupported;
  }
  if (!encode_fn()) {
    *why = "driver entry point cuTensorMapEncodeTiled not available";
    return cudaErrorNotSupported;
  }
  ensure_context();
  CUtensorMap ta, tb, tsa, tsb;
  const bool img = ws != nullptr && images_fit(M, N, K, true) &&
                   ws_bytes >= (size_t)workspace_bytes(M, N, K, true);
  (void)cudaGetLastError();  // drop a stale error left by an earlier call
  if (!make_code_map(&ta, qa, M, K / 2, pair::BM) || !make_code_map(&tb, qb, N, K / 2, pair::BNH) ||
      !(img ? prepare_images(sa, M, sb, N, K, true, static_cast<uint8_t*>(ws), ws_bytes, &tsa, &tsb, st)
            : (make_scale_map(&tsa, sa, M, K, 1, 4, 64) && make_scale_map(&tsb, sb, N, K, 2, 4, 64)))) {
    *why = "cuTensorMapEncodeTiled rejected the operand layout";
    return cudaErrorInvalidValue;
  }
  const int num_tiles = (int)(((M + 255) / 256) * ((N + pair::BNP - 1) / pair::BNP));
  const int pairs = d.sms / 2;
  const int grid = 2 * (num_tiles < pairs ? num_tiles : pairs);
  int64_t gm = kGroupBytes / (256 * (K / 2));
  gm = gm < 4 ? 4 : (gm > 32 ? 32 : gm);
  const OrientArgs none{};
  if (img)
    pair::mxf4_gemm_pair_kernel<0, pair::kNvf4, true><<<grid, THREADS, pair::NVI_SMEM_BYTES, st>>>(
        ta, tb, tsa, tsb, c, (int)c_bf16, ldc, (int)M, (int)N, (int)K, (int)gm, alpha, none, none);
  else
    pair::mxf4_gemm_pair_kernel<0, pair::kNvf4><<<grid, THREADS, pair::NV_SMEM_BYTES, st>>>(
        ta, tb, tsa, tsb, c, (int)c_bf16, ldc, (int)M, (int)N, (int)K, (int)gm, alpha, none, none);
  return cudaGetLastError();
}

cudaError_t read_device_error(cudaStream_t st, uint32_t* err) {
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(err, g_gemm_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  if (*err) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
  }
  uint32_t qerr = 0;
  e = read_quant_error(&qerr);
  if (!*err) *err = qerr;
  return e;
}

}  // namespace mx
