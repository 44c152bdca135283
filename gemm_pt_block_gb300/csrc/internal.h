// internal.h -- launchers shared between the C-ABI layer and the kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "mx_device.cuh"

namespace mx {

// One output orientation of the quantizer, already validated. The Philox round
// keys and per-lane sign words are precomputed on the host (see api.cu).
struct OrientArgs {
  int32_t block;        // 0: 1-D (1x32, or 1x16 with nv), 1: 32x32, 2: 64x64
  int32_t roundup;      // scale mode: 0 floor, 1 round-up
  int32_t sr;           // 0: nearest-even, 1: stochastic
  int32_t mma_layout;   // scale array layout: 0 row-major, 1 tensor-core tiles
  int32_t wht;          // rotate 32-runs along the quantization axis first
  int32_t e4m3;         // element format: 0 E2M1 (MXFP4), 1 one byte per element (MXFP8)
  int32_t e5m2;         // with e4m3 set: 0 E4M3 elements, 1 E5M2 elements
  int32_t nv;           // 1x16 blocks with E4M3 scales (NVFP4); block is then 0
  float nv_p2k;         // NVFP4: 2^tensor_exp
  float nv_zmul;        // NVFP4: 2^-tensor_exp / 6 rounded to fp32 (first guess only)
  uint32_t sign_mask;
  uint64_t seed;
  uint32_t stream;
  uint8_t* q;           // packed codes [out_rows, K/2]
  uint8_t* s;           // scales
  PhiloxKeys keys;      // the ten round keys of `seed`
  uint32_t sm_half[2];  // sign bits of local elements, lane holding block half 0 / 1
  uint32_t sm_inter[2]; // sign bits of local elements, lane holding even / odd block elements
  uint32_t xw[2][8];    // sign bits placed on bf16 word pairs (bits 15 and 31), per half
  float sgn[32];        // rotation signs s_i as factors +-1 (all +1 without rotation)
  uint64_t q_bytes;     // extent of q and s in bytes (checked in bounds-checking builds)
  uint64_t s_bytes;
};

// Device error word value of a store outside its output (bounds-checking builds).
constexpr uint32_t kErrBounds = 7;

// Fills keys, sm_*, xw and sgn from seed and sign_mask.
void prepare_orient(OrientArgs* o);

// All launchers return the cudaError_t of the launch.
cudaError_t launch_quantize(const void* x, bool f32_in, int64_t rows, int64_t cols, int64_t ld,
                            const OrientArgs* row, const OrientArgs* col, cudaStream_t st);
// fmt: 0 MXFP4, 1 MXFP8 (E4M3 codes), 2 NVFP4 (E4M3 scales per 16, times p2k),
// 3 MXFP8 with E5M2 codes.
cudaError_t launch_dequantize(const uint8_t* q, const uint8_t* s, bool mma_layout, int64_t rows,
                              int64_t cols, int fmt, float p2k, float* out, cudaStream_t st);
cudaError_t launch_hadamard32(const void* x, bool f32_in, int64_t rows, int64_t cols, int64_t ld,
                              uint32_t sign_mask, bool inverse, float* y, cudaStream_t st);
// Max |x| into *amax (device) and, when tensor_exp is non-NULL, the NVFP4
// per-tensor exponent derived from it (device int).
cudaError_t launch_amax(const void* x, bool f32_in, int64_t rows, int64_t cols, int64_t ld,
                        float* amax, int32_t* tensor_exp, cudaStream_t st);
// qout / qcol: also quantize C row-wise / column-wise (C^T along M) in the
// epilogue (nullptr: not produced; column-wise needs M % 256 == 0); with
// either, c may be nullptr (no C output). ws: optional workspace of ws_bytes;
// when it holds workspace_bytes(M, N, K) and no column-wise output is asked
// for, the CTA-pair GEMM reads its scales as replicated images built there
// first (same results, fewer tensor-memory copies).
int64_t workspace_bytes(int64_t M, int64_t N, int64_t K, bool nv);
// Size and address (this device) of the library's static GEMM scratch.
// Per-device caches (attributes, scratch addresses) cover device ordinals
// 0 .. kMaxDevices - 1; a call on a higher ordinal returns cudaErrorInvalidDevice.
constexpr int kMaxDevices = 64;
constexpr size_t kStaticScratchBytes = 96ull << 20;
cudaError_t static_scratch(void** p);
cudaError_t launch_gemm(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                        const uint8_t* sb, int64_t M, int64_t N, int64_t K, void* c,
                        bool c_bf16, int64_t ldc, const OrientArgs* qout, const OrientArgs* qcol,
                        void* ws, size_t ws_bytes, cudaStream_t st, const char** why);
// Reads and clears the quantizer's device error word.
cudaError_t read_quant_error(uint32_t* err);
// Reads and clears the device error words (synchronizes st).
cudaError_t read_device_error(cudaStream_t st, uint32_t* err);
// MXFP8 GEMM (E4M3, or E5M2 with e5m2, codes [M, K], [N, K] bytes, both
// operands the same format; E8M0 scales in the tensor-core layout): CTA pairs,
// M % 256 == 0, N % 256 == 0, K % 128 == 0.
cudaError_t launch_gemm_f8(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                           const uint8_t* sb, int64_t M, int64_t N, int64_t K, bool e5m2, void* c,
                           bool c_bf16, int64_t ldc, cudaStream_t st, const char** why);
// NVFP4 GEMM (E2M1 codes [M, K/2], [N, K/2]; E4M3 scales per 16 in the
// tensor-core layout with K/16 scale columns): C = alpha * sum, alpha a power
// of two; CTA pairs, M % 256 == 0, N % 256 == 0, K % 256 == 0.
cudaError_t launch_gemm_nv(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                           const uint8_t* sb, int64_t M, int64_t N, int64_t K, float alpha,
                           void* c, bool c_bf16, int64_t ldc, void* ws, size_t ws_bytes,
                           cudaStream_t st, const char** why);
// One-thread kernel whose bounded wait never completes (sets the error word).
cudaError_t launch_wait_probe(cudaStream_t st);

}  // namespace mx
