"""GB300-native MXFP4 training hot path.

A thin Python binding over the C ABI of ``libmxfp4.so`` (declared in
``include/mxfp4.h``). PyTorch supplies device memory and streams; every step
of the computation runs in the library's sm_103a kernels. There is no CPU or
PyTorch fallback: if the library is missing or fails to load, every call
raises.

Calls (same names as the C ABI):
  mxfp4_quantize    fused rotation + E8M0 scale + E2M1 rounding + packing,
                    row-wise and/or column-wise in one pass
  mxfp4_dequantize  codes * 2^(scale - 127) -> fp32
  mxfp4_gemm        block-scaled MXFP4 GEMM on tcgen05 tensor cores (fp32 or
                    bf16 C); mxfp4_gemm_quantize with the quantizer in its
                    epilogue; mxfp8_gemm (E4M3) and nvfp4_gemm (1x16 blocks,
                    E4M3 scales)
  hadamard32        stand-alone 32-point block rotation
  mxfp4_tensor_amax device max-abs and NVFP4 per-tensor exponent
                    (tensor_amax, nvfp4_tensor_exp)
"""
from .binding import (  # noqa: F401
    BLOCK_1X32,
    BLOCK_32X32,
    BLOCK_64X64,
    BLOCK_1X16,
    DTYPE_BF16,
    DTYPE_F32,
    FORMAT_E2M1,
    FORMAT_E4M3,
    FORMAT_E5M2,
    LAYOUT_MMA,
    LAYOUT_ROWMAJOR,
    ROUND_RTN,
    ROUND_SR,
    SCALE_FLOOR,
    SCALE_ROUNDUP,
    Mxfp4Error,
    QuantParams,
    device_status,
    selftest_wait_timeout,
    hadamard32,
    lib,
    lib_path,
    mxfp4_dequantize,
    mxfp4_gemm,
    mxfp4_gemm_noalloc,
    mxfp4_gemm_quantize,
    mxfp8_gemm,
    gemm_workspace_size,
    nvfp4_gemm,
    nvfp4_tensor_exp,
    tensor_amax,
    mxfp4_quantize,
    scale_numel,
)
from .linear import LinearRecipe, Mxfp4Linear, mxfp4_linear, recipe_1d, recipe_2d_sr  # noqa: F401
