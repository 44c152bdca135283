"""The C ABI library loads, exports every function include/mxfp4.h declares,
and rejects bad arguments on the host (no GPU needed for these paths)."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxfp4.h")


@pytest.fixture(scope="module")
def L():
    from gemm_pt_block_gb300 import build as b

    b.build()
    import gemm_pt_block_gb300 as mx

    return mx.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_four_hot_path_calls():
    names = _declared_functions()
    for n in ["mxfp4_quantize", "mxfp4_dequantize", "mxfp4_gemm", "hadamard32"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", L._name], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\S+)", out))
    for name in _declared_functions():
        assert name in exported, name


def test_header_compiles_as_c():
    src = '#include "mxfp4.h"\nint main(void){ mxfp4_quant_params p = {0}; (void)p; return 0; }\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-x", "c", "-", "-fsyntax-only"], input=src, text=True, capture_output=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(L):
    names = [L.mxfp4_status_string(i).decode() for i in range(8)]
    assert names == ["MXFP4_OK", "MXFP4_ERR_INVALID_ARG", "MXFP4_ERR_SHAPE", "MXFP4_ERR_ALIGN",
                     "MXFP4_ERR_UNSUPPORTED", "MXFP4_ERR_CUDA", "MXFP4_ERR_TIMEOUT",
                     "MXFP4_ERR_BOUNDS"]
    assert L.mxfp4_bounds_check_shrink(16) == 4      # the regular library refuses the diagnostic


def test_host_side_validation(L):
    import gemm_pt_block_gb300 as mx
    from gemm_pt_block_gb300.binding import _CParams

    P = ctypes.c_void_p
    good = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails validation
    p = mx.QuantParams()._c()
    # no orientation requested
    assert L.mxfp4_quantize(good, 0, 32, 32, 32, None, None, None, None, None, None, None) == 1
    # cols not a multiple of 32
    assert L.mxfp4_quantize(good, 0, 32, 48, 48, ctypes.byref(p), good, good, None, None, None, None) == 2
    # ld < cols
    assert L.mxfp4_quantize(good, 0, 32, 64, 32, ctypes.byref(p), good, good, None, None, None, None) == 2
    # misaligned x
    assert L.mxfp4_quantize(P((1 << 20) + 2), 0, 32, 32, 32, ctypes.byref(p), good, good,
                            None, None, None, None) == 3
    # bad enum
    bad = _CParams(5, 0, 0, 0, 0, 0, 0, 0, 0)
    assert L.mxfp4_quantize(good, 0, 32, 32, 32, ctypes.byref(bad), good, good, None, None, None, None) == 1
    # reserved field
    bad = _CParams(0, 0, 0, 0, 0, 0, 0, 0, 7)
    assert L.mxfp4_quantize(good, 0, 32, 32, 32, ctypes.byref(bad), good, good, None, None, None, None) == 1
    # size limit of the 32-bit unit counter: rows * cols / 16 must stay below 2^31
    assert L.mxfp4_quantize(good, 0, 65536, 524288, 524288, ctypes.byref(p), good, good,
                            None, None, None, None) == 2
    assert b"2^31" in L.mxfp4_last_error()
    assert L.mxfp4_quantize(good, 0, 1 << 22, 1 << 17, 1 << 17, ctypes.byref(p), good, good,
                            None, None, None, None) == 2
    # dimensions whose product would overflow int64 are rejected as shapes
    # before any pointer or size arithmetic
    huge = 1 << 40
    assert L.mxfp4_quantize(None, 0, huge, huge, huge, ctypes.byref(p), None, None,
                            None, None, None, None) == 2
    assert b"too large" in L.mxfp4_last_error()
    assert L.mxfp4_dequantize(None, None, 0, huge, huge, None, None) == 2
    assert L.hadamard32(None, 0, huge, huge, huge, 0, 0, None, None) == 2
    # column output needs rows % 32
    assert L.mxfp4_quantize(good, 0, 48, 32, 32, None, None, None, ctypes.byref(p), good, good, None) == 2
    # tensor-core scale layout needs 128-row tiles
    pm = mx.QuantParams(scale_layout=mx.LAYOUT_MMA)._c()
    assert L.mxfp4_quantize(good, 0, 64, 128, 128, ctypes.byref(pm), good, good, None, None, None, None) == 2
    # GEMM shapes
    assert L.mxfp4_gemm(good, good, good, good, 100, 256, 256, good, 256, None) == 2
    assert L.mxfp4_gemm(good, good, good, good, 128, 192, 256, good, 192, None) == 2
    assert L.mxfp4_gemm(good, good, good, good, 128, 256, 192, good, 256, None) == 2
    assert L.mxfp4_gemm(good, good, good, good, 128, 256, 0, good, 256, None) == 2
    assert L.mxfp4_gemm(good, good, good, good, 128, 256, 256, good, 100, None) == 2
    assert L.mxfp4_gemm(None, good, good, good, 128, 256, 256, good, 256, None) == 1
    assert L.mxfp4_gemm(good, good, good, good, 128, 256, 256, P((1 << 20) + 4), 256, None) == 3
    # bf16 / fp32 C selection
    assert L.mxfp4_gemm_ex(good, good, good, good, 128, 256, 256, good, 2, 256, None, 0, None) == 1
    assert L.mxfp4_gemm_ex(good, good, good, good, 100, 256, 256, good, 0, 256, None, 0, None) == 2
    assert L.mxfp4_gemm_ex(good, good, good, good, 128, 256, 256, good, 0, 260, None, 0, None) == 3
    # misaligned workspace
    assert L.mxfp4_gemm_ex(good, good, good, good, 256, 256, 256, good, 0, 256, P((1 << 20) + 8),
                           1 << 20, None) == 3
    assert L.mxfp4_gemm_workspace_size(256, 512, 1024, 32) == 4 * (256 + 512) * 1024 // 32
    assert L.mxfp4_gemm_workspace_size(256, 512, 1024, 16) == 4 * (256 + 512) * 1024 // 16
    assert L.mxfp4_gemm_workspace_size(256, 512, 1024, 8) == 0
    # the static-scratch GEMM: images above its 96 MiB are refused before any device call
    assert L.mxfp4_gemm_noalloc(good, good, good, good, 16384, 16384, 32768, good, 16384, None) == 2
    assert L.mxfp4_gemm_noalloc(good, good, good, good, 256, 256, 256, None, 256, None) == 1
    assert L.mxfp4_gemm_noalloc(good, good, good, good, 12288, 12288, 32768 + 256, good, 12288,
                                None) == 2
    # dimensions are validated before the image size is formed (no overflow)
    assert L.mxfp4_gemm_noalloc(good, good, good, good, 1 << 62, 1 << 62, 1 << 62, good, 1 << 62,
                                None) == 2
    assert b"too large" in L.mxfp4_last_error()
    assert L.mxfp4_gemm_noalloc(good, good, good, good, 256, 320, 256, good, 320, None) == 2
    # workspace size: A's K and B's N rounded up to 256
    assert L.mxfp4_gemm_workspace_size(256, 384, 640, 32) == 4 * (256 * 768 + 512 * 640) // 32
    assert L.mxfp4_gemm_workspace_size(384, 384, 384, 16) == 4 * (384 * 384 + 512 * 384) // 16
    assert L.mxfp8_gemm(good, good, good, good, 256, 256, 256, good, 3, 256, None) == 1
    assert L.mxfp8_gemm(good, good, good, good, 64, 256, 128, good, 0, 256, None) == 2
    assert L.mxfp8_gemm_ex(good, good, good, good, 256, 256, 128, 0, good, 0, 256, None) == 1
    assert L.mxfp8_gemm_ex(good, good, good, good, 256, 256, 128, 3, good, 0, 256, None) == 1
    assert L.mxfp8_gemm_ex(good, good, good, good, 256, 192, 128, 2, good, 0, 256, None) == 2
    pe5 = mx.QuantParams(rounding=mx.ROUND_SR, elem_format=mx.FORMAT_E5M2)._c()
    assert L.mxfp4_quantize(good, 0, 32, 32, 32, ctypes.byref(pe5), good, good, None, None, None, None) == 4
    pe3 = _CParams(0, 0, 0, 0, 0, 0, 0, 0, 3)
    assert L.mxfp4_quantize(good, 0, 32, 32, 32, ctypes.byref(pe3), good, good, None, None, None, None) == 1
    # NVFP4: tensor_exp only with 1x16 blocks, in range; E2M1 elements only
    pe = mx.QuantParams(tensor_exp=1)._c()
    assert L.mxfp4_quantize(good, 0, 32, 32, 32, ctypes.byref(pe), good, good, None, None, None, None) == 1
    pe = mx.QuantParams(block=mx.BLOCK_1X16, tensor_exp=101)._c()
    assert L.mxfp4_quantize(good, 0, 32, 32, 32, ctypes.byref(pe), good, good, None, None, None, None) == 1
    pe = mx.QuantParams(block=mx.BLOCK_1X16, elem_format=mx.FORMAT_E4M3)._c()
    assert L.mxfp4_quantize(good, 0, 32, 32, 32, ctypes.byref(pe), good, good, None, None, None, None) == 4
    assert L.nvfp4_gemm(good, good, 0, good, good, 0, 256, 256, 96, good, 1, 256, None, 0, None) == 2
    assert L.nvfp4_gemm(good, good, 100, good, good, 30, 256, 256, 256, good, 1, 256, None, 0, None) == 1
    assert L.nvfp4_gemm(good, good, 0, good, good, 0, 256, 256, 256, good, 7, 256, None, 0, None) == 1
    pq = mx.QuantParams()._c()
    assert L.mxfp4_gemm_quantize(good, good, good, good, 128, 256, 256, good, 5, 256,
                                 ctypes.byref(pq), good, good, None, None, None, None, 0, None) == 1
    pnv = mx.QuantParams(block=mx.BLOCK_1X16)._c()
    assert L.mxfp4_gemm_quantize(good, good, good, good, 128, 256, 256, good, 1, 256,
                                 ctypes.byref(pnv), good, good, None, None, None, None, 0, None) == 4
    # no orientation; column-wise NVFP4 output (not fused)
    assert L.mxfp4_gemm_quantize(good, good, good, good, 256, 256, 256, good, 1, 256,
                                 None, None, None, None, None, None, None, 0, None) == 1
    assert L.mxfp4_gemm_quantize(good, good, good, good, 128, 256, 256, good, 1, 256,
                                 None, None, None, ctypes.byref(pnv), good, good, None, 0, None) == 4
    # dequantize / hadamard32
    assert L.mxfp4_dequantize(good, good, 1, 64, 128, good, None) == 2
    assert L.mxfp4_dequantize(good, good, 2, 64, 128, good, None) == 1
    assert L.mxfp4_dequantize_ex(good, good, 0, 3, 1, 0, 64, 128, good, None) == 4   # 1x16 + E4M3
    assert L.mxfp4_dequantize_ex(good, good, 0, 0, 0, 2, 64, 128, good, None) == 1   # tensor_exp
    assert L.mxfp4_dequantize_ex(good, good, 0, 7, 0, 0, 64, 128, good, None) == 1   # block
    assert L.mxfp4_dequantize_ex(good, good, 1, 3, 0, 0, 64, 128, good, None) == 2   # MMA rows
    assert L.hadamard32(good, 0, 4, 40, 40, 0, 0, good, None) == 2
    assert L.hadamard32(good, 0, 4, 32, 32, 0, 2, good, None) == 1
    assert b"multiple of 32" in L.mxfp4_last_error() or len(L.mxfp4_last_error()) > 0


def test_binding_refuses_cpu_tensors():
    import torch

    import gemm_pt_block_gb300 as mx

    with pytest.raises(ValueError):
        mx.mxfp4_quantize(torch.zeros(32, 32, dtype=torch.bfloat16), mx.QuantParams())
