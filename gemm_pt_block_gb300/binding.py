"""ctypes marshalling for libmxfp4.so: torch tensors in, pointers and sizes out.

Nothing here computes: each function checks that tensors live on a CUDA
device with the expected dtype, contiguity and size (the C ABI takes raw
pointers and cannot check extents), allocates outputs the caller did not
pass, and forwards raw pointers plus the current CUDA stream to the C ABI.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libmxfp4.so"

BLOCK_1X32, BLOCK_32X32, BLOCK_64X64, BLOCK_1X16 = 0, 1, 2, 3
FORMAT_E2M1, FORMAT_E4M3, FORMAT_E5M2 = 0, 1, 2
SCALE_FLOOR, SCALE_ROUNDUP = 0, 1
ROUND_RTN, ROUND_SR = 0, 1
LAYOUT_ROWMAJOR, LAYOUT_MMA = 0, 1
DTYPE_BF16, DTYPE_F32 = 0, 1

_STATUS = {
    0: "MXFP4_OK", 1: "MXFP4_ERR_INVALID_ARG", 2: "MXFP4_ERR_SHAPE", 3: "MXFP4_ERR_ALIGN",
    4: "MXFP4_ERR_UNSUPPORTED", 5: "MXFP4_ERR_CUDA", 6: "MXFP4_ERR_TIMEOUT",
    7: "MXFP4_ERR_BOUNDS",
}


class Mxfp4Error(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{_STATUS.get(status, status)}: {detail}")
        self.status = status


class _CParams(ctypes.Structure):
    _fields_ = [
        ("block", ctypes.c_int32),
        ("scale_mode", ctypes.c_int32),
        ("rounding", ctypes.c_int32),
        ("scale_layout", ctypes.c_int32),
        ("wht", ctypes.c_int32),
        ("wht_sign_mask", ctypes.c_uint32),
        ("seed", ctypes.c_uint64),
        ("sr_stream", ctypes.c_uint32),
        ("elem_format", ctypes.c_uint32),
        ("tensor_exp", ctypes.c_int32),
    ]


@dataclass(frozen=True)
class QuantParams:
    """Parameters of one quantizer output orientation (see mxfp4_quant_params)."""
    block: int = BLOCK_1X32
    scale_mode: int = SCALE_FLOOR
    rounding: int = ROUND_RTN
    scale_layout: int = LAYOUT_ROWMAJOR
    wht: bool = False
    wht_sign_mask: int = 0
    seed: int = 0
    sr_stream: int = 0
    elem_format: int = 0          # FORMAT_E2M1 (MXFP4), FORMAT_E4M3 or FORMAT_E5M2 (MXFP8)
    tensor_exp: int = 0           # BLOCK_1X16 (NVFP4): per-tensor factor 2^tensor_exp

    def _c(self) -> _CParams:
        return _CParams(self.block, self.scale_mode, self.rounding, self.scale_layout,
                        int(bool(self.wht)), self.wht_sign_mask & 0xFFFFFFFF,
                        self.seed & 0xFFFFFFFFFFFFFFFF, self.sr_stream & 0xFFFFFFFF,
                        self.elem_format, self.tensor_exp)

    def code_cols(self, k: int) -> int:
        """Bytes of codes per output row for K elements."""
        return k if self.elem_format in (FORMAT_E4M3, FORMAT_E5M2) else k // 2

    def scale_cols(self, k: int) -> int:
        """Scale bytes per output row for K elements (one per block along K)."""
        return k // 16 if self.block == BLOCK_1X16 else k // 32


_lib = None


def lib_path() -> str:
    return os.path.join(HERE, _LIB_NAME)


def load_library(path: str) -> ctypes.CDLL:
    """Loads a build of the library at `path` and declares its C signatures
    (the regular libmxfp4.so, or the bounds-checking libmxfp4_bc.so that the
    tests use)."""
    L = ctypes.CDLL(path)
    P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    L.mxfp4_quantize.restype = i32
    L.mxfp4_quantize.argtypes = [P, i32, i64, i64, i64, ctypes.POINTER(_CParams), P, P,
                                 ctypes.POINTER(_CParams), P, P, P]
    L.mxfp4_dequantize.restype = i32
    L.mxfp4_dequantize.argtypes = [P, P, i32, i64, i64, P, P]
    L.mxfp4_dequantize_ex.restype = i32
    L.mxfp4_dequantize_ex.argtypes = [P, P, i32, i32, ctypes.c_uint32, i32, i64, i64, P, P]
    L.mxfp4_gemm.restype = i32
    L.mxfp4_gemm.argtypes = [P, P, P, P, i64, i64, i64, P, i64, P]
    sz = ctypes.c_size_t
    L.mxfp4_gemm_ex.restype = i32
    L.mxfp4_gemm_ex.argtypes = [P, P, P, P, i64, i64, i64, P, i32, i64, P, sz, P]
    L.mxfp4_gemm_noalloc.restype = i32
    L.mxfp4_gemm_noalloc.argtypes = [P, P, P, P, i64, i64, i64, P, i64, P]
    L.mxfp4_gemm_workspace_size.restype = sz
    L.mxfp4_gemm_workspace_size.argtypes = [i64, i64, i64, i32]
    L.nvfp4_gemm.restype = i32
    L.nvfp4_gemm.argtypes = [P, P, i32, P, P, i32, i64, i64, i64, P, i32, i64, P, sz, P]
    L.mxfp8_gemm.restype = i32
    L.mxfp8_gemm.argtypes = [P, P, P, P, i64, i64, i64, P, i32, i64, P]
    L.mxfp8_gemm_ex.restype = i32
    L.mxfp8_gemm_ex.argtypes = [P, P, P, P, i64, i64, i64, ctypes.c_uint32, P, i32, i64, P]
    L.mxfp4_gemm_quantize.restype = i32
    L.mxfp4_gemm_quantize.argtypes = [P, P, P, P, i64, i64, i64, P, i32, i64,
                                      ctypes.POINTER(_CParams), P, P,
                                      ctypes.POINTER(_CParams), P, P, P, sz, P]
    L.mxfp4_tensor_amax.restype = i32
    L.mxfp4_tensor_amax.argtypes = [P, i32, i64, i64, i64, P, P, P]
    L.hadamard32.restype = i32
    L.hadamard32.argtypes = [P, i32, i64, i64, i64, ctypes.c_uint32, i32, P, P]
    L.mxfp4_status_string.restype = ctypes.c_char_p
    L.mxfp4_status_string.argtypes = [i32]
    L.mxfp4_last_error.restype = ctypes.c_char_p
    L.mxfp4_last_error.argtypes = []
    L.mxfp4_device_status.restype = i32
    L.mxfp4_device_status.argtypes = [P]
    L.mxfp4_selftest_wait_timeout.restype = i32
    L.mxfp4_selftest_wait_timeout.argtypes = [P]
    L.mxfp4_bounds_check_shrink.restype = i32
    L.mxfp4_bounds_check_shrink.argtypes = [i64]
    return L


def lib() -> ctypes.CDLL:
    """Loads libmxfp4.so (built by gemm_pt_block_gb300.build). Raises if absent."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built; run gemm_pt_block_gb300.build.build() "
                               "(there is no fallback implementation)")
        _lib = load_library(path)
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise Mxfp4Error(status, lib().mxfp4_last_error().decode())


def _stream(t: torch.Tensor, stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream(t.device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _cuda2d(x: torch.Tensor, name: str) -> None:
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dim() != 2 or (x.shape[1] > 1 and x.stride(1) != 1):
        raise ValueError(f"{name} must be 2-D with unit column stride")


def scale_numel(rows: int, k: int, block: int = BLOCK_1X32) -> int:
    return rows * (k // 16 if block == BLOCK_1X16 else k // 32)


def _buffer(t: torch.Tensor, numel: int, dtype: torch.dtype, name: str) -> None:
    """A caller-supplied buffer the library reads or writes as `numel` dense
    elements of `dtype`: on a CUDA device, contiguous and large enough (the C
    ABI takes raw pointers and cannot check extents itself)."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements; {numel} are needed")


def _matrix_out(c: torch.Tensor, M: int, N: int, ldc: int, name: str = "c") -> None:
    """C [M, N] with row stride ldc inside c's storage, unit column stride."""
    if not c.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if c.dim() != 2 or c.shape[0] < M or c.shape[1] < N or (N > 1 and c.stride(1) != 1):
        raise ValueError(f"{name} must be 2-D, at least [{M}, {N}], with unit column stride")
    if ldc < N:
        raise ValueError(f"ldc ({ldc}) < N ({N})")
    es = c.element_size()
    room = c.untyped_storage().nbytes() - c.storage_offset() * es
    if M > 0 and N > 0 and ((M - 1) * ldc + N) * es > room:
        raise ValueError(f"{name}'s storage is too small for [{M}, {N}] with ldc {ldc}")


def _operand(q: torch.Tensor, s: torch.Tensor, rows: int, K: int, code_bytes: int, scale_div: int,
             name: str) -> None:
    _buffer(q, rows * K * code_bytes // 2, torch.uint8, "q" + name)
    _buffer(s, rows * (K // scale_div), torch.uint8, "s" + name)


def _scales_out(rows: int, k: int, p: QuantParams, dev) -> torch.Tensor:
    if p.scale_layout == LAYOUT_MMA:
        return torch.empty(scale_numel(rows, k, p.block), dtype=torch.uint8, device=dev)
    return torch.empty((rows, p.scale_cols(k)), dtype=torch.uint8, device=dev)


def mxfp4_quantize(x: torch.Tensor, row: QuantParams | None = None, col: QuantParams | None = None,
                   *, q_row=None, s_row=None, q_col=None, s_col=None, stream=None):
    """Quantize x [rows, cols] (bf16 or fp32) row-wise and/or column-wise.

    Returns (q_row, s_row, q_col, s_col); entries for an orientation not asked
    for are None. Codes are [rows, cols/2] (row-wise) / [cols, rows/2]
    (column-wise) uint8; scales are [out_rows, K/32] (K/16 for NVFP4's 1x16
    blocks; row-major layout) or flat (tensor-core layout).
    """
    _cuda2d(x, "x")
    if x.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif x.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise TypeError("x must be bfloat16 or float32")
    rows, cols = x.shape
    ld = x.stride(0) if rows > 1 else cols
    dev = x.device
    if row is not None:
        q_row = torch.empty((rows, row.code_cols(cols)), dtype=torch.uint8, device=dev) if q_row is None else q_row
        s_row = _scales_out(rows, cols, row, dev) if s_row is None else s_row
    if col is not None:
        q_col = torch.empty((cols, col.code_cols(rows)), dtype=torch.uint8, device=dev) if q_col is None else q_col
        s_col = _scales_out(cols, rows, col, dev) if s_col is None else s_col
    if row is not None:
        _buffer(q_row, rows * row.code_cols(cols), torch.uint8, "q_row")
        _buffer(s_row, scale_numel(rows, cols, row.block), torch.uint8, "s_row")
    if col is not None:
        _buffer(q_col, cols * col.code_cols(rows), torch.uint8, "q_col")
        _buffer(s_col, scale_numel(cols, rows, col.block), torch.uint8, "s_col")
    rp = row._c() if row is not None else None
    cp = col._c() if col is not None else None
    _check(lib().mxfp4_quantize(
        _ptr(x), dt, rows, cols, ld,
        ctypes.byref(rp) if rp is not None else None, _ptr(q_row if row else None),
        _ptr(s_row if row else None),
        ctypes.byref(cp) if cp is not None else None, _ptr(q_col if col else None),
        _ptr(s_col if col else None), _stream(x, stream)))
    return (q_row if row else None, s_row if row else None,
            q_col if col else None, s_col if col else None)


def mxfp4_dequantize(q: torch.Tensor, s: torch.Tensor, rows: int, cols: int,
                     scale_layout: int = LAYOUT_ROWMAJOR, *, params: QuantParams | None = None,
                     out=None, stream=None):
    """fp32 [rows, cols] reconstruction of codes q with scales s. `params` (the
    parameters the tensor was quantized with) selects the format: MXFP4 by
    default, MXFP8 (elem_format E4M3) or NVFP4 (block 1x16, its tensor_exp);
    its scale_layout is used when given."""
    if not q.is_cuda or not s.is_cuda:
        raise ValueError("q and s must be CUDA tensors")
    p = QuantParams() if params is None else params
    _buffer(q, rows * p.code_cols(cols), torch.uint8, "q")
    _buffer(s, scale_numel(rows, cols, p.block), torch.uint8, "s")
    out = torch.empty((rows, cols), dtype=torch.float32, device=q.device) if out is None else out
    _buffer(out, rows * cols, torch.float32, "out")
    if params is None:
        _check(lib().mxfp4_dequantize(_ptr(q), _ptr(s), scale_layout, rows, cols, _ptr(out),
                                      _stream(q, stream)))
    else:
        _check(lib().mxfp4_dequantize_ex(_ptr(q), _ptr(s), params.scale_layout, params.block,
                                         params.elem_format, params.tensor_exp, rows, cols,
                                         _ptr(out), _stream(q, stream)))
    return out


def _check_operands(qa, sa, qb, sb) -> None:
    for t, n in ((qa, "qa"), (sa, "sa"), (qb, "qb"), (sb, "sb")):
        if not t.is_cuda or t.dtype != torch.uint8:
            raise ValueError(f"{n} must be a CUDA uint8 tensor")


def _c_dtype(c, out_dtype) -> int:
    dt = c.dtype if c is not None else out_dtype
    if dt == torch.float32:
        return DTYPE_F32
    if dt == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError("C must be float32 or bfloat16")


def gemm_workspace_size(M: int, N: int, K: int, scale_block: int = 32) -> int:
    """Bytes of the optional GEMM workspace (scale images): 4 (M + N) K / scale_block."""
    return int(lib().mxfp4_gemm_workspace_size(M, N, K, scale_block))


def _workspace(workspace, M: int, N: int, K: int, scale_block: int, device):
    """(pointer, bytes) for the C call: a caller tensor, none (False), or a fresh
    caller-owned tensor from PyTorch's allocator when the CTA-pair GEMM can use it."""
    if workspace is False or (workspace is None and M % 256 != 0):
        return None, 0
    if workspace is None:
        workspace = torch.empty(gemm_workspace_size(M, N, K, scale_block), dtype=torch.uint8,
                                device=device)
    if not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    return workspace, workspace.numel() * workspace.element_size()


def mxfp4_gemm(qa: torch.Tensor, sa: torch.Tensor, qb: torch.Tensor, sb: torch.Tensor,
               M: int, N: int, K: int, *, c=None, ldc: int | None = None,
               out_dtype: torch.dtype = torch.float32, workspace=None, stream=None):
    """C[M, N] = deq(A) deq(B)^T (fp32 sums, stored as fp32 or bf16: out_dtype, or
    c's dtype); A, B K-major packed codes, scales in tensor-core layout.

    `workspace`: None (default) lets the call use a scratch tensor for its scale
    images (mxfp4_gemm_ex; same result, faster), a CUDA tensor supplies it,
    False calls the plain mxfp4_gemm entry point (fp32 C) without one."""
    _check_operands(qa, sa, qb, sb)
    _operand(qa, sa, M, K, 1, 32, "a")
    _operand(qb, sb, N, K, 1, 32, "b")
    cdt = _c_dtype(c, out_dtype)
    if c is None:
        c = torch.empty((M, N), dtype=out_dtype, device=qa.device)
    ldc = c.stride(0) if ldc is None else ldc
    _matrix_out(c, M, N, ldc)
    if workspace is False and cdt == DTYPE_F32:
        _check(lib().mxfp4_gemm(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K, _ptr(c), ldc,
                                _stream(qa, stream)))
        return c
    ws, nbytes = _workspace(workspace, M, N, K, 32, qa.device)
    _check(lib().mxfp4_gemm_ex(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K, _ptr(c), cdt,
                               ldc, _ptr(ws), nbytes, _stream(qa, stream)))
    return c


def mxfp4_gemm_noalloc(qa: torch.Tensor, sa: torch.Tensor, qb: torch.Tensor, sb: torch.Tensor,
                       M: int, N: int, K: int, *, c=None, ldc: int | None = None, stream=None):
    """mxfp4_gemm on the scale-image path with the library's static scratch
    (no workspace, no allocation); fp32 C."""
    _check_operands(qa, sa, qb, sb)
    _operand(qa, sa, M, K, 1, 32, "a")
    _operand(qb, sb, N, K, 1, 32, "b")
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=qa.device)
    if c.dtype != torch.float32:
        raise TypeError("c must be float32")
    ldc = c.stride(0) if ldc is None else ldc
    _matrix_out(c, M, N, ldc)
    _check(lib().mxfp4_gemm_noalloc(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K, _ptr(c), ldc,
                                    _stream(qa, stream)))
    return c


def mxfp8_gemm(qa: torch.Tensor, sa: torch.Tensor, qb: torch.Tensor, sb: torch.Tensor,
               M: int, N: int, K: int, *, c=None, ldc: int | None = None,
               out_dtype: torch.dtype = torch.float32, elem_format: int = FORMAT_E4M3,
               stream=None):
    """C[M, N] = deq(A) deq(B)^T for MXFP8 operands: E4M3 (or, with
    elem_format=FORMAT_E5M2, E5M2) codes [M, K] / [N, K], E8M0 scales in
    tensor-core layout; C fp32 or bf16 as in mxfp4_gemm."""
    _check_operands(qa, sa, qb, sb)
    _operand(qa, sa, M, K, 2, 32, "a")
    _operand(qb, sb, N, K, 2, 32, "b")
    cdt = _c_dtype(c, out_dtype)
    if c is None:
        c = torch.empty((M, N), dtype=out_dtype, device=qa.device)
    ldc = c.stride(0) if ldc is None else ldc
    _matrix_out(c, M, N, ldc)
    if elem_format == FORMAT_E4M3:
        _check(lib().mxfp8_gemm(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K, _ptr(c), cdt, ldc,
                                _stream(qa, stream)))
    else:
        _check(lib().mxfp8_gemm_ex(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K, elem_format,
                                   _ptr(c), cdt, ldc, _stream(qa, stream)))
    return c


def nvfp4_gemm(qa: torch.Tensor, sa: torch.Tensor, ka: int, qb: torch.Tensor, sb: torch.Tensor,
               kb: int, M: int, N: int, K: int, *, c=None, ldc: int | None = None,
               out_dtype: torch.dtype = torch.float32, workspace=None, stream=None):
    """C[M, N] = 2^(ka + kb) deq(A) deq(B)^T for NVFP4 operands: E2M1 codes [M, K/2] /
    [N, K/2], E4M3 scales per 16 in tensor-core layout, ka / kb their tensor_exp.
    `workspace` as in mxfp4_gemm (False: none)."""
    _check_operands(qa, sa, qb, sb)
    _operand(qa, sa, M, K, 1, 16, "a")
    _operand(qb, sb, N, K, 1, 16, "b")
    cdt = _c_dtype(c, out_dtype)
    if c is None:
        c = torch.empty((M, N), dtype=out_dtype, device=qa.device)
    ldc = c.stride(0) if ldc is None else ldc
    _matrix_out(c, M, N, ldc)
    ws, nbytes = _workspace(workspace, M, N, K, 16, qa.device)
    _check(lib().nvfp4_gemm(_ptr(qa), _ptr(sa), ka, _ptr(qb), _ptr(sb), kb, M, N, K, _ptr(c), cdt,
                            ldc, _ptr(ws), nbytes, _stream(qa, stream)))
    return c


def mxfp4_gemm_quantize(qa: torch.Tensor, sa: torch.Tensor, qb: torch.Tensor, sb: torch.Tensor,
                        M: int, N: int, K: int, out: QuantParams | None = None, *,
                        col: QuantParams | None = None, with_c: bool = False, c=None,
                        out_dtype: torch.dtype = torch.float32, q_out=None, s_out=None,
                        q_col=None, s_col=None, workspace=None, stream=None):
    """GEMM whose epilogue quantizes C: row-wise with `out` and/or column-wise
    (C^T along M) with `col`. Returns (q_out, s_out, c) when only `out` is
    given, else (q_out, s_out, q_col, s_col, c) (None for an orientation not
    asked for); c is None unless with_c (or c given; fp32 or bf16). The codes
    and scales equal mxfp4_quantize(C, out, col) of the fp32 C."""
    _check_operands(qa, sa, qb, sb)
    if out is None and col is None:
        raise ValueError("out (row-wise) or col params are required")
    cdt = _c_dtype(c, out_dtype)
    if c is None and with_c:
        c = torch.empty((M, N), dtype=out_dtype, device=qa.device)
    if out is not None:
        q_out = torch.empty((M, out.code_cols(N)), dtype=torch.uint8, device=qa.device) if q_out is None else q_out
        s_out = _scales_out(M, N, out, qa.device) if s_out is None else s_out
    if col is not None:
        q_col = torch.empty((N, col.code_cols(M)), dtype=torch.uint8, device=qa.device) if q_col is None else q_col
        s_col = _scales_out(N, M, col, qa.device) if s_col is None else s_col
    _operand(qa, sa, M, K, 1, 32, "a")
    _operand(qb, sb, N, K, 1, 32, "b")
    if out is not None:
        _buffer(q_out, M * out.code_cols(N), torch.uint8, "q_out")
        _buffer(s_out, scale_numel(M, N, out.block), torch.uint8, "s_out")
    if col is not None:
        _buffer(q_col, N * col.code_cols(M), torch.uint8, "q_col")
        _buffer(s_col, scale_numel(N, M, col.block), torch.uint8, "s_col")
    ldc = c.stride(0) if c is not None else N
    if c is not None:
        _matrix_out(c, M, N, ldc)
    op = out._c() if out is not None else None
    cp = col._c() if col is not None else None
    ws, nbytes = _workspace(workspace if col is None else False, M, N, K, 32, qa.device)
    _check(lib().mxfp4_gemm_quantize(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K,
                                     _ptr(c) if c is not None else None, cdt, ldc,
                                     ctypes.byref(op) if op is not None else None,
                                     _ptr(q_out if out is not None else None),
                                     _ptr(s_out if out is not None else None),
                                     ctypes.byref(cp) if cp is not None else None,
                                     _ptr(q_col if col is not None else None),
                                     _ptr(s_col if col is not None else None),
                                     _ptr(ws), nbytes, _stream(qa, stream)))
    if col is None:
        return q_out, s_out, c
    return (q_out if out is not None else None, s_out if out is not None else None,
            q_col, s_col, c)


def hadamard32(x: torch.Tensor, sign_mask: int = 0, inverse: bool = False, *, y=None, stream=None):
    _cuda2d(x, "x")
    dt = DTYPE_BF16 if x.dtype == torch.bfloat16 else DTYPE_F32
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("x must be bfloat16 or float32")
    rows, cols = x.shape
    ld = x.stride(0) if rows > 1 else cols
    y = torch.empty((rows, cols), dtype=torch.float32, device=x.device) if y is None else y
    _buffer(y, rows * cols, torch.float32, "y")
    _check(lib().hadamard32(_ptr(x), dt, rows, cols, ld, sign_mask & 0xFFFFFFFF, int(bool(inverse)),
                            _ptr(y), _stream(x, stream)))
    return y


def tensor_amax(x: torch.Tensor, *, amax=None, tensor_exp=None, stream=None):
    """Device max |x| and NVFP4 per-tensor exponent (the smallest k with
    2688 * 2^k >= max |x|): returns (amax, tensor_exp) as one-element CUDA
    tensors (float32, int32), filled asynchronously on the stream."""
    _cuda2d(x, "x")
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("x must be bfloat16 or float32")
    dt = DTYPE_BF16 if x.dtype == torch.bfloat16 else DTYPE_F32
    rows, cols = x.shape
    ld = x.stride(0) if rows > 1 else cols
    amax = torch.empty(1, dtype=torch.float32, device=x.device) if amax is None else amax
    tensor_exp = torch.empty(1, dtype=torch.int32, device=x.device) if tensor_exp is None else tensor_exp
    _buffer(amax, 1, torch.float32, "amax")
    _buffer(tensor_exp, 1, torch.int32, "tensor_exp")
    _check(lib().mxfp4_tensor_amax(_ptr(x), dt, rows, cols, ld, _ptr(amax), _ptr(tensor_exp),
                                   _stream(x, stream)))
    return amax, tensor_exp


def nvfp4_tensor_exp(x: torch.Tensor, stream=None) -> int:
    """The NVFP4 per-tensor exponent of x from tensor_amax, read back to the
    host (synchronizes the stream)."""
    _, k = tensor_amax(x, stream=stream)
    return int(k.item())


def device_status(stream=None) -> int:
    """Synchronizes the stream and returns (and clears) the GEMM's device error word."""
    s = torch.cuda.current_stream() if stream is None else stream
    return int(lib().mxfp4_device_status(ctypes.c_void_p(s.cuda_stream)))


def selftest_wait_timeout(stream=None) -> None:
    """Enqueue the bounded-wait self-test (a wait that can only run out); its
    outcome, MXFP4_ERR_TIMEOUT, is then read with device_status()."""
    s = torch.cuda.current_stream() if stream is None else stream
    _check(lib().mxfp4_selftest_wait_timeout(ctypes.c_void_p(s.cuda_stream)))
