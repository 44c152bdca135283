"""CPU oracle for the MXFP4 hot path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, independent restatement of what the CUDA library computes
(see ``mxfp4_oracle.c`` for the definitions and the pages each step follows).
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the product path never does.

The GEMM reference is the fp64 sum of dequantized products, computed either
by brute force for listed output elements (``gemm_pairs``) or as a dequantize
followed by a numpy fp64 matrix product (``gemm_ref``), the library primitive
standing in for the plain triple loop.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_mxfp4.so")

BLOCK_1X32, BLOCK_32X32, BLOCK_64X64, BLOCK_1X16 = 0, 1, 2, 3
FORMAT_E2M1, FORMAT_E4M3, FORMAT_E5M2 = 0, 1, 2
SCALE_FLOOR, SCALE_ROUNDUP = 0, 1
ROUND_RTN, ROUND_SR = 0, 1
LAYOUT_ROWMAJOR, LAYOUT_MMA = 0, 1
DTYPE_BF16, DTYPE_F32 = 0, 1

GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def build(force: bool = False) -> str:
    """Compile the C oracle in place (plain gcc, IEEE fp32, no contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "mxfp4_oracle.h"))
    ):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = [
            os.environ.get("CC", "gcc"), "-O2", "-std=c99", "-ffp-contract=off",
            "-fno-fast-math", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Params(ctypes.Structure):
    _fields_ = [
        ("block", ctypes.c_int),
        ("scale_mode", ctypes.c_int),
        ("rounding", ctypes.c_int),
        ("scale_layout", ctypes.c_int),
        ("wht", ctypes.c_int),
        ("wht_sign_mask", ctypes.c_uint32),
        ("seed", ctypes.c_uint64),
        ("sr_stream", ctypes.c_uint32),
        ("elem_format", ctypes.c_int),
        ("tensor_exp", ctypes.c_int),
    ]


@dataclass(frozen=True)
class Params:
    block: int = BLOCK_1X32
    scale_mode: int = SCALE_FLOOR
    rounding: int = ROUND_RTN
    wht: bool = False
    wht_sign_mask: int = 0
    seed: int = 0
    sr_stream: int = 0
    elem_format: int = 0        # FORMAT_E2M1 (MXFP4), FORMAT_E4M3 or FORMAT_E5M2 (MXFP8)
    tensor_exp: int = 0         # BLOCK_1X16 (NVFP4): per-tensor factor 2^tensor_exp

    def _c(self) -> _Params:
        return _Params(self.block, self.scale_mode, self.rounding, LAYOUT_ROWMAJOR,
                       int(bool(self.wht)), self.wht_sign_mask & 0xFFFFFFFF,
                       self.seed & 0xFFFFFFFFFFFFFFFF, self.sr_stream & 0xFFFFFFFF,
                       self.elem_format, self.tensor_exp)

    def scale_cols(self, k: int) -> int:
        """Scale bytes per output row for quantization axis length k."""
        return k // 16 if self.block == BLOCK_1X16 else k // 32


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        L.orc_e2m1_value.restype = ctypes.c_float
        L.orc_e2m1_value.argtypes = [ctypes.c_int]
        L.orc_philox4x32_10.argtypes = [P, P, P]
        L.orc_sr_bits.restype = ctypes.c_uint32
        L.orc_sr_bits.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64]
        L.orc_wht32.argtypes = [P, ctypes.c_uint32, ctypes.c_int, P]
        L.orc_scale_exponent.restype = ctypes.c_int
        L.orc_scale_exponent.argtypes = [ctypes.c_float, ctypes.c_int]
        L.orc_round_rtn.restype = ctypes.c_int
        L.orc_round_rtn.argtypes = [ctypes.c_float]
        L.orc_round_sr.restype = ctypes.c_int
        L.orc_round_sr.argtypes = [ctypes.c_float, ctypes.c_uint32]
        L.orc_e4m3_value.restype = ctypes.c_float
        L.orc_e4m3_value.argtypes = [ctypes.c_int]
        L.orc_round_e4m3_rtn.restype = ctypes.c_int
        L.orc_round_e4m3_rtn.argtypes = [ctypes.c_float]
        L.orc_scale_exponent_fmt.restype = ctypes.c_int
        L.orc_scale_exponent_fmt.argtypes = [ctypes.c_float, ctypes.c_int, ctypes.c_int]
        L.orc_dequantize_e4m3_f64.restype = ctypes.c_int
        L.orc_dequantize_e4m3_f64.argtypes = [P, P, ctypes.c_int, i64, i64, P]
        L.orc_dequantize_fp8_f64.restype = ctypes.c_int
        L.orc_dequantize_fp8_f64.argtypes = [P, P, ctypes.c_int, i64, i64, ctypes.c_int, P]
        L.orc_e5m2_value.restype = ctypes.c_float
        L.orc_e5m2_value.argtypes = [ctypes.c_int]
        L.orc_round_e5m2_rtn.restype = ctypes.c_int
        L.orc_round_e5m2_rtn.argtypes = [ctypes.c_float]
        for fn in (L.orc_quantize_rows, L.orc_quantize_cols):
            fn.restype = ctypes.c_int
            fn.argtypes = [P, ctypes.c_int, i64, i64, i64, ctypes.POINTER(_Params), i64, i64, P, P]
        L.orc_mma_scale_offset.restype = i64
        L.orc_mma_scale_offset.argtypes = [i64, i64, i64, i64]
        L.orc_scales_to_mma.restype = ctypes.c_int
        L.orc_scales_to_mma.argtypes = [P, i64, i64, P]
        for fn in (L.orc_dequantize_f32, L.orc_dequantize_f64):
            fn.restype = ctypes.c_int
            fn.argtypes = [P, P, ctypes.c_int, i64, i64, P]
        L.orc_hadamard32.restype = ctypes.c_int
        L.orc_hadamard32.argtypes = [P, ctypes.c_int, i64, i64, i64, ctypes.c_uint32, ctypes.c_int, P]
        L.orc_gemm_pairs.restype = ctypes.c_int
        L.orc_gemm_pairs.argtypes = [P, P, P, P, ctypes.c_int, i64, i64, i64, i64, P, P, P, P]
        L.orc_nv_scale_code.restype = ctypes.c_int
        L.orc_nv_scale_code.argtypes = [ctypes.c_float, ctypes.c_int, ctypes.c_int]
        L.orc_dequantize_nv_f64.restype = ctypes.c_int
        L.orc_dequantize_nv_f64.argtypes = [P, P, ctypes.c_int, i64, i64, ctypes.c_int, P]
        L.orc_tensor_amax.restype = ctypes.c_float
        L.orc_tensor_amax.argtypes = [P, ctypes.c_int, i64, i64, i64]
        L.orc_nv_tensor_exp.restype = ctypes.c_int
        L.orc_nv_tensor_exp.argtypes = [ctypes.c_float]
        L.orc_gemm_pairs_nv.restype = ctypes.c_int
        L.orc_gemm_pairs_nv.argtypes = [P, P, ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int,
                                        i64, i64, i64, i64, P, P, P, P]
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def _as_input(x: np.ndarray):
    """x: uint16 array of bf16 bit patterns, or float32. Returns (array, dtype, ld)."""
    if x.dtype == np.uint16:
        dt = DTYPE_BF16
    elif x.dtype == np.float32:
        dt = DTYPE_F32
    else:
        raise TypeError("oracle input must be bf16 bits (uint16) or float32")
    if x.ndim != 2 or x.strides[1] != x.itemsize or x.strides[0] % x.itemsize:
        raise ValueError("oracle input must be 2-D with unit column stride")
    return x, dt, x.strides[0] // x.itemsize


# ------------------------------------------------------------------ scalars --

def e2m1_value(code: int) -> float:
    return float(lib().orc_e2m1_value(code))


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return [int(v) for v in out]


def sr_bits(seed: int, stream: int, i: int) -> int:
    return int(lib().orc_sr_bits(seed, stream, i))


def wht32(v, sign_mask: int = 0, inverse: bool = False) -> np.ndarray:
    a = np.ascontiguousarray(v, dtype=np.float32)
    assert a.shape == (32,)
    out = np.zeros(32, dtype=np.float32)
    lib().orc_wht32(_ptr(a), sign_mask & 0xFFFFFFFF, int(inverse), _ptr(out))
    return out


def scale_exponent(M: float, mode: int) -> int:
    return int(lib().orc_scale_exponent(ctypes.c_float(M), mode))


def round_rtn(v: float) -> int:
    return int(lib().orc_round_rtn(ctypes.c_float(v)))


def e4m3_value(code: int) -> float:
    return float(lib().orc_e4m3_value(code))


def round_e4m3_rtn(v: float) -> int:
    return int(lib().orc_round_e4m3_rtn(ctypes.c_float(v)))


def e5m2_value(code: int) -> float:
    return float(lib().orc_e5m2_value(code))


def round_e5m2_rtn(v: float) -> int:
    return int(lib().orc_round_e5m2_rtn(ctypes.c_float(v)))


def scale_exponent_fmt(M: float, mode: int, fmt: int) -> int:
    return int(lib().orc_scale_exponent_fmt(ctypes.c_float(M), mode, fmt))


def round_sr(v: float, r16: int) -> int:
    return int(lib().orc_round_sr(ctypes.c_float(v), r16))


def tensor_amax(x: np.ndarray) -> float:
    """Largest |x| over a 2-D bf16-bits (uint16) or float32 array."""
    x, dt, ld = _as_input(x)
    rows, cols = x.shape
    return float(lib().orc_tensor_amax(_ptr(x), dt, rows, cols, ld))


def nv_tensor_exp(amax: float) -> int:
    """NVFP4 per-tensor exponent: smallest k with 2688 * 2^k >= amax (0 for 0)."""
    return int(lib().orc_nv_tensor_exp(ctypes.c_float(amax)))


def nv_scale_code(M: float, k: int, mode: int) -> int:
    """E4M3 code of the NVFP4 block scale for block max-abs M under factor 2^k."""
    return int(lib().orc_nv_scale_code(ctypes.c_float(M), k, mode))


# ------------------------------------------------------------------ tensors --

def quantize_rows(x: np.ndarray, p: Params, r0: int = 0, r1: int | None = None):
    """Row-wise codes [r1-r0, cols/2] and row-major scales [r1-r0, cols/32]."""
    x, dt, ld = _as_input(x)
    rows, cols = x.shape
    r1 = rows if r1 is None else r1
    q = np.zeros((r1 - r0, cols if p.elem_format in (FORMAT_E4M3, FORMAT_E5M2) else cols // 2),
                 dtype=np.uint8)
    s = np.zeros((r1 - r0, p.scale_cols(cols)), dtype=np.uint8)
    cp = p._c()
    rc = lib().orc_quantize_rows(_ptr(x), dt, rows, cols, ld, ctypes.byref(cp), r0, r1, _ptr(q), _ptr(s))
    if rc:
        raise ValueError(f"oracle quantize_rows failed ({rc})")
    return q, s


def quantize_cols(x: np.ndarray, p: Params, c0: int = 0, c1: int | None = None):
    """Column-wise codes [c1-c0, rows/2] and row-major scales [c1-c0, rows/32]."""
    x, dt, ld = _as_input(x)
    rows, cols = x.shape
    c1 = cols if c1 is None else c1
    q = np.zeros((c1 - c0, rows if p.elem_format in (FORMAT_E4M3, FORMAT_E5M2) else rows // 2),
                 dtype=np.uint8)
    s = np.zeros((c1 - c0, p.scale_cols(rows)), dtype=np.uint8)
    cp = p._c()
    rc = lib().orc_quantize_cols(_ptr(x), dt, rows, cols, ld, ctypes.byref(cp), c0, c1, _ptr(q), _ptr(s))
    if rc:
        raise ValueError(f"oracle quantize_cols failed ({rc})")
    return q, s


def mma_scale_offset(r: int, kb: int, rows: int, nkb: int) -> int:
    return int(lib().orc_mma_scale_offset(r, kb, rows, nkb))


def scales_to_mma(s: np.ndarray) -> np.ndarray:
    s = np.ascontiguousarray(s, dtype=np.uint8)
    rows, nkb = s.shape
    out = np.zeros(rows * nkb, dtype=np.uint8)
    if lib().orc_scales_to_mma(_ptr(s), rows, nkb, _ptr(out)):
        raise ValueError("scales_to_mma needs rows % 128 == 0 and nkb % 4 == 0")
    return out


def dequantize(q: np.ndarray, s: np.ndarray, rows: int, cols: int,
               layout: int = LAYOUT_ROWMAJOR, f64: bool = False, fmt: int = FORMAT_E2M1) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    if fmt in (FORMAT_E4M3, FORMAT_E5M2):
        out = np.zeros((rows, cols), dtype=np.float64)
        if lib().orc_dequantize_fp8_f64(_ptr(q), _ptr(s), layout, rows, cols, fmt, _ptr(out)):
            raise ValueError("oracle dequantize: bad shape")
        return out if f64 else out.astype(np.float32)
    out = np.zeros((rows, cols), dtype=np.float64 if f64 else np.float32)
    fn = lib().orc_dequantize_f64 if f64 else lib().orc_dequantize_f32
    if fn(_ptr(q), _ptr(s), layout, rows, cols, _ptr(out)):
        raise ValueError("oracle dequantize: bad shape")
    return out


def dequantize_nv(q: np.ndarray, s: np.ndarray, rows: int, cols: int, tensor_exp: int = 0,
                  layout: int = LAYOUT_ROWMAJOR) -> np.ndarray:
    """NVFP4 reconstruction (fp64): E2M1 code x E4M3 scale x 2^tensor_exp."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    out = np.zeros((rows, cols), dtype=np.float64)
    if lib().orc_dequantize_nv_f64(_ptr(q), _ptr(s), layout, rows, cols, tensor_exp, _ptr(out)):
        raise ValueError("oracle dequantize_nv: bad shape")
    return out


def hadamard32(x: np.ndarray, sign_mask: int = 0, inverse: bool = False) -> np.ndarray:
    x, dt, ld = _as_input(x)
    rows, cols = x.shape
    y = np.zeros((rows, cols), dtype=np.float32)
    if lib().orc_hadamard32(_ptr(x), dt, rows, cols, ld, sign_mask & 0xFFFFFFFF, int(inverse), _ptr(y)):
        raise ValueError("oracle hadamard32: bad shape")
    return y


def gemm_pairs(qa, sa, qb, sb, M, N, K, ms, ns, layout=LAYOUT_MMA):
    """Brute-force fp64 C[m, n] and sum_k |a*b| for the listed (m, n)."""
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    c = np.zeros(len(ms), dtype=np.float64)
    a = np.zeros(len(ms), dtype=np.float64)
    arrs = [np.ascontiguousarray(t, dtype=np.uint8) for t in (qa, sa, qb, sb)]
    rc = lib().orc_gemm_pairs(*[_ptr(t) for t in arrs], layout, M, N, K, len(ms),
                              _ptr(ms), _ptr(ns), _ptr(c), _ptr(a))
    if rc:
        raise ValueError(f"oracle gemm_pairs failed ({rc})")
    return c, a


def gemm_ref(qa, sa, qb, sb, M, N, K, layout=LAYOUT_MMA, rows=None):
    """fp64 reference C = deq(A) deq(B)^T and the tolerance base sum_k |a*b|.

    ``rows`` restricts the output to a subset of A's rows (all of B is used).
    """
    A = dequantize(qa, sa, M, K, layout, f64=True)
    B = dequantize(qb, sb, N, K, layout, f64=True)
    if rows is not None:
        A = A[np.asarray(rows)]
    return A @ B.T, np.abs(A) @ np.abs(B).T


def gemm_ref_nv(qa, sa, ka, qb, sb, kb, M, N, K, layout=LAYOUT_MMA):
    """fp64 reference C = deq(A) deq(B)^T for NVFP4 operands (per-tensor
    factors 2^ka, 2^kb) and the tolerance base sum_k |a*b|."""
    A = dequantize_nv(qa, sa, M, K, ka, layout)
    B = dequantize_nv(qb, sb, N, K, kb, layout)
    return A @ B.T, np.abs(A) @ np.abs(B).T


def gemm_pairs_nv(qa, sa, ka, qb, sb, kb, M, N, K, ms, ns, layout=LAYOUT_MMA):
    """Brute-force fp64 C[m, n] and sum_k |a*b| of NVFP4 operands for listed (m, n)."""
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    c = np.zeros(len(ms), dtype=np.float64)
    a = np.zeros(len(ms), dtype=np.float64)
    qa, sa, qb, sb = [np.ascontiguousarray(t, dtype=np.uint8) for t in (qa, sa, qb, sb)]
    rc = lib().orc_gemm_pairs_nv(_ptr(qa), _ptr(sa), ka, _ptr(qb), _ptr(sb), kb, layout, M, N, K,
                                 len(ms), _ptr(ms), _ptr(ns), _ptr(c), _ptr(a))
    if rc:
        raise ValueError(f"oracle gemm_pairs_nv failed ({rc})")
    return c, a
