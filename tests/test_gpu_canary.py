"""Guard bands around every output: nothing writes outside its buffer.

Each call's outputs (and the GEMM's workspace) are carved out of one device
arena filled with 0xA5, with 4 KB guard bands between and around them; for a
C with ldc > N the columns past N of every row are guard bytes too. After the
call every byte outside the bytes the call may write must still be 0xA5. The
shapes are ragged against the kernels' tiles (64 x 64 quantizer tiles,
256 x 256 GEMM tiles, 128-row GEMM tiles) so the edge masking is exercised.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import cuda_params

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GUARD = 4096
FILL = 0xA5


class Arena:
    """Regions of given byte sizes inside one 0xA5-filled buffer, 256-byte
    aligned, separated by GUARD bytes; `allow` marks the bytes a call may write."""

    def __init__(self, sizes):
        self.offs, off = [], GUARD
        for s in sizes:
            self.offs.append(off)
            off += (s + 255) // 256 * 256 + GUARD
        self.buf = torch.full((off,), FILL, dtype=torch.uint8, device=DEV)
        self.allowed = np.zeros(off, dtype=bool)

    def region(self, i, dtype, shape, writable=None):
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        t = self.buf[self.offs[i]:self.offs[i] + n].view(dtype).view(*shape)
        if writable is None:
            self.allowed[self.offs[i]:self.offs[i] + n] = True
        else:
            for a, b in writable:
                self.allowed[self.offs[i] + a:self.offs[i] + b] = True
        return t

    def check(self, what):
        torch.cuda.synchronize()
        b = self.buf.cpu().numpy()
        bad = np.flatnonzero((b != FILL) & ~self.allowed)
        assert bad.size == 0, f"{what}: {bad.size} guard bytes written, first at arena offset {bad[0]}"


def _scale_bytes(rows, k, p):
    return rows * (k // 16 if p.block == oracle.BLOCK_1X16 else k // 32)


def _code_bytes(rows, k, p):
    return rows * (k if p.elem_format in (oracle.FORMAT_E4M3, oracle.FORMAT_E5M2) else k // 2)


QUANT_CASES = [
    # (rows, cols, row params, col params, layout)
    (150, 352, oracle.Params(), None, 0),                                           # row kernel, ragged rows
    (150, 352, oracle.Params(rounding=oracle.ROUND_SR, wht=True, wht_sign_mask=9), None, 0),
    (256, 384, oracle.Params(), None, 1),                                           # row kernel, MMA layout
    (160, 352, oracle.Params(block=oracle.BLOCK_32X32, scale_mode=oracle.SCALE_ROUNDUP),
     oracle.Params(block=oracle.BLOCK_32X32, scale_mode=oracle.SCALE_ROUNDUP), 0),  # weights profile
    (160, 352, oracle.Params(), oracle.Params(rounding=oracle.ROUND_SR, wht=True, seed=2), 0),  # activations
    (160, 352, oracle.Params(rounding=oracle.ROUND_SR, seed=3, sr_stream=1),
     oracle.Params(rounding=oracle.ROUND_SR, wht=True, seed=3, sr_stream=1), 0),   # gradients
    (256, 384, oracle.Params(block=oracle.BLOCK_32X32, rounding=oracle.ROUND_SR, seed=4),
     oracle.Params(block=oracle.BLOCK_32X32, rounding=oracle.ROUND_SR, seed=4), 1),
    (192, 320, oracle.Params(block=oracle.BLOCK_64X64), oracle.Params(block=oracle.BLOCK_64X64), 0),
    (160, 352, None, oracle.Params(elem_format=oracle.FORMAT_E4M3), 0),
    (150, 352, oracle.Params(elem_format=oracle.FORMAT_E5M2, wht=True, wht_sign_mask=5),
     None, 0),
    (256, 384, oracle.Params(elem_format=oracle.FORMAT_E5M2, block=oracle.BLOCK_32X32),
     oracle.Params(elem_format=oracle.FORMAT_E5M2, block=oracle.BLOCK_32X32), 1),
    (160, 352, oracle.Params(block=oracle.BLOCK_1X16, tensor_exp=-3),
     oracle.Params(block=oracle.BLOCK_1X16, tensor_exp=-3, rounding=oracle.ROUND_SR), 0),
]


@pytest.mark.parametrize("case", range(len(QUANT_CASES)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantizer_writes_only_its_outputs(case, dtype):
    import gemm_pt_block_gb300 as mx

    rows, cols, pr, pc, layout = QUANT_CASES[case]
    x = synth.student_t(rows, cols, 3.0, seed=500 + case).to(dtype).to(DEV)
    sizes = []
    if pr:
        sizes += [_code_bytes(rows, cols, pr), _scale_bytes(rows, cols, pr)]
    if pc:
        sizes += [_code_bytes(cols, rows, pc), _scale_bytes(cols, rows, pc)]
    ar = Arena(sizes)
    i, kw = 0, {}
    if pr:
        kw["q_row"] = ar.region(0, torch.uint8, (sizes[0],))
        kw["s_row"] = ar.region(1, torch.uint8, (sizes[1],))
        i = 2
    if pc:
        kw["q_col"] = ar.region(i, torch.uint8, (sizes[i],))
        kw["s_col"] = ar.region(i + 1, torch.uint8, (sizes[i + 1],))
    mx.mxfp4_quantize(x, cuda_params(pr, layout) if pr else None,
                      cuda_params(pc, layout) if pc else None, **kw)
    ar.check(f"quantize case {case}")
    assert mx.device_status() == 0


def _operands(M, N, K, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    qa = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    qb = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    sa = torch.randint(120, 135, (M * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    sb = torch.randint(120, 135, (N * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    return qa, sa, qb, sb


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (384, 768, 1024), (768, 512, 2304),
                                   (128, 384, 384), (256, 384, 640), (512, 128, 1152)])
@pytest.mark.parametrize("c_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("images", [False, True])
def test_gemm_writes_only_c_rows_up_to_n(M, N, K, c_dtype, images):
    import gemm_pt_block_gb300 as mx

    ldc = N + 40
    esz = 4 if c_dtype == torch.float32 else 2
    ws_bytes = mx.gemm_workspace_size(M, N, K)
    ar = Arena([M * ldc * esz, ws_bytes])
    c = ar.region(0, c_dtype, (M, ldc), writable=[(m * ldc * esz, (m * ldc + N) * esz) for m in range(M)])
    ws = ar.region(1, torch.uint8, (ws_bytes,)) if images else False
    t = _operands(M, N, K, M + N + K)
    mx.mxfp4_gemm(*t, M, N, K, c=c, ldc=ldc, workspace=ws)
    ar.check(f"gemm {M}x{N}x{K}")
    assert mx.device_status() == 0
    want = mx.mxfp4_gemm(*t, M, N, K, workspace=False, out_dtype=c_dtype)
    assert torch.equal(c[:, :N], want)


@pytest.mark.parametrize("M,N,K", [(128, 384, 384), (384, 640, 1152), (256, 128, 128)])
@pytest.mark.parametrize("kind", ["nvfp4", "nvfp4-images", "mxfp8", "mxfp8-e5m2"])
def test_nvfp4_and_mxfp8_gemms_write_only_c(M, N, K, kind):
    """The NVFP4 and MXFP8 GEMMs on shapes with a last M, N or K tile of 128:
    nothing outside C's first N columns (and the NVFP4 workspace) is written."""
    import gemm_pt_block_gb300 as mx

    ldc = N + 40
    g = torch.Generator(device=DEV).manual_seed(M + N + K)
    nv = kind.startswith("nvfp4")
    kb = K // 2 if nv else K
    qa = torch.randint(0, 120, (M, kb), dtype=torch.uint8, device=DEV, generator=g)
    qb = torch.randint(0, 120, (N, kb), dtype=torch.uint8, device=DEV, generator=g)
    lo, hi = (40, 70) if nv else (120, 135)
    per = 16 if nv else 32
    sa = torch.randint(lo, hi, (M * K // per,), dtype=torch.uint8, device=DEV, generator=g)
    sb = torch.randint(lo, hi, (N * K // per,), dtype=torch.uint8, device=DEV, generator=g)
    ws_bytes = mx.gemm_workspace_size(M, N, K, 16) if kind == "nvfp4-images" else 0
    ar = Arena([M * ldc * 4, max(ws_bytes, 16)])
    c = ar.region(0, torch.float32, (M, ldc), writable=[(m * ldc * 4, (m * ldc + N) * 4) for m in range(M)])
    if nv:
        ws = ar.region(1, torch.uint8, (ws_bytes,)) if ws_bytes else False
        mx.nvfp4_gemm(qa, sa, -2, qb, sb, 1, M, N, K, c=c, ldc=ldc, workspace=ws)
        want = mx.nvfp4_gemm(qa, sa, -2, qb, sb, 1, M, N, K, workspace=False)
    else:
        fmt = mx.FORMAT_E5M2 if kind.endswith("e5m2") else mx.FORMAT_E4M3
        mx.mxfp8_gemm(qa, sa, qb, sb, M, N, K, c=c, ldc=ldc, elem_format=fmt)
        want = mx.mxfp8_gemm(qa, sa, qb, sb, M, N, K, elem_format=fmt)
    ar.check(f"{kind} {M}x{N}x{K}")
    assert mx.device_status() == 0
    assert torch.equal(c[:, :N], want)


@pytest.mark.parametrize("col", [False, True])
@pytest.mark.parametrize("M,N,K", [(512, 768, 1024), (256, 384, 640), (384, 640, 1152)])
def test_fused_epilogue_quantizer_writes_only_its_outputs(col, M, N, K):
    import gemm_pt_block_gb300 as mx

    p = mx.QuantParams(rounding=mx.ROUND_SR, wht=True, seed=6)
    sizes = [M * N // 2, M * N // 32] + ([N * M // 2, N * M // 32] if col else [])
    ar = Arena(sizes)
    kw = dict(q_out=ar.region(0, torch.uint8, (sizes[0],)), s_out=ar.region(1, torch.uint8, (sizes[1],)))
    if col:
        kw.update(q_col=ar.region(2, torch.uint8, (sizes[2],)), s_col=ar.region(3, torch.uint8, (sizes[3],)))
    t = _operands(M, N, K, 77)
    mx.mxfp4_gemm_quantize(*t, M, N, K, p, col=p if col else None, **kw)
    ar.check("fused epilogue")
    assert mx.device_status() == 0


def test_dequantize_and_rotation_write_only_their_outputs():
    import gemm_pt_block_gb300 as mx

    rows, cols = 96, 352
    x = synth.student_t(rows, cols, 3.0, seed=9).to(DEV)
    q, s, _, _ = mx.mxfp4_quantize(x, mx.QuantParams())
    ar = Arena([rows * cols * 4, rows * cols * 4])
    mx.mxfp4_dequantize(q, s, rows, cols, out=ar.region(0, torch.float32, (rows, cols)))
    mx.hadamard32(x, 0x1234, y=ar.region(1, torch.float32, (rows, cols)))
    ar.check("dequantize / hadamard32")
