"""MXFP8 GEMM (E4M3 operands, E8M0 scales per 32 elements) against the fp64
product of the oracle's dequantized operands."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _codes(rows, k, seed):
    """Random finite E4M3 codes (0x7F / 0xFF are NaN)."""
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 256, size=(rows, k), dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38          # replace NaN codes by 1.0
    return c


def _scales(rows, k, seed, lo=118, hi=136):
    rng = np.random.default_rng(seed)
    s = rng.integers(lo, hi, size=(rows, k // 32), dtype=np.uint8)
    return oracle.scales_to_mma(s), s


def _run(qa, sa, qb, sb, M, N, K):
    import gemm_pt_block_gb300 as mx

    t = [torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (qa, sa, qb, sb)]
    c = mx.mxfp8_gemm(*t, M, N, K)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    return c.cpu().numpy().astype(np.float64)


def test_mxfp8_gemm_all_ones_exact():
    M, N, K = 256, 256, 128
    qa = np.full((M, K), 0x38, np.uint8)           # E4M3 1.0
    qb = np.full((N, K), 0x38, np.uint8)
    s = oracle.scales_to_mma(np.full((256, K // 32), 127, np.uint8))
    c = _run(qa, s, qb, s, M, N, K)
    assert np.all(c == K)


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (256, 512, 384), (512, 768, 1024), (1024, 1280, 2048),
                                   (128, 128, 128), (128, 384, 384), (384, 640, 1152), (640, 384, 256)])
def test_mxfp8_gemm_random_within_tolerance(M, N, K):
    qa, qb = _codes(M, K, M + 1), _codes(N, K, N + 2)
    sa, sa_rm = _scales(M, K, K + 3)
    sb, sb_rm = _scales(N, K, K + 4)
    c = _run(qa, sa, qb, sb, M, N, K)
    A = oracle.dequantize(qa, sa_rm, M, K, f64=True, fmt=oracle.FORMAT_E4M3)
    B = oracle.dequantize(qb, sb_rm, N, K, f64=True, fmt=oracle.FORMAT_E4M3)
    ref, ab = A @ B.T, np.abs(A) @ np.abs(B).T
    assert np.all(np.abs(c - ref) <= 1e-5 * ab + 1e-30)


def test_mxfp8_quantize_then_gemm_end_to_end():
    """Quantize bf16 X and W to MXFP8 on the GPU and multiply: equals the fp64
    product of the dequantized codes, and is close to the bf16 product."""
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 256, 512
    g = torch.Generator().manual_seed(5)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = torch.randn(N, K, generator=g).to(torch.bfloat16)
    p = mx.QuantParams(mx.BLOCK_1X32, mx.SCALE_ROUNDUP, mx.ROUND_RTN, mx.LAYOUT_MMA,
                       elem_format=mx.FORMAT_E4M3)
    qx, sx, _, _ = mx.mxfp4_quantize(x.to(DEV), p)
    qw, sw, _, _ = mx.mxfp4_quantize(w.to(DEV), p)
    c = mx.mxfp8_gemm(qx, sx, qw, sw, M, N, K).cpu().numpy().astype(np.float64)
    A = oracle.dequantize(qx.cpu().numpy(), sx.cpu().numpy(), M, K, oracle.LAYOUT_MMA, True,
                          oracle.FORMAT_E4M3)
    B = oracle.dequantize(qw.cpu().numpy(), sw.cpu().numpy(), N, K, oracle.LAYOUT_MMA, True,
                          oracle.FORMAT_E4M3)
    ref, ab = A @ B.T, np.abs(A) @ np.abs(B).T
    assert np.all(np.abs(c - ref) <= 1e-5 * ab + 1e-30)
    exact = x.double().numpy() @ w.double().numpy().T
    rel = np.linalg.norm(c - exact) / np.linalg.norm(exact)
    assert rel < 0.05                      # E4M3 keeps ~3 mantissa bits


def test_mxfp8_gemm_rejects_bad_shapes():
    import gemm_pt_block_gb300 as mx

    z = torch.zeros(128 * 128, dtype=torch.uint8, device=DEV)
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp8_gemm(z, z, z, z, 64, 128, 128)       # M % 128 != 0
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp8_gemm(z, z, z, z, 128, 128, 96)       # K % 128 != 0
