"""MXFP8 with E5M2 elements (the other OCP FP8 format): the quantizer, the
reconstruction and the E5M2 GEMM against the oracle, and the fused GEMM
epilogue with E5M2 output against the stand-alone quantizer."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import assert_same, gpu_quantize, oracle_input, oracle_quantize

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
E5 = oracle.FORMAT_E5M2


def _input(rows, cols, dtype, seed):
    x = synth.laplace(rows, cols, 1e-3, seed=seed, outlier_frac=0.01)
    x[:, 3] *= 1e4                    # an outlier channel: wide exponent range in a block
    return x if dtype == "bf16" else x.float()


@pytest.mark.parametrize("orient", ["row", "col", "both"])
@pytest.mark.parametrize("block", [oracle.BLOCK_1X32, oracle.BLOCK_32X32, oracle.BLOCK_64X64])
@pytest.mark.parametrize("scale", [oracle.SCALE_FLOOR, oracle.SCALE_ROUNDUP])
@pytest.mark.parametrize("wht", [(False, 0), (True, 0x5A5A5A5A)], ids=["nowht", "rndwht"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_e5m2_quantize_matches_oracle(orient, block, scale, wht, dtype):
    rows, cols = (192, 320) if block == oracle.BLOCK_64X64 else (160, 352)
    if orient == "row" and block == oracle.BLOCK_1X32:
        rows = 150                    # row kernel, ragged row count
    x = _input(rows, cols, dtype, seed=201 + block)
    p = oracle.Params(block=block, scale_mode=scale, wht=wht[0], wht_sign_mask=wht[1], elem_format=E5)
    prow = p if orient in ("row", "both") else None
    pcol = p if orient in ("col", "both") else None
    assert_same(gpu_quantize(x.to(DEV), prow, pcol), oracle_quantize(oracle_input(x), prow, pcol),
                f"e5m2 {orient}")


def test_e5m2_every_bf16_value_and_mma_layout():
    bits = np.arange(65536, dtype=np.uint32)
    keep = (bits & 0x7F80) != 0x7F80
    vals = bits[keep].astype(np.uint16)
    n = (vals.size // 64) * 64
    x = vals[:n].reshape(-1, 64)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    for mode in (oracle.SCALE_FLOOR, oracle.SCALE_ROUNDUP):
        p = oracle.Params(elem_format=E5, scale_mode=mode)
        assert_same(gpu_quantize(xt.to(DEV), p, None), oracle_quantize(x, p, None), "e5m2 bf16 sweep")
    xm = _input(256, 384, "bf16", seed=203)
    pm = oracle.Params(block=oracle.BLOCK_32X32, elem_format=E5)
    assert_same(gpu_quantize(xm.to(DEV), pm, pm, 1, 1), oracle_quantize(oracle_input(xm), pm, pm, 1, 1),
                "e5m2 mma")


def test_e5m2_dequantize_every_code():
    import gemm_pt_block_gb300 as mx

    rows, cols = 64, 256
    q = np.tile(np.arange(256, dtype=np.uint8), rows * cols // 256).reshape(rows, cols)
    s = np.random.default_rng(5).integers(100, 160, size=(rows, cols // 32), dtype=np.uint8)
    p = mx.QuantParams(elem_format=mx.FORMAT_E5M2)
    got = mx.mxfp4_dequantize(torch.from_numpy(q).to(DEV), torch.from_numpy(s).to(DEV), rows, cols,
                              params=p).cpu().numpy().astype(np.float64)
    want = oracle.dequantize(q, s, rows, cols, f64=True, fmt=E5)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])          # infinities included


def _finite_codes(rows, k, seed):
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 256, size=(rows, k), dtype=np.uint8)
    c[(c & 0x7C) == 0x7C] = 0x3C      # exponent field 31 (inf / NaN) -> 1.0
    return c


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (256, 512, 384), (512, 768, 1024)])
def test_e5m2_gemm_within_tolerance(M, N, K):
    import gemm_pt_block_gb300 as mx

    qa, qb = _finite_codes(M, K, M + 1), _finite_codes(N, K, N + 2)
    rng = np.random.default_rng(K)
    sa_rm = rng.integers(100, 130, size=(M, K // 32), dtype=np.uint8)
    sb_rm = rng.integers(100, 130, size=(N, K // 32), dtype=np.uint8)
    t = [torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
         for a in (qa, oracle.scales_to_mma(sa_rm), qb, oracle.scales_to_mma(sb_rm))]
    c = mx.mxfp8_gemm(*t, M, N, K, elem_format=mx.FORMAT_E5M2)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    A = oracle.dequantize(qa, sa_rm, M, K, f64=True, fmt=E5)
    B = oracle.dequantize(qb, sb_rm, N, K, f64=True, fmt=E5)
    ref, ab = A @ B.T, np.abs(A) @ np.abs(B).T
    got = c.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-5 * ab + 1e-30)


def test_e5m2_gemm_exact_products():
    """Powers of two with unit scales: every partial sum is exact in fp32."""
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 256, 256
    rng = np.random.default_rng(9)
    qa = (0x3C + 4 * rng.integers(-2, 3, size=(M, K))).astype(np.uint8)   # 2^-2 .. 2^2
    qb = (0x3C + 4 * rng.integers(-2, 3, size=(N, K))).astype(np.uint8)
    qb[:, ::3] |= 0x80                                                    # some negatives
    s = oracle.scales_to_mma(np.full((256, K // 32), 127, np.uint8))
    t = [torch.from_numpy(a).to(DEV) for a in (qa, s, qb, s)]
    c = mx.mxfp8_gemm(*t, M, N, K, elem_format=mx.FORMAT_E5M2).cpu().numpy().astype(np.float64)
    A = oracle.dequantize(qa, np.full((M, K // 32), 127, np.uint8), M, K, f64=True, fmt=E5)
    B = oracle.dequantize(qb, np.full((N, K // 32), 127, np.uint8), N, K, f64=True, fmt=E5)
    assert np.array_equal(c, A @ B.T)


def test_e5m2_quantize_then_gemm_and_fused_output():
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 512, 512
    g = torch.Generator().manual_seed(6)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = torch.randn(N, K, generator=g).to(torch.bfloat16)
    p = mx.QuantParams(mx.BLOCK_1X32, mx.SCALE_ROUNDUP, mx.ROUND_RTN, mx.LAYOUT_MMA,
                       elem_format=mx.FORMAT_E5M2)
    qx, sx, _, _ = mx.mxfp4_quantize(x.to(DEV), p)
    qw, sw, _, _ = mx.mxfp4_quantize(w.to(DEV), p)
    c = mx.mxfp8_gemm(qx, sx, qw, sw, M, N, K, elem_format=mx.FORMAT_E5M2)
    A = oracle.dequantize(qx.cpu().numpy(), sx.cpu().numpy(), M, K, oracle.LAYOUT_MMA, True, E5)
    B = oracle.dequantize(qw.cpu().numpy(), sw.cpu().numpy(), N, K, oracle.LAYOUT_MMA, True, E5)
    ref, ab = A @ B.T, np.abs(A) @ np.abs(B).T
    got = c.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-5 * ab + 1e-30)
    exact = x.double().numpy() @ w.double().numpy().T
    assert np.linalg.norm(got - exact) / np.linalg.norm(exact) < 0.1    # E5M2 keeps 2 mantissa bits
    # the MXFP4 GEMM's epilogue writing E5M2 codes equals quantizing its fp32 C
    g4 = torch.Generator(device=DEV).manual_seed(7)
    qa = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=DEV, generator=g4)
    qb = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=DEV, generator=g4)
    sa = torch.randint(120, 134, (M * K // 32,), dtype=torch.uint8, device=DEV, generator=g4)
    sb = torch.randint(120, 134, (N * K // 32,), dtype=torch.uint8, device=DEV, generator=g4)
    c4 = mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K)
    for block in (mx.BLOCK_1X32, mx.BLOCK_32X32):
        pe = mx.QuantParams(block, mx.SCALE_ROUNDUP, mx.ROUND_RTN, mx.LAYOUT_MMA, elem_format=mx.FORMAT_E5M2)
        ref = mx.mxfp4_quantize(c4, pe, pe)
        q, s, qc, sc, _ = mx.mxfp4_gemm_quantize(qa, sa, qb, sb, M, N, K, pe, col=pe)
        torch.cuda.synchronize()
        assert torch.equal(q, ref[0]) and torch.equal(s, ref[1])
        assert torch.equal(qc, ref[2]) and torch.equal(sc, ref[3])


def test_e5m2_rejects():
    import gemm_pt_block_gb300 as mx

    x = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(mx.Mxfp4Error):        # stochastic rounding is E2M1-only
        mx.mxfp4_quantize(x, mx.QuantParams(rounding=mx.ROUND_SR, elem_format=mx.FORMAT_E5M2))
    z = torch.zeros(256 * 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(mx.Mxfp4Error):        # not an 8-bit element format
        mx.mxfp8_gemm(z, z, z, z, 256, 256, 128, elem_format=mx.FORMAT_E2M1)
