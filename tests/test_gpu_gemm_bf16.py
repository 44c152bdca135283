"""GEMM outputs stored as bf16 (mxfp4_gemm_ex, mxfp8_gemm and the fused
quantize with a bf16 C) against the fp64 oracle.

Each bf16 value is the fp32 sum rounded to nearest-even, so: exact cases match
the oracle's value rounded to bf16 bit for bit; the rest stay within the fp32
bound plus half a bf16 unit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import bf16_to_f64, cuda_params, gemm_tolerance_check_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _dev(*arrays):
    return [torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in arrays]


def test_bf16_c_exact_products_round_like_the_oracle():
    """Unit scales except one block per row / column: every partial sum is exact
    in fp32, so the bf16 output is the oracle's value rounded to bf16."""
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 512, 1024
    qa, qb = synth.random_codes(M, K, 21), synth.random_codes(N, K, 22)
    sa_rm = np.full((M, K // 32), 127, np.uint8)
    sb_rm = np.full((N, K // 32), 127, np.uint8)
    rng = np.random.default_rng(23)
    sa_rm[np.arange(M), rng.integers(0, K // 32, M)] = 129
    sb_rm[np.arange(N), rng.integers(0, K // 32, N)] = 125
    sa, sb = oracle.scales_to_mma(sa_rm), oracle.scales_to_mma(sb_rm)
    c = mx.mxfp4_gemm(*_dev(qa, sa, qb, sb), M, N, K, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert c.dtype == torch.bfloat16 and mx.device_status() == 0
    ref, _ = oracle.gemm_ref(qa, sa, qb, sb, M, N, K)
    want = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16)  # exact fp32, then RNE
    assert torch.equal(c.cpu().view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 768), (384, 768, 2304),
                                   (1280, 2560, 4096), (256, 384, 640), (384, 640, 1152)])
def test_bf16_c_within_tolerance(M, N, K):
    import gemm_pt_block_gb300 as mx

    qa, qb = synth.random_codes(M, K, M + 5), synth.random_codes(N, K, N + 6)
    sa, sb = synth.random_scales(M, K, K + 7), synth.random_scales(N, K, K + 8)
    t = _dev(qa, sa, qb, sb)
    c = mx.mxfp4_gemm(*t, M, N, K, out_dtype=torch.bfloat16)
    c32 = mx.mxfp4_gemm(*t, M, N, K)
    torch.cuda.synchronize()
    ref, absref = oracle.gemm_ref(qa, sa, qb, sb, M, N, K)
    gemm_tolerance_check_bf16(bf16_to_f64(c), ref, absref)
    # the bf16 store is the fp32 result rounded to nearest-even
    assert torch.equal(c.cpu().view(torch.int16), c32.cpu().to(torch.bfloat16).view(torch.int16))


def test_bf16_c_ldc_leaves_padding():
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 256, 512
    qa, qb = synth.random_codes(M, K, 71), synth.random_codes(N, K, 72)
    sa, sb = synth.random_scales(M, K, 73), synth.random_scales(N, K, 74)
    big = torch.full((M, N + 40), -3.0, dtype=torch.bfloat16, device=DEV)
    mx.mxfp4_gemm(*_dev(qa, sa, qb, sb), M, N, K, c=big[:, :N], ldc=N + 40)
    out = big.cpu()
    assert torch.all(out[:, N:] == -3.0)
    ref, absref = oracle.gemm_ref(qa, sa, qb, sb, M, N, K)
    gemm_tolerance_check_bf16(out[:, :N].double().numpy(), ref, absref)


def test_mxfp8_gemm_bf16_c():
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 512, 640
    rng = np.random.default_rng(81)
    qa = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    qb = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x38            # NaN codes -> 1.0
    qb[(qb & 0x7F) == 0x7F] = 0x38
    sa_rm = rng.integers(118, 136, size=(M, K // 32), dtype=np.uint8)
    sb_rm = rng.integers(118, 136, size=(N, K // 32), dtype=np.uint8)
    t = _dev(qa, oracle.scales_to_mma(sa_rm), qb, oracle.scales_to_mma(sb_rm))
    c = mx.mxfp8_gemm(*t, M, N, K, out_dtype=torch.bfloat16)
    c32 = mx.mxfp8_gemm(*t, M, N, K)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert torch.equal(c.cpu().view(torch.int16), c32.cpu().to(torch.bfloat16).view(torch.int16))
    A = oracle.dequantize(qa, sa_rm, M, K, f64=True, fmt=oracle.FORMAT_E4M3)
    B = oracle.dequantize(qb, sb_rm, N, K, f64=True, fmt=oracle.FORMAT_E4M3)
    gemm_tolerance_check_bf16(bf16_to_f64(c), A @ B.T, np.abs(A) @ np.abs(B).T)


@pytest.mark.parametrize("M", [128, 256])
def test_fused_quantize_with_bf16_c(M):
    """The fused codes come from the fp32 sums whatever C's storage type."""
    import gemm_pt_block_gb300 as mx

    N, K = 512, 1024
    qa, qb = synth.random_codes(M, K, 91), synth.random_codes(N, K, 92)
    sa, sb = synth.random_scales(M, K, 93), synth.random_scales(N, K, 94)
    t = _dev(qa, sa, qb, sb)
    p = cuda_params(oracle.Params(block=oracle.BLOCK_32X32, scale_mode=oracle.SCALE_ROUNDUP,
                                  rounding=oracle.ROUND_SR, wht=True, wht_sign_mask=0x5A5A1234,
                                  seed=3, sr_stream=2), 1)
    q1, s1, c1 = mx.mxfp4_gemm_quantize(*t, M, N, K, p, with_c=True, out_dtype=torch.bfloat16)
    q2, s2, c2 = mx.mxfp4_gemm_quantize(*t, M, N, K, p, with_c=True)
    torch.cuda.synchronize()
    assert c1.dtype == torch.bfloat16 and mx.device_status() == 0
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    assert torch.equal(c1.cpu().view(torch.int16), c2.cpu().to(torch.bfloat16).view(torch.int16))
    rq, rs = oracle.quantize_rows(c2.cpu().numpy(), oracle.Params(
        block=oracle.BLOCK_32X32, scale_mode=oracle.SCALE_ROUNDUP, rounding=oracle.ROUND_SR,
        wht=True, wht_sign_mask=0x5A5A1234, seed=3, sr_stream=2))
    assert np.array_equal(q1.cpu().numpy(), rq)
    assert np.array_equal(s1.cpu().numpy(), oracle.scales_to_mma(rs))
