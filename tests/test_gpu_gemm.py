"""CUDA block-scaled MXFP4 GEMM vs the fp64 oracle.

Exact-arithmetic cases must match bit for bit; everything else must satisfy
|C - ref| <= 1e-5 * sum_k |a_k b_k| element-wise (ref = fp64 sum of the
dequantized products)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import assert_same, cuda_params, gemm_tolerance_check

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _gemm(qa, sa, qb, sb, M, N, K):
    import gemm_pt_block_gb300 as mx

    t = [torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (qa, sa, qb, sb)]
    c = mx.mxfp4_gemm(*t, M, N, K)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    return c.cpu().numpy()


def test_gemm_all_ones_exact():
    M, N, K = 128, 256, 256
    ones = np.full((M, K // 2), 0x22, dtype=np.uint8)
    onesb = np.full((N, K // 2), 0x22, dtype=np.uint8)
    c = _gemm(ones, np.full(M * K // 32, 127, np.uint8), onesb, np.full(N * K // 32, 127, np.uint8), M, N, K)
    assert np.all(c == K)


def test_gemm_one_hot_rows_exact():
    """A has one nonzero code per row: C's row m is that value times column k(m) of B."""
    M, N, K = 128, 256, 512
    qa = np.zeros((M, K // 2), dtype=np.uint8)
    ks = (np.arange(M) * 37) % K
    for m in range(M):
        code = 0x6 if m % 3 else 0xB            # 4.0 or -1.5
        qa[m, ks[m] // 2] = code << (4 * (ks[m] & 1))
    sa = np.full(M * K // 32, 127, np.uint8)
    qb = synth.random_codes(N, K, 11)
    sb = synth.random_scales(N, K, 12)
    c = _gemm(qa, sa, qb, sb, M, N, K)
    ref, _ = oracle.gemm_ref(qa, sa, qb, sb, M, N, K)
    assert np.array_equal(c.astype(np.float64), ref)


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (128, 384, 384), (256, 384, 640),
                                   (384, 640, 1152)])
def test_gemm_per_block_scales_exact(M, N, K):
    """Unit scales except one block per row / column: checks each scale's slot,
    including the last K step and last output tile of 128 when N or K is 128
    more than a multiple of 256."""
    qa = synth.random_codes(M, K, 21)
    qb = synth.random_codes(N, K, 22)
    sa_rm = np.full((M, K // 32), 127, np.uint8)
    sb_rm = np.full((N, K // 32), 127, np.uint8)
    rng = np.random.default_rng(23)
    sa_rm[np.arange(M), rng.integers(0, K // 32, M)] = 129
    sb_rm[np.arange(N), rng.integers(0, K // 32, N)] = 125
    sa, sb = oracle.scales_to_mma(sa_rm), oracle.scales_to_mma(sb_rm)
    c = _gemm(qa, sa, qb, sb, M, N, K)
    ref, _ = oracle.gemm_ref(qa, sa, qb, sb, M, N, K)
    # products are multiples of 2^-4 below 2^10; partial sums stay exact in fp32
    assert np.array_equal(c.astype(np.float64), ref)


# Shapes whose N or K is 128 more than a multiple of 256 (a last output tile of
# 128 columns, a last K step of 128) next to the aligned ones.
ODD_SHAPES = [(128, 128, 128), (256, 128, 128), (128, 384, 384), (256, 384, 640), (384, 640, 1152),
              (256, 256, 384), (256, 384, 256), (768, 1152, 1408)]


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 768), (384, 768, 2304),
                                   (2048, 4096, 512), (1280, 2560, 4096)] + ODD_SHAPES)
def test_gemm_random_within_tolerance(M, N, K):
    qa, qb = synth.random_codes(M, K, M + 1), synth.random_codes(N, K, N + 2)
    sa, sb = synth.random_scales(M, K, K + 3), synth.random_scales(N, K, K + 4)
    c = _gemm(qa, sa, qb, sb, M, N, K)
    ref, absref = oracle.gemm_ref(qa, sa, qb, sb, M, N, K)
    gemm_tolerance_check(c, ref, absref)


def test_gemm_wide_scale_range_and_ldc():
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 256, 1024
    qa, qb = synth.random_codes(M, K, 51), synth.random_codes(N, K, 52)
    sa, sb = synth.random_scales(M, K, 53, 90, 160), synth.random_scales(N, K, 54, 90, 160)
    big = torch.full((M, N + 64), -7.0, device=DEV)
    t = [torch.from_numpy(a).to(DEV) for a in (qa, sa, qb, sb)]
    mx.mxfp4_gemm(*t, M, N, K, c=big, ldc=N + 64)
    out = big.cpu().numpy()
    assert np.all(out[:, N:] == -7.0)                  # nothing written past N
    ref, absref = oracle.gemm_ref(qa, sa, qb, sb, M, N, K)
    gemm_tolerance_check(out[:, :N], ref, absref)


def test_gemm_repeatable():
    M, N, K = 512, 512, 2048
    qa, qb = synth.random_codes(M, K, 61), synth.random_codes(N, K, 62)
    sa, sb = synth.random_scales(M, K, 63), synth.random_scales(N, K, 64)
    a = _gemm(qa, sa, qb, sb, M, N, K)
    b = _gemm(qa, sa, qb, sb, M, N, K)
    assert np.array_equal(a, b)


def test_linear_layer_tiny_end_to_end():
    """X [512,1024] N(0,1) with 8 outlier columns x50, W [512,1024] N(0,0.02); both
    rotated by the same random-sign 32-point transform, 1x32 floor scales, W by
    nearest-even and X by stochastic rounding (seed 0); then Y = Xq Wq^T."""
    import gemm_pt_block_gb300 as mx

    T, D, F = 512, 1024, 512
    x = synth.normal_outlier_cols(T, D, 1.0, 8, 50.0, seed=1000)
    w = synth.normal(F, D, 0.02, seed=1000 + 100)
    mask = synth.sign_mask(1000)
    px = oracle.Params(rounding=oracle.ROUND_SR, wht=True, wht_sign_mask=mask, seed=0)
    pw = oracle.Params(wht=True, wht_sign_mask=mask)
    qx, sx, _, _ = mx.mxfp4_quantize(x.to(DEV), cuda_params(px, 1))
    qw, sw, _, _ = mx.mxfp4_quantize(w.to(DEV), cuda_params(pw, 1))
    y = mx.mxfp4_gemm(qx, sx, qw, sw, T, F, D).cpu().numpy()
    rqx, rsx = oracle.quantize_rows(synth.bf16_bits(x), px)
    rqw, rsw = oracle.quantize_rows(synth.bf16_bits(w), pw)
    assert_same([qx.cpu().numpy(), sx.cpu().numpy(), qw.cpu().numpy(), sw.cpu().numpy()],
                [rqx, oracle.scales_to_mma(rsx), rqw, oracle.scales_to_mma(rsw)], "operands")
    ref, absref = oracle.gemm_ref(rqx, oracle.scales_to_mma(rsx), rqw, oracle.scales_to_mma(rsw), T, F, D)
    gemm_tolerance_check(y, ref, absref)
    # the rotation cancels in the product: Y approximates X W^T
    exact = x.double().numpy() @ w.double().numpy().T
    rel = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert rel < 0.25


@pytest.mark.parametrize("M,N,K", [(8192, 14336, 4096), (8192, 4096, 14336), (14336, 4096, 8192)])
def test_gemm_full_size_sampled_rows(M, N, K):
    """Workload-sized Fprop / Dgrad / Wgrad shapes in the launch configuration the
    benchmark times; the oracle checks a sample of full output rows."""
    qa, qb = synth.random_codes(M, K, 7), synth.random_codes(N, K, 8)
    sa, sb = synth.random_scales(M, K, 9), synth.random_scales(N, K, 10)
    c = _gemm(qa, sa, qb, sb, M, N, K)
    rows = np.array([0, 1, 127, 128, M // 2 + 77, M - 1])
    ms = np.repeat(rows, 64)
    ns = np.tile(np.linspace(0, N - 1, 64).astype(np.int64), len(rows))
    ref, absref = oracle.gemm_pairs(qa, sa, qb, sb, M, N, K, ms, ns)
    gemm_tolerance_check(c[ms, ns], ref, absref)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (256, 512, 768), (512, 768, 2304),
                                   (1024, 1280, 4096), (16384, 8192, 28672), (256, 128, 128),
                                   (256, 384, 640), (512, 640, 1152), (768, 1152, 1408)])
def test_gemm_scale_images_bit_identical(M, N, K):
    """The workspace path (scales rewritten as replicated images, 128x256b
    tensor-memory copies) gives the same bits as the plain entry point, for
    fp32 and bf16 C; also against the oracle on sampled rows."""
    import gemm_pt_block_gb300 as mx

    g = torch.Generator(device=DEV).manual_seed(M + K)
    qa = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    qb = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    sa = torch.randint(118, 137, (M * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    sb = torch.randint(118, 137, (N * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    nimg = mx.gemm_workspace_size(M, N, K)
    ceil256 = lambda v: (v + 255) // 256 * 256
    assert nimg == 4 * (M * ceil256(K) + ceil256(N) * K) // 32
    ws = torch.full((nimg,), 0xAB, dtype=torch.uint8, device=DEV)
    plain = mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K, workspace=False)
    img = mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K, workspace=ws)
    img16 = mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K, workspace=ws, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert torch.equal(plain, img)
    assert torch.equal(img16.view(torch.int16), plain.to(torch.bfloat16).view(torch.int16))
    rows = np.array([0, 1, 129, M // 2 + 3, M - 1])
    ms = np.repeat(rows, 16)
    ns = np.tile(np.linspace(0, N - 1, 16).astype(np.int64), len(rows))
    ref, absref = oracle.gemm_pairs(qa.cpu().numpy(), sa.cpu().numpy(), qb.cpu().numpy(),
                                    sb.cpu().numpy(), M, N, K, ms, ns)
    gemm_tolerance_check(img[torch.from_numpy(ms), torch.from_numpy(ns)].cpu().numpy(), ref, absref)


def test_gemm_workspace_too_small_falls_back():
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 512, 512
    g = torch.Generator(device=DEV).manual_seed(3)
    qa = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    qb = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    sa = torch.randint(120, 135, (M * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    sb = torch.randint(120, 135, (N * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    small = torch.empty(mx.gemm_workspace_size(M, N, K) - 16, dtype=torch.uint8, device=DEV)
    a = mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K, workspace=small)
    b = mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K, workspace=False)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
