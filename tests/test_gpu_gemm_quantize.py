"""GEMM with the quantizer fused into its epilogue: codes and scales must be
bit-identical to quantizing the GEMM's own fp32 output (mxfp4_quantize with
cols = N), and that quantization must equal the oracle's on the same fp32
values; the optional fp32 output must equal the plain GEMM's."""
from __future__ import annotations

import itertools

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import gemm_tolerance_check

pytestmark = pytest.mark.gpu
DEV = "cuda"
MASK = 0xC0FFEE11

# CTA-pair kernel; 1-CTA kernel (M % 256 = 128); N and K 128 past a multiple of 256
SHAPES = [(256, 512, 512), (384, 256, 768), (256, 384, 640)]
VARIANTS = list(itertools.product((0, 1), (0, 1), (0, 1), (False, True), (0, 1)))


def _operands(M, N, K, seed):
    qa, qb = synth.random_codes(M, K, seed), synth.random_codes(N, K, seed + 1)
    sa, sb = synth.random_scales(M, K, seed + 2), synth.random_scales(N, K, seed + 3)
    return qa, sa, qb, sb, [torch.from_numpy(a).to(DEV) for a in (qa, sa, qb, sb)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("block,smode,rnd,wht,layout", VARIANTS)
def test_fused_equals_quantize_of_gemm_output(M, N, K, block, smode, rnd, wht, layout):
    import gemm_pt_block_gb300 as mx

    p = mx.QuantParams(block, smode, rnd, layout, wht, MASK if wht else 0, 99, 3)
    *_, t = _operands(M, N, K, M + N + K)
    c = mx.mxfp4_gemm(*t, M, N, K)
    ref = mx.mxfp4_quantize(c, p)
    q, s, c2 = mx.mxfp4_gemm_quantize(*t, M, N, K, p, with_c=True)
    q_only, s_only, none = mx.mxfp4_gemm_quantize(*t, M, N, K, p)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert none is None
    assert torch.equal(c2, c)
    assert torch.equal(q, ref[0]) and torch.equal(s, ref[1])
    assert torch.equal(q_only, ref[0]) and torch.equal(s_only, ref[1])


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fused_against_oracle(M, N, K):
    import gemm_pt_block_gb300 as mx

    p = mx.QuantParams(mx.BLOCK_1X32, mx.SCALE_ROUNDUP, mx.ROUND_SR, mx.LAYOUT_MMA, True, MASK, 5, 2)
    qa, sa, qb, sb, t = _operands(M, N, K, 7 * M + K)
    q, s, c = mx.mxfp4_gemm_quantize(*t, M, N, K, p, with_c=True)
    torch.cuda.synchronize()
    cn = c.cpu().numpy()
    ref, ab = oracle.gemm_ref(qa, sa, qb, sb, M, N, K)
    gemm_tolerance_check(cn, ref, ab)
    op = oracle.Params(p.block, p.scale_mode, p.rounding, p.wht, p.wht_sign_mask, p.seed, p.sr_stream)
    oq, os_ = oracle.quantize_rows(np.ascontiguousarray(cn, dtype=np.float32), op)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy(), oracle.scales_to_mma(os_))


def test_fused_rejects_bad_arguments():
    import gemm_pt_block_gb300 as mx

    p = mx.QuantParams(mx.BLOCK_1X32, mx.SCALE_FLOOR, mx.ROUND_RTN, mx.LAYOUT_MMA)
    *_, t = _operands(256, 256, 256, 3)
    z = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)   # room for N = 320
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp4_gemm_quantize(t[0], t[1], z, z, 256, 320, 256, p)   # N % 128 != 0
    with pytest.raises(ValueError):                           # B smaller than N = 320 rows
        mx.mxfp4_gemm_quantize(*t, 256, 320, 256, p)
    bad = mx.QuantParams(5, mx.SCALE_FLOOR, mx.ROUND_RTN, mx.LAYOUT_MMA)
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp4_gemm_quantize(*t, 256, 256, 256, bad)        # bad block


@pytest.mark.parametrize("block", [0, 1])
def test_fused_mxfp8_output(block):
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 512, 512
    p = mx.QuantParams(block, mx.SCALE_ROUNDUP, mx.ROUND_RTN, mx.LAYOUT_MMA,
                       elem_format=mx.FORMAT_E4M3)
    *_, t = _operands(M, N, K, 17)
    c = mx.mxfp4_gemm(*t, M, N, K)
    ref = mx.mxfp4_quantize(c, p)
    q, s, _ = mx.mxfp4_gemm_quantize(*t, M, N, K, p)
    torch.cuda.synchronize()
    assert q.shape == (M, N)
    assert torch.equal(q, ref[0]) and torch.equal(s, ref[1])


# ------------------------------------------------ column-wise (C^T along M) --

# CTA-pair kernel; the last of them with a last M tile of 128 rows
COL_SHAPES = [(256, 512, 512), (512, 256, 768), (256, 640, 384), (384, 256, 768), (640, 384, 384)]


@pytest.mark.parametrize("M,N,K", COL_SHAPES)
@pytest.mark.parametrize("block,smode,rnd,wht,layout", VARIANTS)
def test_fused_columns_equal_quantize_of_gemm_output(M, N, K, block, smode, rnd, wht, layout):
    """Column-wise output alone and together with a row-wise one: bit-identical
    to mxfp4_quantize(C, row, col) of the kernel's own fp32 C."""
    import gemm_pt_block_gb300 as mx

    p = mx.QuantParams(block, smode, rnd, layout, wht, MASK if wht else 0, 77, 4)
    prow = mx.QuantParams(1 - block, smode, 1 - rnd, layout, not wht, 0x1234 if not wht else 0, 77, 4)
    *_, t = _operands(M, N, K, 3 * M + N)
    c = mx.mxfp4_gemm(*t, M, N, K)
    ref = mx.mxfp4_quantize(c, prow, p)
    q_r, s_r, q_c, s_c, c2 = mx.mxfp4_gemm_quantize(*t, M, N, K, prow, col=p, with_c=True)
    n_r, n_s, q_c1, s_c1, none = mx.mxfp4_gemm_quantize(*t, M, N, K, col=p)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert none is None and n_r is None and n_s is None
    assert torch.equal(c2, c)
    assert torch.equal(q_r, ref[0]) and torch.equal(s_r, ref[1])
    assert torch.equal(q_c, ref[2]) and torch.equal(s_c, ref[3])
    assert torch.equal(q_c1, ref[2]) and torch.equal(s_c1, ref[3])


def test_fused_columns_against_oracle_with_bf16_c():
    """Both orientations with rotation + SR from one GEMM (bf16 C stored),
    against the oracle's quantization of the fp32 C."""
    import gemm_pt_block_gb300 as mx

    M, N, K = 512, 512, 1024
    p = mx.QuantParams(mx.BLOCK_32X32, mx.SCALE_ROUNDUP, mx.ROUND_SR, mx.LAYOUT_MMA, True, MASK, 5, 2)
    qa, sa, qb, sb, t = _operands(M, N, K, 11)
    c32 = mx.mxfp4_gemm(*t, M, N, K)
    q_r, s_r, q_c, s_c, c16 = mx.mxfp4_gemm_quantize(*t, M, N, K, p, col=p, with_c=True,
                                                     out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(c16.cpu().view(torch.int16), c32.cpu().to(torch.bfloat16).view(torch.int16))
    cn = c32.cpu().numpy()
    op = oracle.Params(p.block, p.scale_mode, p.rounding, p.wht, p.wht_sign_mask, p.seed, p.sr_stream)
    oq, os_ = oracle.quantize_rows(cn, op)
    cq, cs = oracle.quantize_cols(cn, op)
    assert np.array_equal(q_r.cpu().numpy(), oq)
    assert np.array_equal(s_r.cpu().numpy(), oracle.scales_to_mma(os_))
    assert np.array_equal(q_c.cpu().numpy(), cq)
    assert np.array_equal(s_c.cpu().numpy(), oracle.scales_to_mma(cs))


def test_fused_columns_mxfp8_and_rejects():
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 512, 512
    p = mx.QuantParams(mx.BLOCK_1X32, mx.SCALE_ROUNDUP, mx.ROUND_RTN, mx.LAYOUT_MMA,
                       elem_format=mx.FORMAT_E4M3)
    *_, t = _operands(M, N, K, 21)
    c = mx.mxfp4_gemm(*t, M, N, K)
    ref = mx.mxfp4_quantize(c, None, p)
    _, _, q_c, s_c, _ = mx.mxfp4_gemm_quantize(*t, M, N, K, col=p)
    torch.cuda.synchronize()
    assert q_c.shape == (N, M)
    assert torch.equal(q_c, ref[2]) and torch.equal(s_c, ref[3])
    with pytest.raises(mx.Mxfp4Error):                         # 64x64 blocks
        mx.mxfp4_gemm_quantize(*t, M, N, K, col=mx.QuantParams(mx.BLOCK_64X64))


def test_fused_columns_full_size_sampled():
    """Fprop's 70B shape (16384 x 28672 x 8192) in the benchmark's launch
    configuration: both orientations with rotation + SR, no C. Whole outputs
    against the standalone quantizer on the plain GEMM's C, and sampled output
    rows of each orientation against the oracle."""
    import gemm_pt_block_gb300 as mx

    M, N, K = 16384, 28672, 8192
    g = torch.Generator(device=DEV).manual_seed(5)
    qa = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    qb = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    sa = torch.randint(120, 135, (M * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    sb = torch.randint(120, 135, (N * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    p = mx.QuantParams(mx.BLOCK_1X32, mx.SCALE_ROUNDUP, mx.ROUND_SR, mx.LAYOUT_ROWMAJOR, True, MASK, 9, 1)
    q_r, s_r, q_c, s_c, _ = mx.mxfp4_gemm_quantize(qa, sa, qb, sb, M, N, K, p, col=p)
    c = mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K)
    ref = mx.mxfp4_quantize(c, p, p)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert torch.equal(q_r, ref[0]) and torch.equal(s_r, ref[1])
    assert torch.equal(q_c, ref[2]) and torch.equal(s_c, ref[3])
    cn = c.cpu().numpy()
    del ref, c
    op = oracle.Params(p.block, p.scale_mode, p.rounding, p.wht, p.wht_sign_mask, p.seed, p.sr_stream)
    for r0 in (0, M - 32):
        oq, os_ = oracle.quantize_rows(cn, op, r0, r0 + 32)
        assert np.array_equal(q_r[r0:r0 + 32].cpu().numpy(), oq)
        assert np.array_equal(s_r[r0:r0 + 32].cpu().numpy(), os_)
    for c0 in (0, N - 32):
        oq, os_ = oracle.quantize_cols(cn, op, c0, c0 + 32)
        assert np.array_equal(q_c[c0:c0 + 32].cpu().numpy(), oq)
        assert np.array_equal(s_c[c0:c0 + 32].cpu().numpy(), os_)


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (512, 768, 2304)])
def test_fused_row_output_same_with_and_without_workspace(M, N, K):
    """Row-wise fused output on the scale-image path (workspace) and the plain
    path: identical codes, scales and C."""
    import gemm_pt_block_gb300 as mx

    p = mx.QuantParams(mx.BLOCK_32X32, mx.SCALE_ROUNDUP, mx.ROUND_SR, mx.LAYOUT_MMA, True, MASK, 8, 1)
    *_, t = _operands(M, N, K, 5 * M + K)
    a = mx.mxfp4_gemm_quantize(*t, M, N, K, p, with_c=True)
    b = mx.mxfp4_gemm_quantize(*t, M, N, K, p, with_c=True, workspace=False)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    for x, y in zip(a, b):
        assert torch.equal(x, y)
