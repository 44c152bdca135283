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

SHAPES = [(256, 512, 512), (384, 256, 768)]   # CTA-pair kernel; 1-CTA kernel (M % 256 = 128)
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
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp4_gemm_quantize(*t, 256, 384, 256, p)          # N % 256 != 0
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
