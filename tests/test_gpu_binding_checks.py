"""The Python binding refuses caller buffers that the C ABI cannot check
(raw pointers carry no extent): too small, wrong dtype, not contiguous, or C
rows that would run past the tensor's storage. Every case raises before any
kernel is launched, and a correct call right after still works."""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"
U8 = dict(dtype=torch.uint8, device=DEV)


def test_quantize_outputs_are_checked():
    import gemm_pt_block_gb300 as mx

    x = torch.randn(128, 256, device=DEV).to(torch.bfloat16)
    p = mx.QuantParams()
    with pytest.raises(ValueError):                      # codes one byte short
        mx.mxfp4_quantize(x, p, q_row=torch.empty(128 * 128 - 1, **U8))
    with pytest.raises(TypeError):                       # scales not uint8
        mx.mxfp4_quantize(x, p, s_row=torch.empty(128 * 8, dtype=torch.int32, device=DEV))
    with pytest.raises(ValueError):                      # not contiguous
        mx.mxfp4_quantize(x, p, q_row=torch.empty(128, 256, **U8)[:, ::2])
    with pytest.raises(ValueError):                      # column output sized for rows
        mx.mxfp4_quantize(x, None, p, q_col=torch.empty(128 * 128, **U8)[: 256 * 64 - 16])
    q, s, _, _ = mx.mxfp4_quantize(x, p)
    assert q.shape == (128, 128) and s.shape == (128, 8)


def test_gemm_operands_and_c_are_checked():
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 256, 256
    pm = mx.QuantParams(scale_layout=mx.LAYOUT_MMA)
    a = torch.randn(M, K, device=DEV).to(torch.bfloat16)
    b = torch.randn(N, K, device=DEV).to(torch.bfloat16)
    qa, sa, _, _ = mx.mxfp4_quantize(a, pm)
    qb, sb, _, _ = mx.mxfp4_quantize(b, pm)
    with pytest.raises(ValueError):                      # A's codes hold fewer than M rows
        mx.mxfp4_gemm(qa[: M // 2], sa, qb, sb, M, N, K)
    with pytest.raises(ValueError):                      # B's scales too short
        mx.mxfp4_gemm(qa, sa, qb, sb[:-1], M, N, K)
    with pytest.raises(ValueError):                      # C too small
        mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K, c=torch.empty(M - 1, N, device=DEV))
    with pytest.raises(ValueError):                      # ldc < N
        mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K, c=torch.empty(M, N, device=DEV), ldc=N - 8)
    with pytest.raises(ValueError):                      # rows of ldc run past C's storage
        mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K, c=torch.empty(M, N, device=DEV), ldc=N + 64)
    with pytest.raises(ValueError):                      # fused outputs too small
        mx.mxfp4_gemm_quantize(qa, sa, qb, sb, M, N, K, pm, q_out=torch.empty(16, **U8))
    with pytest.raises(ValueError):                      # MXFP8 codes are one byte per element
        mx.mxfp8_gemm(qa, sa, qb, sb, M, N, K)
    c = mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K)
    assert c.shape == (M, N) and torch.isfinite(c).all()


def test_other_outputs_are_checked():
    import gemm_pt_block_gb300 as mx

    x = torch.randn(128, 256, device=DEV).to(torch.bfloat16)
    q, s, _, _ = mx.mxfp4_quantize(x, mx.QuantParams())
    with pytest.raises(ValueError):
        mx.mxfp4_dequantize(q, s, 128, 256, out=torch.empty(128, 255, device=DEV))
    with pytest.raises(ValueError):
        mx.mxfp4_dequantize(q[:64], s, 128, 256)
    with pytest.raises(ValueError):
        mx.hadamard32(x, y=torch.empty(100, 256, device=DEV))
    with pytest.raises(TypeError):
        mx.tensor_amax(x, amax=torch.empty(1, dtype=torch.float64, device=DEV))
    assert mx.mxfp4_dequantize(q, s, 128, 256).shape == (128, 256)
