"""Device max-abs and NVFP4 per-tensor exponent (mxfp4_tensor_amax) against the
oracle: bf16 and fp32, strided rows, outliers, zeros and subnormals, tensors
large enough for many CTAs, and the exponent feeding the NVFP4 quantizer."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import assert_same, gpu_quantize, oracle_input, oracle_quantize

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _check(x: torch.Tensor):
    import gemm_pt_block_gb300 as mx

    a, k = mx.tensor_amax(x.to(DEV) if not x.is_cuda else x)
    torch.cuda.synchronize()
    want_a = oracle.tensor_amax(oracle_input(x.cpu() if x.is_cuda else x))
    assert float(a.item()) == want_a
    assert int(k.item()) == oracle.nv_tensor_exp(want_a)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols", [(1, 32), (96, 160), (1000, 4096), (8192, 32)])
def test_amax_matches_oracle(dtype, rows, cols):
    x = synth.laplace(rows, cols, 1e-3, seed=rows + cols, outlier_frac=0.001).to(dtype)
    _check(x)
    _check(-x.abs())


def test_amax_strided_zero_tiny_and_huge():
    wide = synth.student_t(64, 320, 3.0, seed=3)
    xs = wide.to(DEV)[:, 32:288]
    xs_host = wide[:, 32:288].contiguous()
    import gemm_pt_block_gb300 as mx

    a, k = mx.tensor_amax(xs)
    torch.cuda.synchronize()
    assert float(a.item()) == oracle.tensor_amax(oracle_input(xs_host))
    _check(torch.zeros(32, 64, dtype=torch.bfloat16))
    tiny = torch.full((32, 64), 1e-40, dtype=torch.float32)          # fp32 subnormals
    _check(tiny)
    _check(torch.full((32, 64), 3.0e38, dtype=torch.float32))
    e = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    a, k = mx.tensor_amax(e)
    torch.cuda.synchronize()
    assert float(a.item()) == 0.0 and int(k.item()) == 0


def test_amax_exponent_drives_nvfp4_quantizer():
    import gemm_pt_block_gb300 as mx

    x = synth.student_t(256, 512, 3.0, seed=11)
    x[3, 7] = 5000.0
    k = mx.nvfp4_tensor_exp(x.to(DEV))
    assert k == oracle.nv_tensor_exp(oracle.tensor_amax(oracle_input(x)))
    p = oracle.Params(block=oracle.BLOCK_1X16, scale_mode=oracle.SCALE_ROUNDUP, tensor_exp=k)
    assert_same(gpu_quantize(x.to(DEV), p, p), oracle_quantize(oracle_input(x), p, p), "nvfp4 with device k")
