"""mxfp4_gemm_noalloc, the GEMM entry point for callers that cannot allocate
device memory (a framework that owns every byte of device memory through its
own pool, a latency-bounded host loop that must not wait on the driver's
allocator, a plugin handed only its inputs and outputs). It runs the
scale-image GEMM on a static 96 MiB array inside the library instead of a
caller workspace.

Checked through the C ABI: two calls in a row give the same C as the plain
entry point and as mxfp4_gemm_ex with a caller workspace (the same image
path); the largest shape whose images fill the array exactly is accepted, one
K step more is refused before any device work, and M % 256 == 128 (which uses
no images) is not limited. This file is collected last so that a run stopping
at its first failure has run every other test already.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCRATCH = 96 << 20


def _operands(M, N, K, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    qa = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    qb = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    sa = torch.randint(118, 137, (M * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    sb = torch.randint(118, 137, (N * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    return qa, sa, qb, sb


def _check_two_calls(M, N, K, seed):
    import gemm_pt_block_gb300 as mx

    t = _operands(M, N, K, seed)
    want = mx.mxfp4_gemm(*t, M, N, K, workspace=False)
    ws = torch.empty(max(mx.gemm_workspace_size(M, N, K), 16), dtype=torch.uint8, device=DEV)
    want_img = mx.mxfp4_gemm(*t, M, N, K, workspace=ws)
    first = mx.mxfp4_gemm_noalloc(*t, M, N, K)
    second = mx.mxfp4_gemm_noalloc(*t, M, N, K)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert torch.equal(want_img, want)
    assert torch.equal(first, want)
    assert torch.equal(second, want)


@pytest.mark.parametrize("M,N,K,seed", [(512, 768, 2304, 1), (16384, 8192, 28672, 2),
                                        (256, 384, 640, 5)])
def test_noalloc_matches_the_other_entry_points_on_two_calls(M, N, K, seed):
    _check_two_calls(M, N, K, seed)


def test_noalloc_accepts_images_that_fill_its_scratch_exactly():
    M, N, K = 12288, 12288, 32768
    assert 4 * (M + N) * K // 32 == SCRATCH
    _check_two_calls(M, N, K, 3)


def test_noalloc_without_images_is_not_limited_by_the_scratch():
    M, N, K = 12416, 12288, 32768        # M % 256 == 128: the one-CTA kernel, no images
    assert 4 * (M + N) * K // 32 > SCRATCH
    _check_two_calls(M, N, K, 4)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import gemm_pt_block_gb300 as mx

    # Through the C ABI directly: the library must refuse these shapes before
    # it touches any buffer (the binding would already refuse the tiny ones).
    z = torch.zeros(16, dtype=torch.uint8, device=DEV)
    c = torch.empty(16, dtype=torch.float32, device=DEV)
    L = mx.lib()
    P = ctypes.c_void_p
    for M, N, K in ((12288, 12288, 32768 + 256), (32768, 32768, 32768)):
        assert 4 * (M + N) * K // 32 > SCRATCH
        st = L.mxfp4_gemm_noalloc(P(z.data_ptr()), P(z.data_ptr()), P(z.data_ptr()), P(z.data_ptr()),
                                  M, N, K, P(c.data_ptr()), N,
                                  P(torch.cuda.current_stream().cuda_stream))
        assert st == 2, L.mxfp4_last_error()
    with pytest.raises(ValueError):                 # the binding checks extents first
        mx.mxfp4_gemm_noalloc(z, z, z, z, 12288, 12288, 32768 + 256, c=c, ldc=12288)
