"""mxfp4_gemm_noalloc: the scale-image GEMM path with the library's static
scratch instead of a caller workspace. Two calls against the plain entry point
(bit-identical), and the size limit."""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _operands(M, N, K, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    qa = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    qb = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    sa = torch.randint(118, 137, (M * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    sb = torch.randint(118, 137, (N * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    return qa, sa, qb, sb


def test_noalloc_matches_plain_entry_point_on_two_calls():
    import gemm_pt_block_gb300 as mx

    for (M, N, K), seed in (((512, 768, 2304), 1), ((16384, 8192, 28672), 2)):
        t = _operands(M, N, K, seed)
        want = mx.mxfp4_gemm(*t, M, N, K, workspace=False)
        got = mx.mxfp4_gemm_noalloc(*t, M, N, K)
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        assert torch.equal(got, want)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import gemm_pt_block_gb300 as mx

    M, N, K = 32768, 32768, 32768      # images 4 * 65536 * 1024 bytes = 256 MiB
    z = torch.zeros(16, dtype=torch.uint8, device=DEV)
    c = torch.empty(16, dtype=torch.float32, device=DEV)
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.mxfp4_gemm_noalloc(z, z, z, z, M, N, K, c=c, ldc=N)
    assert e.value.status == 2
