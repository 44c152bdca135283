"""The bounds-checking build (MXFP4_BOUNDS_CHECK): every kernel store is
checked against the extent its call computed for that output, and a store
outside it is skipped and reported as MXFP4_ERR_BOUNDS. Every kernel family
runs here on shapes ragged against its tiles and must report no bounds error
and give the regular library's bits; a positive control shrinks the checked
extents and watches the check fire (the stores past the shrunk extent are
skipped, so nothing leaves its buffer)."""
from __future__ import annotations

import contextlib

import pytest
import torch

import oracle
import synth
from _util import cuda_params
from test_gpu_canary import QUANT_CASES

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def bc_lib():
    from gemm_pt_block_gb300 import binding
    from gemm_pt_block_gb300 import build as b

    return binding.load_library(b.build(bounds_check=True))


@contextlib.contextmanager
def _using(lib):
    from gemm_pt_block_gb300 import binding

    saved = binding.lib()
    binding._lib = lib
    try:
        yield
    finally:
        binding._lib = saved


def _both(bc_lib, fn):
    """fn() on the regular library, then on the bounds-checking one; returns
    both results and the checked build's device status."""
    import gemm_pt_block_gb300 as mx

    want = fn()
    torch.cuda.synchronize()
    with _using(bc_lib):
        got = fn()
        status = mx.device_status()
    return want, got, status


def _equal(a, b):
    if isinstance(a, (tuple, list)):
        return all(_equal(x, y) for x, y in zip(a, b))
    if a is None:
        return b is None
    return torch.equal(a, b)


@pytest.mark.parametrize("case", range(len(QUANT_CASES)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantizer_stores_stay_inside(bc_lib, case, dtype):
    import gemm_pt_block_gb300 as mx

    rows, cols, pr, pc, layout = QUANT_CASES[case]
    x = synth.student_t(rows, cols, 3.0, seed=700 + case).to(dtype).to(DEV)
    fn = lambda: mx.mxfp4_quantize(x, cuda_params(pr, layout) if pr else None,
                                   cuda_params(pc, layout) if pc else None)
    want, got, status = _both(bc_lib, fn)
    assert status == 0
    assert _equal(want, got)


def _operands(M, N, K, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    qa = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    qb = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    sa = torch.randint(120, 135, (M * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    sb = torch.randint(120, 135, (N * K // 32,), dtype=torch.uint8, device=DEV, generator=g)
    return qa, sa, qb, sb


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (384, 768, 1024), (768, 512, 2304),
                                   (128, 384, 384), (256, 384, 640), (512, 128, 1152)])
@pytest.mark.parametrize("c_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("images", [False, True])
def test_gemm_stores_stay_inside(bc_lib, M, N, K, c_dtype, images):
    import gemm_pt_block_gb300 as mx

    t = _operands(M, N, K, M + N + K)
    c = torch.empty(M, N + 40, dtype=c_dtype, device=DEV)
    fn = lambda: mx.mxfp4_gemm(*t, M, N, K, c=c.zero_(), ldc=N + 40,
                               workspace=None if images else False).clone()
    want, got, status = _both(bc_lib, fn)
    assert status == 0
    assert torch.equal(want, got)


@pytest.mark.parametrize("M,N,K", [(512, 768, 1024), (256, 384, 640), (384, 640, 1152)])
def test_fused_epilogue_and_other_gemms_stay_inside(bc_lib, M, N, K):
    import gemm_pt_block_gb300 as mx

    t = _operands(M, N, K, 5)
    p = mx.QuantParams(rounding=mx.ROUND_SR, wht=True, wht_sign_mask=0x1234, seed=6,
                       scale_layout=mx.LAYOUT_MMA)
    for fn in (lambda: mx.mxfp4_gemm_quantize(*t, M, N, K, p, col=p, with_c=True),
               lambda: mx.mxfp4_gemm_quantize(*t, M, N, K, p, out_dtype=torch.bfloat16, with_c=True),
               lambda: mx.mxfp4_gemm_noalloc(*t, M, N, K)):
        want, got, status = _both(bc_lib, fn)
        assert status == 0
        assert _equal(want, got)
    tn = (t[0], torch.randint(40, 70, (M * K // 16,), dtype=torch.uint8, device=DEV),
          t[2], torch.randint(40, 70, (N * K // 16,), dtype=torch.uint8, device=DEV))
    for ws in (None, False):
        fn = lambda: mx.nvfp4_gemm(tn[0], tn[1], -1, tn[2], tn[3], 2, M, N, K, workspace=ws)
        want, got, status = _both(bc_lib, fn)
        assert status == 0 and torch.equal(want, got)
    q8a = torch.randint(0, 120, (M, K), dtype=torch.uint8, device=DEV)
    q8b = torch.randint(0, 120, (N, K), dtype=torch.uint8, device=DEV)
    for fmt in (mx.FORMAT_E4M3, mx.FORMAT_E5M2):
        fn = lambda: mx.mxfp8_gemm(q8a, t[1], q8b, t[3], M, N, K, elem_format=fmt)
        want, got, status = _both(bc_lib, fn)
        assert status == 0 and torch.equal(want, got)


def test_dequantize_rotation_and_amax_stay_inside(bc_lib):
    import gemm_pt_block_gb300 as mx

    x = synth.student_t(96, 352, 3.0, seed=9).to(DEV)
    q, s, _, _ = mx.mxfp4_quantize(x, mx.QuantParams())
    for fn in (lambda: mx.mxfp4_dequantize(q, s, 96, 352),
               lambda: mx.hadamard32(x, 0x1234),
               lambda: mx.tensor_amax(x)):
        want, got, status = _both(bc_lib, fn)
        assert status == 0
        assert _equal(want, got)


def test_the_check_fires_on_a_shrunk_extent(bc_lib):
    """With every code and scale extent 16 bytes short, the last stores of
    each output are skipped and reported; everything before them is written
    as usual, and the 16 bytes the call was not allowed to touch keep their
    fill. The regular library refuses the diagnostic."""
    import gemm_pt_block_gb300 as mx
    from gemm_pt_block_gb300 import binding

    assert binding.lib().mxfp4_bounds_check_shrink(16) == 4
    for rows, cols, pr, pc, layout in (QUANT_CASES[0], QUANT_CASES[5]):
        x = synth.student_t(rows, cols, 3.0, seed=11).to(DEV)
        prow = cuda_params(pr, layout) if pr else None
        pcol = cuda_params(pc, layout) if pc else None
        want = mx.mxfp4_quantize(x, prow, pcol)
        outs = [None if w is None else torch.full_like(w, 0xA5) for w in want]
        with _using(bc_lib):
            assert bc_lib.mxfp4_bounds_check_shrink(16) == 0
            try:
                mx.mxfp4_quantize(x, prow, pcol, q_row=outs[0], s_row=outs[1], q_col=outs[2],
                                  s_col=outs[3])
                status = mx.device_status()
            finally:
                bc_lib.mxfp4_bounds_check_shrink(0)
        assert status == 7
        for w, o in zip(want, outs):
            if w is None:
                continue
            w, o = w.reshape(-1), o.reshape(-1)
            assert torch.all(o[-16:] == 0xA5)            # past the shrunk extent: skipped
            n = o.numel() - 16
            assert torch.equal(o[: n - 32], w[: n - 32])  # well before it: written
