"""Parity at the exact launches the benchmark times on the 70B-dense-shaped
layer (tokens 16384, d 8192, ffn 28672): the three dual-orientation quantizer
calls with the step's own inputs and parameters (activation X, weight W,
output gradient dY, each on its compile-time kernel profile), and the Fprop
and Wgrad GEMM shapes on the scale-image path.

The oracle checks sampled bands: 32-row bands of the row-wise output and
32-column bands of the column-wise output at the start, the middle and the end,
plus the tile rows (64-row) 1, 2 and 3, where the persistent tile kernel's CTAs
take their second, third and fourth tiles (the third stage of the load ring
wraps there) for every grid size the kernel can be launched with on one GPU.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bench
import oracle
import synth
from _util import gemm_tolerance_check

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _oracle_params(p):
    return oracle.Params(p.block, p.scale_mode, p.rounding, p.wht, p.wht_sign_mask, p.seed,
                         p.sr_stream, p.elem_format, p.tensor_exp)


def _mma_rows(s_mma: np.ndarray, r0: int, nrows: int, total_rows: int, nkb: int) -> np.ndarray:
    """Rows r0 .. r0 + nrows of a scale array stored in the tensor-core layout,
    gathered into row-major order."""
    offs = np.array([[oracle.mma_scale_offset(r, kb, total_rows, nkb) for kb in range(nkb)]
                     for r in range(r0, r0 + nrows)], dtype=np.int64)
    return s_mma[offs]


@pytest.mark.parametrize("name", ["X", "W", "dY"])
def test_70b_step_quantizer_launch_matches_oracle(name):
    import gemm_pt_block_gb300 as mx

    spec = bench.make_spec("70b-layer")
    q = {o.name: o for o in spec.quants}[name]
    x = bench.gen_input(q, torch.device(DEV))
    qr, sr, qc, sc = mx.mxfp4_quantize(x, q.prow, q.pcol)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    xb = synth.bf16_bits(x.cpu())
    rows, cols = q.rows, q.cols
    qr, sr, qc, sc = (t.cpu().numpy() for t in (qr, sr, qc, sc))
    pr, pc = _oracle_params(q.prow), _oracle_params(q.pcol)
    for r0 in sorted({0, 64, 128, 192, 288, rows // 2 + 32, rows - 32}):
        wq, ws = oracle.quantize_rows(xb, pr, r0, r0 + 32)
        assert np.array_equal(qr[r0:r0 + 32], wq), (name, "row codes", r0)
        assert np.array_equal(_mma_rows(sr, r0, 32, rows, cols // 32), ws), (name, "row scales", r0)
    for c0 in sorted({0, 64, 544, cols // 2 + 32, cols - 32}):
        wq, ws = oracle.quantize_cols(xb, pc, c0, c0 + 32)
        assert np.array_equal(qc[c0:c0 + 32], wq), (name, "column codes", c0)
        assert np.array_equal(_mma_rows(sc, c0, 32, cols, rows // 32), ws), (name, "column scales", c0)


@pytest.mark.parametrize("label", ["Fprop", "Wgrad"])
def test_70b_step_gemm_shape_on_image_path(label):
    """The GEMM launch the benchmark times (scale-image workspace) against the
    plain entry point bit for bit and against the oracle's fp64 sums on
    sampled output elements of full rows."""
    import gemm_pt_block_gb300 as mx

    g = {o.label: o for o in bench.make_spec("70b-layer").gemms}[label]
    M, N, K = g.M, g.N, g.K
    gen = torch.Generator(device=DEV).manual_seed(M ^ K)
    qa = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=DEV, generator=gen)
    qb = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=DEV, generator=gen)
    sa = torch.randint(118, 137, (M * K // 32,), dtype=torch.uint8, device=DEV, generator=gen)
    sb = torch.randint(118, 137, (N * K // 32,), dtype=torch.uint8, device=DEV, generator=gen)
    ws = torch.empty(mx.gemm_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    img = mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K, workspace=ws)
    plain = mx.mxfp4_gemm(qa, sa, qb, sb, M, N, K, workspace=False)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert torch.equal(img, plain)
    rows = np.array([0, 255, 256, M // 2 + 129, M - 1])
    ms = np.repeat(rows, 48)
    ns = np.tile(np.linspace(0, N - 1, 48).astype(np.int64), len(rows))
    ref, absref = oracle.gemm_pairs(qa.cpu().numpy(), sa.cpu().numpy(), qb.cpu().numpy(),
                                    sb.cpu().numpy(), M, N, K, ms, ns)
    gemm_tolerance_check(img[torch.from_numpy(ms), torch.from_numpy(ns)].cpu().numpy(), ref, absref)
