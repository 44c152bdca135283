"""Helpers shared by the GPU parity tests: run the CUDA path and the oracle on
the same seeded inputs and return numpy arrays for element-wise comparison."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth


def cuda_params(p: oracle.Params, layout: int):
    import gemm_pt_block_gb300 as mx

    return mx.QuantParams(block=p.block, scale_mode=p.scale_mode, rounding=p.rounding,
                          scale_layout=layout, wht=p.wht, wht_sign_mask=p.wht_sign_mask,
                          seed=p.seed, sr_stream=p.sr_stream, elem_format=p.elem_format,
                          tensor_exp=p.tensor_exp)


def oracle_input(x: torch.Tensor) -> np.ndarray:
    if x.dtype == torch.bfloat16:
        return synth.bf16_bits(x)
    return x.contiguous().numpy()


def gpu_quantize(x_dev: torch.Tensor, prow, pcol, layout_row=0, layout_col=0):
    import gemm_pt_block_gb300 as mx

    r = mx.mxfp4_quantize(x_dev, cuda_params(prow, layout_row) if prow else None,
                          cuda_params(pcol, layout_col) if pcol else None)
    torch.cuda.synchronize()
    return [None if t is None else t.cpu().numpy() for t in r]


def oracle_quantize(xn: np.ndarray, prow, pcol, layout_row=0, layout_col=0):
    out = [None, None, None, None]
    if prow:
        q, s = oracle.quantize_rows(xn, prow)
        out[0], out[1] = q, (oracle.scales_to_mma(s) if layout_row else s)
    if pcol:
        q, s = oracle.quantize_cols(xn, pcol)
        out[2], out[3] = q, (oracle.scales_to_mma(s) if layout_col else s)
    return out


def assert_same(got, want, what=""):
    for i, (g, w) in enumerate(zip(got, want)):
        if w is None:
            assert g is None
            continue
        g = np.asarray(g).reshape(w.shape)
        if not np.array_equal(g, w):
            bad = np.argwhere(g != w)
            raise AssertionError(f"{what} output {i}: {len(bad)} mismatches, first at {bad[:5].tolist()} "
                                 f"got {g[tuple(bad[0])]} want {w[tuple(bad[0])]}")


def gemm_tolerance_check(c: np.ndarray, ref: np.ndarray, absref: np.ndarray, rel: float = 1e-5):
    err = np.abs(c.astype(np.float64) - ref)
    lim = rel * absref
    ok = err <= lim
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        raise AssertionError(f"{len(bad)} GEMM outputs outside |err| <= {rel} sum|ab|; first {i}: "
                             f"got {c[i]!r} ref {ref[i]!r} sum|ab| {absref[i]!r}")
    return float((err / np.maximum(absref, 1e-300)).max())


def bf16_to_f64(c: torch.Tensor) -> np.ndarray:
    return c.float().cpu().numpy().astype(np.float64)


def gemm_tolerance_check_bf16(c: np.ndarray, ref: np.ndarray, absref: np.ndarray,
                              rel: float = 1e-5):
    """C stored as bf16: the fp32 sum's bound plus bf16's rounding, at most 2^-8
    of the fp32 value (half a unit in the 8th significant bit)."""
    err = np.abs(c - ref)
    t = rel * absref
    lim = t + 2.0 ** -8 * (np.abs(ref) + t)
    ok = err <= lim
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        raise AssertionError(f"{len(bad)} bf16 GEMM outputs outside the bound; first {i}: "
                             f"got {c[i]!r} ref {ref[i]!r} sum|ab| {absref[i]!r}")
