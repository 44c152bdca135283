"""MXFP4 linear layer for training: forward and backward through the library's
kernels, with the straight-through estimator.

For Y = X W^T (X [T, D], W [F, D]) the three products are block-scaled MXFP4
GEMMs of quantized operands (Cim, "Pretraining large language models with
MXFP4", Abstract: Fprop, Dgrad and Wgrad):

    Fprop  Y  [T, F] = Xq  . Wq^T      X row-wise,  W row-wise
    Dgrad  dX [T, D] = dYq . Wq        dY row-wise, W column-wise (W^T row-wise)
    Wgrad  dW [F, D] = dYq^T . Xq      dY column-wise, X column-wise

Each tensor is quantized once per pass in both orientations it needs (TIBQ,
"The aha: transposition scrambles the blocks"); the backward pass reuses the
column-wise X and W codes written by the forward pass. An orientation whose
product will not run (no gradient wanted for X or W) is not produced. Gradients flow through
the quantizers unchanged (straight-through). Rotating the Wgrad operands
along T with the same random-sign mask leaves dW's expectation unchanged,
since c H diag(s) is orthogonal (Tseng, "Training LLMs with MXFP4",
Abstract: stochastic rounding with the random Hadamard transform).

Everything runs in the library's CUDA kernels; this module only chains the
calls and keeps the codes between the passes. The GEMMs accumulate in fp32
and store their result in the type it is wanted in: Y in `out_dtype` (fp32 by
default, or bf16), dX in X's dtype and dW in W's dtype (bf16 is the fp32 sum
rounded to nearest-even inside the GEMM's epilogue, so no separate cast runs).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

from .binding import (BLOCK_1X32, BLOCK_32X32, LAYOUT_MMA, ROUND_RTN, ROUND_SR, SCALE_FLOOR,
                      SCALE_ROUNDUP, QuantParams, mxfp4_gemm, mxfp4_quantize)


@dataclass(frozen=True)
class LinearRecipe:
    """Quantization of each operand orientation (scale layouts must be the
    tensor-core layout, which the GEMM consumes)."""
    x_row: QuantParams
    x_col: QuantParams
    w_row: QuantParams
    w_col: QuantParams
    dy_row: QuantParams
    dy_col: QuantParams


def recipe_2d_sr(sign_mask: int = 0, seed: int = 0) -> LinearRecipe:
    """Activations in 1x32 blocks, weights and output gradients in 32x32 blocks
    (TIBQ, "The fix, and its supporting cast"), truncation-free (round-up)
    scales; nearest-even for the forward operands, stochastic rounding for the
    gradient, rotation + stochastic rounding for the Wgrad operands (X and dY
    column-wise, one shared sign mask; mask 0 = deterministic rotation).
    Streams: X 0, dY 1; both orientations of dY share their draws."""
    P = QuantParams
    x_row = P(BLOCK_1X32, SCALE_ROUNDUP, ROUND_RTN, LAYOUT_MMA)
    x_col = P(BLOCK_1X32, SCALE_ROUNDUP, ROUND_SR, LAYOUT_MMA, True, sign_mask, seed, 0)
    w = P(BLOCK_32X32, SCALE_ROUNDUP, ROUND_RTN, LAYOUT_MMA)
    dy_row = P(BLOCK_32X32, SCALE_ROUNDUP, ROUND_SR, LAYOUT_MMA, False, 0, seed, 1)
    dy_col = P(BLOCK_32X32, SCALE_ROUNDUP, ROUND_SR, LAYOUT_MMA, True, sign_mask, seed, 1)
    return LinearRecipe(x_row, x_col, w, w, dy_row, dy_col)


def recipe_1d(sign_mask: int = 0, seed: int = 0) -> LinearRecipe:
    """All operands in 1x32 blocks with OCP floor scales; nearest-even for
    Fprop and Dgrad operands; rotation + stochastic rounding for the Wgrad
    operands only (X and dY column-wise)."""
    P = QuantParams
    rtn = P(BLOCK_1X32, SCALE_FLOOR, ROUND_RTN, LAYOUT_MMA)
    x_col = P(BLOCK_1X32, SCALE_FLOOR, ROUND_SR, LAYOUT_MMA, True, sign_mask, seed, 0)
    dy_col = P(BLOCK_1X32, SCALE_FLOOR, ROUND_SR, LAYOUT_MMA, True, sign_mask, seed, 1)
    return LinearRecipe(rtn, x_col, rtn, rtn, rtn, dy_col)


def _check_shapes(T: int, D: int, F: int) -> None:
    # GEMMs (T,F,D), (T,D,F), (F,D,T) need M, N, K multiples of 128; so does the
    # tensor-core scale layout of every quantized operand.
    if T % 128 or D % 128 or F % 128:
        raise ValueError(f"MXFP4 linear needs T, D, F multiples of 128 (got {T}, {D}, {F})")


class _Mxfp4LinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x: torch.Tensor, w: torch.Tensor, recipe: LinearRecipe, step: int,
                out_dtype: torch.dtype):
        T, D = x.shape
        F = w.shape[0]
        _check_shapes(T, D, F)
        r = recipe
        if step:   # fresh stochastic-rounding draws per training step
            r = replace(r, x_col=replace(r.x_col, seed=r.x_col.seed + step),
                        dy_row=replace(r.dy_row, seed=r.dy_row.seed + step),
                        dy_col=replace(r.dy_col, seed=r.dy_col.seed + step))
        # Column-wise codes only for the backward products that will run:
        # X^T feeds Wgrad (dW), W^T feeds Dgrad (dX).
        need_dx, need_dw = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        xq, xs, xqc, xsc = mxfp4_quantize(x, r.x_row, r.x_col if need_dw else None)
        wq, ws, wqc, wsc = mxfp4_quantize(w, r.w_row, r.w_col if need_dx else None)
        y = mxfp4_gemm(xq, xs, wq, ws, T, F, D, out_dtype=out_dtype)
        ctx.save_for_backward(xqc, xsc, wqc, wsc)
        ctx.recipe, ctx.dims, ctx.dtypes = r, (T, D, F), (x.dtype, w.dtype)
        return y

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        xqc, xsc, wqc, wsc = ctx.saved_tensors
        T, D, F = ctx.dims
        r = ctx.recipe
        need_dx, need_dw = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        dy = dy.contiguous()
        # dY row-wise feeds Dgrad, dY column-wise Wgrad; each element's draw
        # is keyed by its source index, so either one alone has the same bits.
        gq, gs, gqc, gsc = mxfp4_quantize(dy, r.dy_row if need_dx else None,
                                          r.dy_col if need_dw else None)
        xdt, wdt = ctx.dtypes
        dx = mxfp4_gemm(gq, gs, wqc, wsc, T, D, F, out_dtype=xdt) if need_dx else None
        dw = mxfp4_gemm(gqc, gsc, xqc, xsc, F, D, T, out_dtype=wdt) if need_dw else None
        return dx, dw, None, None, None


def mxfp4_linear(x: torch.Tensor, w: torch.Tensor, recipe: LinearRecipe | None = None,
                 step: int = 0, out_dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """Y = X W^T with MXFP4 forward and backward GEMMs; Y in out_dtype (fp32 or
    bf16), gradients in their inputs' dtypes.

    x [T, D] and w [F, D] are bf16 or fp32 CUDA tensors; T, D, F must be
    multiples of 128. `step` offsets the stochastic-rounding seeds so each
    training step draws fresh bits."""
    for t, n in ((x, "x"), (w, "w")):
        if t.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError(f"{n} must be bfloat16 or float32")
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out_dtype must be bfloat16 or float32")
    return _Mxfp4LinearFn.apply(x, w, recipe or recipe_2d_sr(), step, out_dtype)


class Mxfp4Linear(torch.nn.Module):
    """Bias-free linear layer whose three GEMMs run in MXFP4."""

    def __init__(self, in_features: int, out_features: int, recipe: LinearRecipe | None = None,
                 device=None, dtype=torch.bfloat16, out_dtype: torch.dtype = torch.float32):
        super().__init__()
        self.out_dtype = out_dtype
        self.weight = torch.nn.Parameter(torch.empty(out_features, in_features, device=device,
                                                     dtype=dtype))
        torch.nn.init.normal_(self.weight, std=in_features ** -0.5)
        self.recipe = recipe or recipe_2d_sr()
        self.step = 0

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        lead = x.shape[:-1]
        y = mxfp4_linear(x.reshape(-1, x.shape[-1]), self.weight, self.recipe, self.step,
                         self.out_dtype)
        if self.training:
            self.step += 1
        return y.reshape(*lead, y.shape[-1])
