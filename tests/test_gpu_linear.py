"""MXFP4 linear layer (forward Fprop, backward Dgrad and Wgrad through autograd)
against the oracle: each product must equal the fp64 product of the oracle's
quantized operands within |C - ref| <= 1e-5 * sum_k |a_k b_k|."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import gemm_tolerance_check

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _op(p):
    return oracle.Params(p.block, p.scale_mode, p.rounding, p.wht, p.wht_sign_mask, p.seed,
                         p.sr_stream)


def _rows(x, p):
    q, s = oracle.quantize_rows(x, _op(p))
    return q, oracle.scales_to_mma(s)


def _cols(x, p):
    q, s = oracle.quantize_cols(x, _op(p))
    return q, oracle.scales_to_mma(s)


@pytest.mark.parametrize("recipe_name,T,D,F", [("2d_sr", 256, 512, 768), ("1d", 512, 256, 256),
                                                ("2d_sr", 384, 640, 384), ("1d", 128, 384, 640)])
def test_linear_forward_backward_match_oracle(recipe_name, T, D, F):
    import gemm_pt_block_gb300 as mx

    mask = synth.sign_mask(4242)
    recipe = (mx.recipe_2d_sr if recipe_name == "2d_sr" else mx.recipe_1d)(mask, seed=7)
    x = synth.student_t(T, D, 4.0, 4300).float().numpy()
    w = synth.normal(F, D, 0.02, 4301).float().numpy()
    g = synth.laplace(T, F, 1e-3, 4302).float().numpy()

    xd = torch.from_numpy(x).to(DEV).requires_grad_()
    wd = torch.from_numpy(w).to(DEV).requires_grad_()
    y = mx.mxfp4_linear(xd, wd, recipe)
    y.backward(torch.from_numpy(g).to(DEV))
    torch.cuda.synchronize()
    assert mx.device_status() == 0

    xq, xs = _rows(x, recipe.x_row)
    wq, ws = _rows(w, recipe.w_row)
    ref, ab = oracle.gemm_ref(xq, xs, wq, ws, T, F, D)
    gemm_tolerance_check(y.detach().cpu().numpy(), ref, ab)

    gq, gs = _rows(g, recipe.dy_row)
    wqc, wsc = _cols(w, recipe.w_col)
    ref, ab = oracle.gemm_ref(gq, gs, wqc, wsc, T, D, F)
    gemm_tolerance_check(xd.grad.cpu().numpy(), ref, ab)

    gqc, gsc = _cols(g, recipe.dy_col)
    xqc, xsc = _cols(x, recipe.x_col)
    ref, ab = oracle.gemm_ref(gqc, gsc, xqc, xsc, F, D, T)
    gemm_tolerance_check(wd.grad.cpu().numpy(), ref, ab)


def test_linear_module_bf16_and_fresh_draws_per_step():
    import gemm_pt_block_gb300 as mx

    layer = mx.Mxfp4Linear(512, 256, device=DEV)
    x = torch.randn(2, 128, 512, device=DEV, dtype=torch.bfloat16, requires_grad=True)
    y1 = layer(x)
    assert y1.shape == (2, 128, 256) and y1.dtype == torch.float32
    y1.sum().backward()
    g1 = layer.weight.grad.clone()
    assert layer.weight.grad.dtype == torch.bfloat16 and x.grad.dtype == torch.bfloat16
    layer.weight.grad = None
    layer(x).sum().backward()          # next step: new stochastic-rounding seeds
    assert layer.step == 2
    assert not torch.equal(g1, layer.weight.grad)
    assert torch.isfinite(layer.weight.grad.float()).all()


def test_linear_rejects_unsupported_shapes():
    import gemm_pt_block_gb300 as mx

    with pytest.raises(ValueError):      # T not a multiple of 128
        mx.mxfp4_linear(torch.zeros(192, 256, device=DEV), torch.zeros(256, 256, device=DEV))
    with pytest.raises(ValueError):      # F not a multiple of 128
        mx.mxfp4_linear(torch.zeros(256, 256, device=DEV), torch.zeros(320, 256, device=DEV))


def test_first_call_from_a_fresh_thread():
    """Framework worker threads (autograd's backward runs on one) may call in
    before anything has bound the device's context in that thread."""
    import threading

    import gemm_pt_block_gb300 as mx

    x = torch.randn(256, 768, device=DEV)
    r = mx.recipe_2d_sr(0x5A5A5A5A, 3)
    ref = mx.mxfp4_quantize(x, r.dy_row, r.dy_col)
    torch.cuda.synchronize()
    box = {}

    def work():
        try:
            box["out"] = mx.mxfp4_quantize(x, r.dy_row, r.dy_col)
            torch.cuda.synchronize()
        except Exception as e:  # noqa: BLE001 - reported below
            box["err"] = e

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert "err" not in box, box.get("err")
    assert all(torch.equal(a, b) for a, b in zip(box["out"], ref))


def test_linear_bf16_output_and_direct_bf16_gradients():
    """out_dtype=bf16: Y is the fp32 layer's Y rounded to nearest-even; with the
    same dY values the gradients are bit-identical to the fp32-output layer's
    (each written by the GEMM in its input's dtype)."""
    import gemm_pt_block_gb300 as mx

    T, D, F = 256, 512, 768
    r = mx.recipe_2d_sr(synth.sign_mask(77), seed=5)
    x = synth.student_t(T, D, 4.0, 4400).to(DEV)
    w = synth.normal(F, D, 0.02, 4401).to(DEV)
    g = synth.laplace(T, F, 1e-3, 4402).to(DEV)          # bf16
    outs = {}
    for dt in (torch.float32, torch.bfloat16):
        xd, wd = x.clone().requires_grad_(), w.clone().requires_grad_()
        y = mx.mxfp4_linear(xd, wd, r, out_dtype=dt)
        y.backward(g.to(dt))
        torch.cuda.synchronize()
        outs[dt] = (y.detach(), xd.grad, wd.grad)
    y32, dx32, dw32 = outs[torch.float32]
    y16, dx16, dw16 = outs[torch.bfloat16]
    assert y16.dtype == torch.bfloat16 and dx16.dtype == torch.bfloat16 and dw16.dtype == torch.bfloat16
    assert torch.equal(y16.view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(dx16.view(torch.int16), dx32.view(torch.int16))
    assert torch.equal(dw16.view(torch.int16), dw32.view(torch.int16))


def test_linear_partial_gradients_match_full_run():
    """With only W (or only X) wanting a gradient, or none (no_grad), the layer
    skips the orientations whose products do not run; Y and the gradients it
    does compute are bit-identical to the run that computes everything."""
    import gemm_pt_block_gb300 as mx

    T, D, F = 256, 512, 768
    r = mx.recipe_2d_sr(synth.sign_mask(91), seed=11)
    x = synth.student_t(T, D, 4.0, 4500).to(DEV)
    w = synth.normal(F, D, 0.02, 4501).to(DEV)
    g = synth.laplace(T, F, 1e-3, 4502).float().to(DEV)

    def run(gx, gw):
        xd, wd = x.clone().requires_grad_(gx), w.clone().requires_grad_(gw)
        y = mx.mxfp4_linear(xd, wd, r)
        if gx or gw:
            y.backward(g)
        torch.cuda.synchronize()
        return y.detach(), xd.grad, wd.grad

    y, dx, dw = run(True, True)
    y_w, dx_w, dw_w = run(False, True)
    y_x, dx_x, dw_x = run(True, False)
    with torch.no_grad():
        y_n = mx.mxfp4_linear(x, w, r)
    torch.cuda.synchronize()
    assert dx_w is None and dw_x is None
    for yy in (y_w, y_x, y_n):
        assert torch.equal(yy, y)
    assert torch.equal(dw_w, dw)
    assert torch.equal(dx_x, dx)
