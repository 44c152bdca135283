"""The benchmark's bookkeeping on CPU: each workload has the shapes and
recipes of the configuration it stands for, and the algorithmic work that the
roofline fractions divide by is the closed form of the step.

Shapes and recipes follow "Pretraining large language models with MXFP4"
(Abstract: Fprop, Dgrad, Wgrad of one linear layer) and "Stable FP4 Training
via Transposition-Invariant Block Quantization" ("The fix, and its supporting
cast": 32x32 blocks on weights and gradients, round-up scales, stochastic
rounding on the backward operands)."""
from __future__ import annotations

import pytest

import bench
import gemm_pt_block_gb300 as mx


def _gemm(spec, label):
    return {g.label: g for g in spec.gemms}[label]


@pytest.mark.parametrize("name,T,D,F", [("70b-layer", 16384, 8192, 28672),
                                        ("8b-mlp-up", 8192, 4096, 14336)])
def test_layer_step_shapes_are_the_three_tn_products(name, T, D, F):
    s = bench.make_spec(name)
    q = {o.name: o for o in s.quants}
    assert (q["X"].rows, q["X"].cols) == (T, D)
    assert (q["W"].rows, q["W"].cols) == (F, D)
    assert (q["dY"].rows, q["dY"].cols) == (T, F)
    # Fprop Y = X W^T, Dgrad dX = dY W, Wgrad dW = dY^T X, each K-major on both sides
    f, d, w = _gemm(s, "Fprop"), _gemm(s, "Dgrad"), _gemm(s, "Wgrad")
    assert (f.M, f.N, f.K, f.a, f.b) == (T, F, D, ("X", "row"), ("W", "row"))
    assert (d.M, d.N, d.K, d.a, d.b) == (T, D, F, ("dY", "row"), ("W", "col"))
    assert (w.M, w.N, w.K, w.a, w.b) == (F, D, T, ("dY", "col"), ("X", "col"))
    # every operand the GEMMs read is produced by the step's quantizers
    for g in s.gemms:
        for ref in (g.a, g.b):
            p = q[ref[0]].prow if ref[1] == "row" else q[ref[0]].pcol
            assert p is not None


def test_layer_step_work_is_the_closed_form():
    s = bench.make_spec("70b-layer")
    T, D, F = 16384, 8192, 28672
    # three GEMMs of 2 T D F flops each (7.70 TFLOP)
    assert s.gemm_flops() == [2.0 * T * D * F] * 3
    assert abs(sum(s.gemm_flops()) - 3 * 7.696581394432e12) < 1e3
    # per quantize: the bf16 input once, then codes (1/2 B) and E8M0 scales
    # (1/32 B) per element for each of the two orientations
    per_orient = 0.5 + 1 / 32
    assert s.quant_bytes() == [T * D * (2 + 2 * per_orient), F * D * (2 + 2 * per_orient),
                               T * F * (2 + 2 * per_orient)]
    nv = bench.make_spec("70b-layer-nvfp4")
    assert nv.quant_bytes()[2] == T * F * (2 + 2 * (0.5 + 1 / 16))   # E4M3 scale per 16


def test_70b_recipe():
    s = bench.make_spec("70b-layer")
    q = {o.name: o for o in s.quants}
    for name in ("W", "dY"):
        assert q[name].prow.block == q[name].pcol.block == mx.BLOCK_32X32
    assert q["X"].prow.block == q["X"].pcol.block == mx.BLOCK_1X32
    assert all(p.scale_mode == mx.SCALE_ROUNDUP for o in s.quants for p in (o.prow, o.pcol))
    # Fprop operands nearest-even without rotation; the Wgrad operands rotated
    # with random signs and rounded stochastically; Dgrad's dY stochastic
    assert q["X"].prow.rounding == q["W"].prow.rounding == q["W"].pcol.rounding == mx.ROUND_RTN
    assert not (q["X"].prow.wht or q["W"].prow.wht or q["W"].pcol.wht or q["dY"].prow.wht)
    assert q["X"].pcol.wht and q["dY"].pcol.wht and q["X"].pcol.wht_sign_mask != 0
    assert q["X"].pcol.wht_sign_mask == q["dY"].pcol.wht_sign_mask     # same D for both operands
    assert q["dY"].prow.rounding == q["dY"].pcol.rounding == q["X"].pcol.rounding == mx.ROUND_SR
    # both orientations of dY draw the same bits for a source element
    assert (q["dY"].prow.seed, q["dY"].prow.sr_stream) == (q["dY"].pcol.seed, q["dY"].pcol.sr_stream)
    assert q["X"].pcol.sr_stream != q["dY"].pcol.sr_stream
    det = bench.make_spec("70b-layer-det")
    assert all(o.pcol.wht_sign_mask == 0 for o in det.quants if o.pcol.wht)


def test_small_configurations():
    tiny = bench.make_spec("tiny")
    assert [(g.M, g.N, g.K) for g in tiny.gemms] == [(512, 512, 1024)]
    assert tiny.gemm_flops() == [2.0 * 512 * 512 * 1024]
    two = bench.make_spec(bench.TWO_D)
    (w,) = two.quants
    assert (w.rows, w.cols) == (4096, 4096)
    assert w.prow == w.pcol and w.prow.block == mx.BLOCK_32X32 and w.prow.rounding == mx.ROUND_RTN
    assert two.quant_bytes() == [4096 * 4096 * (2 + 2 * (0.5 + 1 / 32))]
    assert sorted(bench.SQUARES.values()) == [1024, 2048, 4096, 8192, 16384]


def test_config_object_names_the_workload_and_l2_policy():
    for name in ("70b-layer", "8b-mlp-up", "tiny", bench.TWO_D):
        c = bench.bench_config(bench.make_spec(name), 1)
        assert c["workload"] and c["l2"] and c["parallelism"] == "1 GPU"
    assert "replicas" in bench.bench_config(bench.make_spec("70b-layer"), 4)["parallelism"]
