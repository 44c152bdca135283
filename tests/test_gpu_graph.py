"""The library's calls captured into a CUDA graph: after one eager call per
entry point (which fills the per-device caches), a captured sequence of
quantize, GEMM (with scale images), fused-epilogue GEMM, NVFP4 max-abs +
GEMM and MXFP8 GEMM calls replays to the eager results bit for bit."""
from __future__ import annotations

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _sequence(mx, t):
    """Enqueue every call once on the current stream; outputs in t."""
    mx.mxfp4_quantize(t["x"], t["prow"], t["pcol"], q_row=t["qx"], s_row=t["sx"], q_col=t["qxc"],
                      s_col=t["sxc"])
    mx.mxfp4_quantize(t["w"], t["wp"], q_row=t["qw"], s_row=t["sw"])
    M, N, K = t["shape"]
    mx.mxfp4_gemm(t["qx"], t["sx"], t["qw"], t["sw"], M, N, K, c=t["c"], workspace=t["ws"])
    mx.mxfp4_gemm(t["qx"], t["sx"], t["qw"], t["sw"], M, N, K, c=t["c16"])
    mx.mxfp4_gemm_quantize(t["qx"], t["sx"], t["qw"], t["sw"], M, N, K, t["fp"], col=t["fp"],
                           q_out=t["fq"], s_out=t["fs"], q_col=t["fqc"], s_col=t["fsc"])
    mx.tensor_amax(t["x"], amax=t["amax"], tensor_exp=t["kexp"])
    mx.mxfp4_quantize(t["x"], t["nvp"], q_row=t["nq"], s_row=t["ns"])
    mx.mxfp4_quantize(t["w"], t["nvp"], q_row=t["nwq"], s_row=t["nws"])
    mx.nvfp4_gemm(t["nq"], t["ns"], -1, t["nwq"], t["nws"], -1, M, N, K, c=t["cn"],
                  workspace=t["wsn"])
    mx.mxfp4_quantize(t["x"], t["f8p"], q_row=t["8q"], s_row=t["8s"])
    mx.mxfp4_quantize(t["w"], t["f8p"], q_row=t["8wq"], s_row=t["8ws"])
    mx.mxfp8_gemm(t["8q"], t["8s"], t["8wq"], t["8ws"], M, N, K, c=t["c8"])


def test_step_replays_from_a_cuda_graph_bit_for_bit():
    import gemm_pt_block_gb300 as mx

    M, N, K = 512, 768, 1024
    u8 = dict(dtype=torch.uint8, device=DEV)
    P = mx.QuantParams
    t = {"shape": (M, N, K),
         "x": synth.student_t(M, K, 4.0, seed=31).to(DEV),
         "w": synth.normal(N, K, 0.02, 32).to(DEV),
         "prow": P(mx.BLOCK_1X32, mx.SCALE_ROUNDUP, mx.ROUND_RTN, mx.LAYOUT_MMA),
         "pcol": P(mx.BLOCK_1X32, mx.SCALE_ROUNDUP, mx.ROUND_SR, mx.LAYOUT_MMA, True, 0xBEEF, 7, 0),
         "wp": P(mx.BLOCK_32X32, mx.SCALE_ROUNDUP, mx.ROUND_RTN, mx.LAYOUT_MMA),
         "fp": P(mx.BLOCK_32X32, mx.SCALE_ROUNDUP, mx.ROUND_SR, mx.LAYOUT_MMA, True, 0x1234, 9, 2),
         "nvp": P(mx.BLOCK_1X16, mx.SCALE_ROUNDUP, mx.ROUND_RTN, mx.LAYOUT_MMA, tensor_exp=-1),
         "f8p": P(mx.BLOCK_1X32, mx.SCALE_ROUNDUP, mx.ROUND_RTN, mx.LAYOUT_MMA,
                  elem_format=mx.FORMAT_E4M3)}
    t.update(qx=torch.empty(M, K // 2, **u8), sx=torch.empty(M * K // 32, **u8),
             qxc=torch.empty(K, M // 2, **u8), sxc=torch.empty(M * K // 32, **u8),
             qw=torch.empty(N, K // 2, **u8), sw=torch.empty(N * K // 32, **u8),
             c=torch.empty(M, N, device=DEV), c16=torch.empty(M, N, dtype=torch.bfloat16, device=DEV),
             ws=torch.empty(mx.gemm_workspace_size(M, N, K), **u8),
             fq=torch.empty(M, N // 2, **u8), fs=torch.empty(M * N // 32, **u8),
             fqc=torch.empty(N, M // 2, **u8), fsc=torch.empty(M * N // 32, **u8),
             amax=torch.empty(1, device=DEV), kexp=torch.empty(1, dtype=torch.int32, device=DEV),
             nq=torch.empty(M, K // 2, **u8), ns=torch.empty(M * K // 16, **u8),
             nwq=torch.empty(N, K // 2, **u8), nws=torch.empty(N * K // 16, **u8),
             cn=torch.empty(M, N, device=DEV), wsn=torch.empty(mx.gemm_workspace_size(M, N, K, 16), **u8))
    t.update({"8q": torch.empty(M, K, **u8), "8s": torch.empty(M * K // 32, **u8),
              "8wq": torch.empty(N, K, **u8), "8ws": torch.empty(N * K // 32, **u8),
              "c8": torch.empty(M, N, device=DEV)})
    outs = [k for k, v in t.items() if isinstance(v, torch.Tensor) and k not in ("x", "w", "ws", "wsn")]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _sequence(mx, t)                      # eager: fills the per-device caches
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    want = {k: t[k].clone() for k in outs}

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _sequence(mx, t)
    for _ in range(2):
        for k in outs:
            t[k].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        for k in outs:
            assert torch.equal(t[k], want[k]), k
