"""Failure detection on the GPU without a fault: a bounded device-side wait is
made to run out (it waits on a barrier that nothing signals), the host reads
MXFP4_ERR_TIMEOUT through the error word, and the same context then runs a
GEMM that still matches the oracle."""
from __future__ import annotations

import time

import pytest
import torch

import oracle
import synth
from _util import gemm_tolerance_check

pytestmark = pytest.mark.gpu

DEV = "cuda"
TIMEOUT = 6   # MXFP4_ERR_TIMEOUT


def test_bounded_wait_runs_out_reports_timeout_and_context_survives():
    import gemm_pt_block_gb300 as mx

    assert mx.device_status() == 0             # nothing pending from earlier tests
    t0 = time.perf_counter()
    mx.selftest_wait_timeout()
    status = mx.device_status()                # synchronizes, reads and clears
    waited = time.perf_counter() - t0
    assert status == TIMEOUT
    assert 1.0 < waited < 60.0                 # the wait ended by its own limit (~2 s)
    assert mx.device_status() == 0             # the word was cleared

    M, N, K = 256, 512, 1024
    qa, qb = synth.random_codes(M, K, 71), synth.random_codes(N, K, 72)
    sa, sb = synth.random_scales(M, K, 73), synth.random_scales(N, K, 74)
    t = [torch.from_numpy(a).to(DEV) for a in (qa, sa, qb, sb)]
    c = mx.mxfp4_gemm(*t, M, N, K)
    torch.cuda.synchronize()
    ref, absref = oracle.gemm_ref(qa, sa, qb, sb, M, N, K)
    gemm_tolerance_check(c.cpu().numpy(), ref, absref)
    assert mx.device_status() == 0
