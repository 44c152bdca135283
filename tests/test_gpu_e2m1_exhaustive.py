"""Every fp32 value in (-8, 8) through the quantizer's E2M1 rounding, against
the oracle, in both rounding modes.

The nearest-even path uses the hardware conversion cvt.rn.satfinite.e2m1x2.f32;
it may stand in for the oracle's direct search only if the two agree on every
value the conversion can see. Stochastic rounding computes its result with an
exact-ceiling construction in fp32 that is argued, not searched; here every
value meets one Philox draw keyed by its source index, the same draw the
oracle takes. Each 32-element block holds a 4.0 and 31 test values, so the
floor-mode scale is 2^0 and the conversion sees the values themselves (those
above 6 saturate). Both signs, in chunks of 2^26 bit patterns.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CHUNK = 1 << 26
END = 0x41000000                       # bit pattern of 8.0: [0, END) covers [0, 8)


def _blocks(first: int, n: int, negative: bool) -> tuple[np.ndarray, int]:
    bits = np.arange(first, first + n, dtype=np.uint32)
    if negative:
        bits |= np.uint32(0x80000000)
    n_blk = (n + 30) // 31
    x = np.full((n_blk, 32), 4.0, dtype=np.float32)
    body = x[:, 1:].reshape(-1)
    body[:n] = bits.view(np.float32)
    x[:, 1:] = body.reshape(n_blk, 31)
    return x, n_blk


def _codes(q: np.ndarray) -> np.ndarray:
    c = np.empty((q.shape[0], 2 * q.shape[1]), dtype=np.uint8)
    c[:, 0::2] = q & 0xF
    c[:, 1::2] = q >> 4
    return c


@pytest.mark.parametrize("rounding", [oracle.ROUND_RTN, oracle.ROUND_SR], ids=["nearest", "stochastic"])
def test_every_fp32_in_open_interval_8(rounding):
    import gemm_pt_block_gb300 as mx

    p = oracle.Params(rounding=rounding, seed=0x5EED, sr_stream=3)
    cp = mx.QuantParams(rounding=rounding, seed=0x5EED, sr_stream=3)
    checked = 0
    for negative in (False, True):
        for first in range(0, END, CHUNK):
            n = min(CHUNK, END - first)
            x, n_blk = _blocks(first, n, negative)
            q, s, _, _ = mx.mxfp4_quantize(torch.from_numpy(x).to(DEV), cp)
            got_q, got_s = q.cpu().numpy(), s.cpu().numpy()
            want_q, want_s = oracle.quantize_rows(x, p)
            assert np.all(want_s == 127) and np.array_equal(got_s, want_s)
            if not np.array_equal(got_q, want_q):
                g = _codes(got_q)[:, 1:].reshape(-1)[:n]
                w = _codes(want_q)[:, 1:].reshape(-1)[:n]
                bad = np.flatnonzero(g != w)
                j = int(bad[0])
                bits = (first + j) | (0x80000000 if negative else 0)
                raise AssertionError(f"{bad.size} codes differ in chunk {first:#x}; first: fp32 bits "
                                     f"{bits:#010x} gpu {g[j]:#x} oracle {w[j]:#x}")
            checked += n
    assert checked == 2 * END
    assert mx.device_status() == 0
