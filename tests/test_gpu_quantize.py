"""CUDA quantizer / rotation / dequantize vs the oracle, bit for bit."""
from __future__ import annotations

import itertools

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import assert_same, cuda_params, gpu_quantize, oracle_input, oracle_quantize

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

BLOCKS = [oracle.BLOCK_1X32, oracle.BLOCK_32X32]
SCALES = [oracle.SCALE_FLOOR, oracle.SCALE_ROUNDUP]
ROUNDS = [oracle.ROUND_RTN, oracle.ROUND_SR]
WHTS = [(False, 0), (True, 0), (True, 0x9E3779B9)]


def _input(rows, cols, dtype, seed):
    x = synth.student_t(rows, cols, 3.0, seed)
    if cols >= 64:
        x[:, 5] *= 40          # an outlier channel inside a block
    return x if dtype == "bf16" else x.float()


@pytest.mark.parametrize("orient", ["row", "col", "both"])
@pytest.mark.parametrize("block,scale,rnd", list(itertools.product(BLOCKS, SCALES, ROUNDS)))
@pytest.mark.parametrize("wht", WHTS, ids=["nowht", "detwht", "rndwht"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_quantize_matrix_rowmajor(orient, block, scale, rnd, wht, dtype):
    """Every parameter combination, 160 x 352 (ragged against the 64 x 64 tiles)."""
    rows, cols = 160, 352
    x = _input(rows, cols, dtype, seed=7 + block + 2 * scale)
    p = oracle.Params(block=block, scale_mode=scale, rounding=rnd, wht=wht[0], wht_sign_mask=wht[1],
                      seed=0xABCDEF0123, sr_stream=5)
    prow = p if orient in ("row", "both") else None
    pcol = p if orient in ("col", "both") else None
    got = gpu_quantize(x.to(DEV), prow, pcol)
    want = oracle_quantize(oracle_input(x), prow, pcol)
    assert_same(got, want, f"{orient}")


@pytest.mark.parametrize("orient", ["row", "col", "both"])
@pytest.mark.parametrize("block,rnd", list(itertools.product(BLOCKS, ROUNDS)))
@pytest.mark.parametrize("wht", WHTS[:2], ids=["nowht", "detwht"])
def test_quantize_matrix_mma_layout(orient, block, rnd, wht):
    rows, cols = 256, 384
    x = _input(rows, cols, "bf16", seed=31)
    p = oracle.Params(block=block, scale_mode=oracle.SCALE_ROUNDUP, rounding=rnd, wht=wht[0],
                      wht_sign_mask=wht[1], seed=77, sr_stream=2)
    prow = p if orient in ("row", "both") else None
    pcol = p if orient in ("col", "both") else None
    got = gpu_quantize(x.to(DEV), prow, pcol, 1, 1)
    want = oracle_quantize(oracle_input(x), prow, pcol, 1, 1)
    assert_same(got, want, f"{orient} mma")


@pytest.mark.parametrize("orient", ["row", "col", "both"])
@pytest.mark.parametrize("scale,rnd", list(itertools.product(SCALES, ROUNDS)))
@pytest.mark.parametrize("wht", WHTS, ids=["nowht", "detwht", "rndwht"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_quantize_64x64_blocks(orient, scale, rnd, wht, dtype):
    """64x64 square blocks: the four consumer warps' 32x32 maxima are combined
    per tile; 192 x 320 (3 x 5 tiles)."""
    rows, cols = 192, 320
    x = _input(rows, cols, dtype, seed=91 + scale)
    p = oracle.Params(block=oracle.BLOCK_64X64, scale_mode=scale, rounding=rnd, wht=wht[0],
                      wht_sign_mask=wht[1], seed=0x5EED, sr_stream=4)
    prow = p if orient in ("row", "both") else None
    pcol = p if orient in ("col", "both") else None
    got = gpu_quantize(x.to(DEV), prow, pcol)
    want = oracle_quantize(oracle_input(x), prow, pcol)
    assert_same(got, want, f"64x64 {orient}")


@pytest.mark.parametrize("pair", ["64row_32col", "1row_64col", "64both_mma"])
def test_quantize_64x64_mixed_and_mma(pair):
    rows, cols = 256, 384
    x = _input(rows, cols, "bf16", seed=93)
    b64 = oracle.Params(block=oracle.BLOCK_64X64, scale_mode=oracle.SCALE_ROUNDUP,
                        rounding=oracle.ROUND_SR, seed=3, sr_stream=1)
    if pair == "64row_32col":
        prow, pcol, lay = b64, oracle.Params(block=oracle.BLOCK_32X32, rounding=oracle.ROUND_SR,
                                            wht=True, wht_sign_mask=0x1357, seed=3, sr_stream=1), 0
    elif pair == "1row_64col":
        prow, pcol, lay = oracle.Params(), b64, 0
    else:
        prow, pcol, lay = b64, b64, 1
    got = gpu_quantize(x.to(DEV), prow, pcol, lay, lay)
    want = oracle_quantize(oracle_input(x), prow, pcol, lay, lay)
    assert_same(got, want, pair)


def test_quantize_64x64_rejects_unaligned_shapes():
    import gemm_pt_block_gb300 as mx

    p = mx.QuantParams(block=mx.BLOCK_64X64)
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp4_quantize(torch.zeros(96, 128, device=DEV, dtype=torch.bfloat16), p)
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp4_quantize(torch.zeros(128, 96, device=DEV, dtype=torch.bfloat16), p)


def test_quantize_mixed_orientation_params():
    """Row-wise RTN/floor next to column-wise rotated SR/round-up in one pass."""
    x = synth.laplace(256, 512, 1e-3, seed=41, outlier_frac=0.001)
    pr = oracle.Params(block=oracle.BLOCK_1X32)
    pc = oracle.Params(block=oracle.BLOCK_32X32, scale_mode=oracle.SCALE_ROUNDUP,
                       rounding=oracle.ROUND_SR, wht=True, wht_sign_mask=12345, seed=1, sr_stream=1)
    for lr, lc in [(0, 0), (1, 1), (0, 1)]:
        assert_same(gpu_quantize(x.to(DEV), pr, pc, lr, lc),
                    oracle_quantize(synth.bf16_bits(x), pr, pc, lr, lc), "mixed")
    # both orientations stochastic: separate draws (different streams or seeds) and shared draws
    for pr2 in [oracle.Params(block=oracle.BLOCK_32X32, rounding=oracle.ROUND_SR, seed=1, sr_stream=2),
                oracle.Params(rounding=oracle.ROUND_SR, seed=2, sr_stream=1),
                oracle.Params(block=oracle.BLOCK_32X32, scale_mode=oracle.SCALE_ROUNDUP,
                              rounding=oracle.ROUND_SR, seed=1, sr_stream=1)]:
        assert_same(gpu_quantize(x.to(DEV), pr2, pc, 1, 1),
                    oracle_quantize(synth.bf16_bits(x), pr2, pc, 1, 1), "both SR")


@pytest.mark.parametrize("shape", [(32, 32), (64, 96), (96, 32), (32, 4096), (4128, 64)])
def test_quantize_small_and_ragged_shapes(shape):
    rows, cols = shape
    x = synth.normal(rows, cols, 1.0, seed=rows + cols)
    p = oracle.Params(rounding=oracle.ROUND_SR, wht=True, wht_sign_mask=3, seed=9)
    p2 = oracle.Params(block=oracle.BLOCK_32X32, scale_mode=oracle.SCALE_ROUNDUP)
    for prow, pcol in [(p, None), (p, p2), (p2, p), (None, p)]:
        assert_same(gpu_quantize(x.to(DEV), prow, pcol), oracle_quantize(synth.bf16_bits(x), prow, pcol),
                    f"{shape}")


def test_quantize_every_bf16_pattern():
    """All 65,280 finite bf16 values, as inputs with every block max they produce."""
    u = np.arange(1 << 16, dtype=np.uint32)
    u[((u >> 7) & 0xFF) == 0xFF] = 0
    bits = u.astype(np.uint16).reshape(256, 256)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    for p in [oracle.Params(), oracle.Params(scale_mode=oracle.SCALE_ROUNDUP),
              oracle.Params(rounding=oracle.ROUND_SR, seed=3),
              oracle.Params(block=oracle.BLOCK_32X32, rounding=oracle.ROUND_SR, seed=4)]:
        assert_same(gpu_quantize(x.to(DEV), p, p), oracle_quantize(bits, p, p), "bf16 sweep")
    # With the rotation on, a block sum must stay finite: magnitudes >= 2^122 are zeroed.
    small = bits.copy()
    small[(small & 0x7FFF) >= 0x7C80] = 0
    xs = torch.from_numpy(small.view(np.int16)).view(torch.bfloat16)
    p = oracle.Params(wht=True, wht_sign_mask=0xF0F0F0F0)
    assert_same(gpu_quantize(xs.to(DEV), p, p), oracle_quantize(small, p, p), "bf16 sweep, rotated")


def test_quantize_rtn_midpoints_and_special_values():
    """Exact ties of the grid, their neighbours, signed zeros, tiny and huge values."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    vals = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, 10), -mids,
                           [0.0, -0.0, 1e-40, -1e-42, 6.0, 5.999999, 7.5]]).astype(np.float32)
    nblk = (len(vals) + 30) // 31
    body = np.zeros(nblk * 31, dtype=np.float32)
    body[: len(vals)] = vals
    # one element 6.0 per block pins the scale to 2^0 in round-up mode
    row = np.hstack([np.full((nblk, 1), 6.0, dtype=np.float32), body.reshape(nblk, 31)]).reshape(-1)
    if row.size % 64:
        row = np.concatenate([row, np.full(32, 6.0, dtype=np.float32)])
    x = np.ascontiguousarray(np.tile(row, (32, 1)))
    xt = torch.from_numpy(x)
    for p in [oracle.Params(scale_mode=oracle.SCALE_ROUNDUP),
              oracle.Params(scale_mode=oracle.SCALE_ROUNDUP, rounding=oracle.ROUND_SR, seed=11)]:
        assert_same(gpu_quantize(xt.to(DEV), p, p), oracle_quantize(x, p, p), "midpoints")
    big = np.full((32, 64), 3.0e38, dtype=np.float32)
    big[:, 1::2] = -1.0e-38
    for p in [oracle.Params(), oracle.Params(scale_mode=oracle.SCALE_ROUNDUP)]:
        assert_same(gpu_quantize(torch.from_numpy(big).to(DEV), p, p), oracle_quantize(big, p, p), "big")
    z = torch.zeros(64, 64, dtype=torch.bfloat16)
    got = gpu_quantize(z.to(DEV), oracle.Params(), oracle.Params())
    assert np.all(got[0] == 0) and np.all(got[1] == 0) and np.all(got[2] == 0)
    nz = -z
    got = gpu_quantize(nz.to(DEV), oracle.Params(), None)
    assert np.all(got[0] == 0x88)


def test_quantize_strided_input_and_empty():
    import gemm_pt_block_gb300 as mx

    wide = synth.normal(96, 320, 1.0, seed=5)
    x = wide[:, 32:288]                      # ld = 320 > cols = 256
    p = oracle.Params(rounding=oracle.ROUND_SR, seed=2, wht=True)
    got = gpu_quantize(wide.to(DEV)[:, 32:288], p, p)
    assert_same(got, oracle_quantize(synth.bf16_bits(x.contiguous()), p, p), "strided")
    e = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    q, s, qc, sc = mx.mxfp4_quantize(e, mx.QuantParams(), mx.QuantParams())
    torch.cuda.synchronize()
    assert q.numel() == 0 and qc.numel() == 0


def test_transposition_invariance_on_gpu():
    """32x32 blocks without rotation: column-wise output is the nibble transpose
    of the row-wise one, for RTN and for SR (draws keyed by source index)."""
    x = synth.normal(256, 192, 0.02, seed=1002)
    for rnd in ROUNDS:
        p = oracle.Params(block=oracle.BLOCK_32X32, scale_mode=oracle.SCALE_ROUNDUP, rounding=rnd, seed=8)
        q, s, qc, sc = gpu_quantize(x.to(DEV), p, p)
        def unpack(qq):
            lo, hi = qq & 15, qq >> 4
            return np.stack([lo, hi], axis=-1).reshape(qq.shape[0], -1)
        assert np.array_equal(unpack(q), unpack(qc).T)
        assert np.array_equal(np.repeat(s, 32, 1), np.repeat(sc, 32, 1).T)


@pytest.mark.parametrize("rnd", ROUNDS)
def test_transposition_invariance_full_2d_config(rnd):
    """The 2D-block configuration at full size (W [4096, 4096] N(0, 0.02),
    32x32 blocks, round-up scales, tensor-core scale layout; nearest rounding
    runs the weights profile, whose codes leave by tile stores): column-wise
    codes and scales are exactly the transposes of the row-wise ones, and the
    same tensor in 1x32 blocks has different row- and column-wise scales for a
    large share of its elements. A row band is checked against the oracle."""
    import gemm_pt_block_gb300 as mx

    x = synth.normal(4096, 4096, 0.02, seed=1001)
    p = oracle.Params(block=oracle.BLOCK_32X32, scale_mode=oracle.SCALE_ROUNDUP, rounding=rnd, seed=8)
    q, s, qc, sc = mx.mxfp4_quantize(x.to(DEV), cuda_params(p, 1), cuda_params(p, 1))
    q, s, qc, sc = (t.cpu().numpy() for t in (q, s, qc, sc))

    def unpack(qq):
        return np.stack([qq & 15, qq >> 4], axis=-1).reshape(qq.shape[0], -1)

    def rowmajor(ss, rows):                   # tensor-core layout -> [rows, nkb]
        nkb = ss.size // rows
        idx = np.arange(rows * nkb, dtype=np.int64).reshape(rows, nkb)
        perm = sum(oracle.scales_to_mma(((idx >> (8 * b)) & 255).astype(np.uint8)).astype(np.int64) << (8 * b)
                   for b in range(3))             # row-major index of each layout position
        out = np.empty(rows * nkb, dtype=np.uint8)
        out[perm] = ss.reshape(-1)
        return out.reshape(rows, nkb)

    assert np.array_equal(unpack(q), unpack(qc).T)
    srow, scol = rowmajor(s, 4096), rowmajor(sc, 4096)
    assert np.array_equal(np.repeat(srow, 32, 1), np.repeat(scol, 32, 1).T)
    band = oracle_input(x[:64])
    oq, os_ = oracle.quantize_rows(band, p)
    assert np.array_equal(q[:64], oq) and np.array_equal(srow[:64], os_)
    p1 = oracle.Params(block=oracle.BLOCK_1X32, scale_mode=oracle.SCALE_ROUNDUP, rounding=rnd, seed=8)
    _, s1, _, sc1 = mx.mxfp4_quantize(x.to(DEV), cuda_params(p1, 1), cuda_params(p1, 1))
    r1, c1 = rowmajor(s1.cpu().numpy(), 4096), rowmajor(sc1.cpu().numpy(), 4096)
    mism = np.mean(np.repeat(r1, 32, 1) != np.repeat(c1, 32, 1).T)
    assert 0.3 < mism < 0.7


def test_hadamard32_matches_oracle_and_fused_path():
    import gemm_pt_block_gb300 as mx

    x = synth.normal_outlier_cols(96, 256, 1.0, 8, 50.0, seed=1001)
    xb = synth.bf16_bits(x)
    mask = synth.sign_mask(1001)
    for inv in (False, True):
        y = mx.hadamard32(x.to(DEV), mask, inv).cpu().numpy()
        assert np.array_equal(y, oracle.hadamard32(xb, mask, inv))
    y32 = x.float()
    y = mx.hadamard32(y32.to(DEV), mask).cpu().numpy()
    assert np.array_equal(y, oracle.hadamard32(y32.numpy(), mask))
    back = mx.hadamard32(mx.hadamard32(x.to(DEV), mask), mask, True).cpu().numpy()
    assert np.allclose(back, x.float().numpy(), rtol=1e-5, atol=1e-5)
    # fused rotation == rotation then quantize of the fp32 result
    pf = oracle.Params(rounding=oracle.ROUND_SR, wht=True, wht_sign_mask=mask, seed=4)
    pn = oracle.Params(rounding=oracle.ROUND_SR, seed=4)
    yd = mx.hadamard32(x.to(DEV), mask)
    assert_same(gpu_quantize(x.to(DEV), pf, None), gpu_quantize(yd, pn, None), "fused")


@pytest.mark.parametrize("layout", [0, 1])
def test_dequantize_matches_oracle(layout):
    import gemm_pt_block_gb300 as mx

    rows, cols = 256, 512
    q = synth.random_codes(rows, cols, seed=3)
    s = synth.random_scales(rows, cols, seed=4, lo=0, hi=255)
    got = mx.mxfp4_dequantize(torch.from_numpy(q).to(DEV), torch.from_numpy(s).to(DEV), rows, cols,
                              layout).cpu().numpy()
    want = oracle.dequantize(q, s.reshape(rows, cols // 32) if layout == 0 else s, rows, cols, layout)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


@pytest.mark.parametrize("rows,cols,seed", [(8192, 4096, 1003), (4096, 4096, 1002)])
def test_quantize_full_size_sampled(rows, cols, seed):
    """Workload-sized tensors in the launch configuration the benchmark times;
    the oracle checks sampled 32-row bands and 32-column bands."""
    x = synth.student_t(rows, cols, 4.0, seed) if seed == 1003 else synth.normal(rows, cols, 0.02, seed)
    xb = synth.bf16_bits(x)
    pr = oracle.Params(block=oracle.BLOCK_1X32)
    pc = oracle.Params(block=oracle.BLOCK_1X32, rounding=oracle.ROUND_SR, wht=True, seed=1, sr_stream=0)
    if seed == 1002:
        pr = pc = oracle.Params(block=oracle.BLOCK_32X32, scale_mode=oracle.SCALE_ROUNDUP)
    q, s, qc, sc = gpu_quantize(x.to(DEV), pr, pc)
    for r0 in [0, rows // 2 + 32, rows - 32]:
        rq, rs = oracle.quantize_rows(xb, pr, r0, r0 + 32)
        assert np.array_equal(q[r0:r0 + 32], rq) and np.array_equal(s[r0:r0 + 32], rs)
    for c0 in [0, cols // 3 // 32 * 32, cols - 32]:
        cq, cs = oracle.quantize_cols(xb, pc, c0, c0 + 32)
        assert np.array_equal(qc[c0:c0 + 32], cq) and np.array_equal(sc[c0:c0 + 32], cs)


def test_quantize_is_deterministic_across_calls_and_streams():
    import gemm_pt_block_gb300 as mx

    x = synth.student_t(512, 1024, 4.0, seed=99).to(DEV)
    p = mx.QuantParams(rounding=mx.ROUND_SR, wht=True, wht_sign_mask=77, seed=3)
    a = mx.mxfp4_quantize(x, p, p)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = mx.mxfp4_quantize(x, p, p)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_nearest_even_dense_fp32_sweep():
    """Scaled values v in (-8, 8): every 256th fp32 pattern, plus 2048 ulps either
    side of every grid point and midpoint, both signs. A 4.0 in each block pins
    the floor-mode scale to 2^0, so v = x and values above 6 saturate. Both
    nearest-even and stochastic rounding must match the oracle exactly."""
    coarse = np.arange(0, 0x41000000, 256, dtype=np.uint32)
    pts = np.array([0, .25, .5, .75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6, 7], dtype=np.float32)
    fine = (pts.view(np.uint32)[:, None].astype(np.int64) + np.arange(-2048, 2049)[None, :]).reshape(-1)
    fine = fine[(fine >= 0) & (fine < 0x41000000)].astype(np.uint32)
    vals = np.concatenate([coarse, fine]).view(np.float32)
    vals = np.concatenate([vals, -vals])
    n_blk = (vals.size + 30) // 31
    body = np.zeros(n_blk * 31, dtype=np.float32)
    body[: vals.size] = vals
    blocks = np.hstack([np.full((n_blk, 1), 4.0, np.float32), body.reshape(n_blk, 31)])
    cols = 4096
    n_rows = (blocks.size + cols - 1) // cols
    n_rows = (n_rows + 31) // 32 * 32
    flat = np.full(n_rows * cols, 4.0, dtype=np.float32)
    flat[: blocks.size] = blocks.reshape(-1)
    x = flat.reshape(n_rows, cols)
    xt = torch.from_numpy(x).to(DEV)
    for p in [oracle.Params(), oracle.Params(rounding=oracle.ROUND_SR, seed=5, sr_stream=9)]:
        got = gpu_quantize(xt, p, None)
        want = oracle_quantize(x, p, None)
        assert np.all(want[1] == 127)
        assert_same(got, want, "dense fp32 sweep")


# ------------------------------------------------------------------ MXFP8 --

@pytest.mark.parametrize("orient", ["row", "col", "both"])
@pytest.mark.parametrize("block", [oracle.BLOCK_1X32, oracle.BLOCK_32X32, oracle.BLOCK_64X64])
@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("wht", WHTS[:2], ids=["nowht", "detwht"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_mxfp8_matches_oracle(orient, block, scale, wht, dtype):
    """E4M3 elements with E8M0 block scales, one byte per element."""
    rows, cols = (192, 320) if block == oracle.BLOCK_64X64 else (160, 352)
    if orient == "row" and block == oracle.BLOCK_1X32:
        rows = 150                         # row kernel, ragged row count
    x = _input(rows, cols, dtype, seed=101 + block)
    p = oracle.Params(block=block, scale_mode=scale, wht=wht[0], wht_sign_mask=wht[1],
                      elem_format=oracle.FORMAT_E4M3)
    prow = p if orient in ("row", "both") else None
    pcol = p if orient in ("col", "both") else None
    got = gpu_quantize(x.to(DEV), prow, pcol)
    want = oracle_quantize(oracle_input(x), prow, pcol)
    assert_same(got, want, f"mxfp8 {orient}")


def test_mxfp8_every_bf16_value_and_mma_layout():
    """Every finite bf16 pattern as input (all block maxima, subnormals,
    saturation), row-wise; then the tensor-core scale layout."""
    import gemm_pt_block_gb300 as mx

    bits = np.arange(65536, dtype=np.uint32)
    keep = (bits & 0x7F80) != 0x7F80
    vals = bits[keep].astype(np.uint16)
    n = (vals.size // 64) * 64
    x = vals[:n].reshape(-1, 64)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    p = oracle.Params(elem_format=oracle.FORMAT_E4M3, scale_mode=oracle.SCALE_ROUNDUP)
    got = gpu_quantize(xt.to(DEV), p, None)
    want = oracle_quantize(x, p, None)
    assert_same(got, want, "mxfp8 bf16 sweep")
    xm = _input(256, 384, "bf16", seed=103)
    pm = oracle.Params(block=oracle.BLOCK_32X32, elem_format=oracle.FORMAT_E4M3)
    assert_same(gpu_quantize(xm.to(DEV), pm, pm, 1, 1), oracle_quantize(oracle_input(xm), pm, pm, 1, 1),
                "mxfp8 mma")
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp4_quantize(xm.to(DEV), mx.QuantParams(rounding=mx.ROUND_SR, elem_format=mx.FORMAT_E4M3))


PROFILES = {   # (row rounding, row rotation, column rounding, column rotation)
    "weights": (oracle.ROUND_RTN, False, oracle.ROUND_RTN, False),
    "activations": (oracle.ROUND_RTN, False, oracle.ROUND_SR, True),
    "gradients": (oracle.ROUND_SR, False, oracle.ROUND_SR, True),
}


@pytest.mark.parametrize("profile", sorted(PROFILES))
@pytest.mark.parametrize("block,scale", list(itertools.product(BLOCKS, SCALES)))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("same_stream", [True, False])
def test_quantize_dual_profiles(profile, block, scale, dtype, same_stream):
    """The dual-orientation recipes that take compile-time kernel profiles
    (weights, activations, output gradients), ragged 160 x 352, against the
    oracle; with and without shared draws between the orientations."""
    rr, rw, cr, cw = PROFILES[profile]
    x = _input(160, 352, dtype, seed=131 + block)
    prow = oracle.Params(block=block, scale_mode=scale, rounding=rr, wht=rw, seed=11, sr_stream=3)
    pcol = oracle.Params(block=block, scale_mode=scale, rounding=cr, wht=cw, wht_sign_mask=0x0BADF00D,
                         seed=11, sr_stream=3 if same_stream else 4)
    got = gpu_quantize(x.to(DEV), prow, pcol)
    want = oracle_quantize(oracle_input(x), prow, pcol)
    assert_same(got, want, profile)
