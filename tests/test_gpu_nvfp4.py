"""NVFP4 (1x16 E2M1 blocks with E4M3 scales under a power-of-two tensor factor):
the CUDA quantizer bit for bit against the oracle, and the NVFP4 GEMM
(tcgen05 kind::mxf4nvf4) within the GEMM tolerance of the fp64 product."""
from __future__ import annotations

import itertools

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import (assert_same, bf16_to_f64, cuda_params, gemm_tolerance_check,
                   gemm_tolerance_check_bf16, gpu_quantize, oracle_input, oracle_quantize)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

SCALES = [oracle.SCALE_FLOOR, oracle.SCALE_ROUNDUP]
ROUNDS = [oracle.ROUND_RTN, oracle.ROUND_SR]
WHTS = [(False, 0), (True, 0), (True, 0x9E3779B9)]


def _k(x: torch.Tensor) -> int:
    """The tensor's NVFP4 exponent as the oracle defines it."""
    return oracle.nv_tensor_exp(oracle.tensor_amax(oracle_input(x.cpu())))


def _input(rows, cols, dtype, seed, scale=1.0):
    x = synth.student_t(rows, cols, 3.0, seed)
    if cols >= 64:
        x[:, 5] *= 40
    x = (x.float() * scale)
    return x.to(torch.bfloat16) if dtype == "bf16" else x


@pytest.mark.parametrize("orient", ["row", "col", "both"])
@pytest.mark.parametrize("scale,rnd", list(itertools.product(SCALES, ROUNDS)))
@pytest.mark.parametrize("wht", WHTS, ids=["nowht", "detwht", "rndwht"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_nvfp4_quantize_matrix(orient, scale, rnd, wht, dtype):
    """Every parameter combination, 160 x 352 (ragged against the 64 x 64 tiles),
    tensor factor from the tensor's max-abs."""
    rows, cols = 160, 352
    x = _input(rows, cols, dtype, seed=17 + scale)
    p = oracle.Params(block=oracle.BLOCK_1X16, scale_mode=scale, rounding=rnd, wht=wht[0],
                      wht_sign_mask=wht[1], seed=0xABCDEF0123, sr_stream=5, tensor_exp=_k(x))
    prow = p if orient in ("row", "both") else None
    pcol = p if orient in ("col", "both") else None
    got = gpu_quantize(x.to(DEV), prow, pcol)
    want = oracle_quantize(oracle_input(x), prow, pcol)
    assert_same(got, want, f"nvfp4 {orient}")


@pytest.mark.parametrize("orient", ["row", "col", "both"])
@pytest.mark.parametrize("rnd", ROUNDS)
def test_nvfp4_quantize_mma_layout(orient, rnd):
    rows, cols = 256, 384
    x = _input(rows, cols, "bf16", seed=33)
    p = oracle.Params(block=oracle.BLOCK_1X16, scale_mode=oracle.SCALE_ROUNDUP, rounding=rnd,
                      wht=True, wht_sign_mask=0x1234567, seed=78, sr_stream=3, tensor_exp=_k(x))
    prow = p if orient in ("row", "both") else None
    pcol = p if orient in ("col", "both") else None
    got = gpu_quantize(x.to(DEV), prow, pcol, 1, 1)
    want = oracle_quantize(oracle_input(x), prow, pcol, 1, 1)
    assert_same(got, want, f"nvfp4 {orient} mma")


@pytest.mark.parametrize("rows", [1, 37, 100])
def test_nvfp4_row_only_any_row_count(rows):
    """Row-wise-only NVFP4 output takes any row count (the row kernel)."""
    cols = 96
    x = _input(rows, cols, "bf16", seed=40 + rows)
    for scale, rnd in itertools.product(SCALES, ROUNDS):
        p = oracle.Params(block=oracle.BLOCK_1X16, scale_mode=scale, rounding=rnd, wht=True,
                          wht_sign_mask=0xF0F0F0F0, seed=9, tensor_exp=_k(x))
        assert_same(gpu_quantize(x.to(DEV), p, None), oracle_quantize(oracle_input(x), p, None),
                    "nvfp4 rows")


@pytest.mark.parametrize("k", [0, 9, -12])
@pytest.mark.parametrize("scale", SCALES)
def test_nvfp4_scale_selection_every_bf16_block_max(k, scale):
    """Each 16-block's max is one positive finite bf16 value (all of them, with
    the other elements of the block at fractions of it): the E4M3 scale codes
    and the codes of the whole block, against the oracle, for both tile and row
    kernels."""
    u = np.arange(1, 0x7F80, dtype=np.uint32)
    nb = len(u)
    nb_pad = (nb + 5) // 6 * 6                      # 6 blocks per 96-element row
    m = np.zeros(nb_pad, dtype=np.uint32)
    m[:nb] = u
    rng = np.random.default_rng(100 + k)
    frac = rng.integers(0, 1 << 16, (nb_pad, 16)).astype(np.uint32)
    # element j of a block: M * (frac / 2^16) rounded to bf16, element 0 = +-M
    Mv = (m << 16).view(np.float32).astype(np.float64)
    vals = Mv[:, None] * frac / 65536.0
    vals[:, 0] = Mv * np.where(rng.integers(0, 2, nb_pad) == 1, -1.0, 1.0)
    x = synth.bf16_from_f64(vals.reshape(-1, 96))
    rows = x.shape[0]
    pad = (32 - rows % 32) % 32
    x = torch.cat([x, torch.zeros(pad, 96, dtype=torch.bfloat16)])
    p = oracle.Params(block=oracle.BLOCK_1X16, scale_mode=scale, tensor_exp=k)
    want = oracle_quantize(oracle_input(x), p, None)
    assert_same(gpu_quantize(x.to(DEV), p, None), want, "row kernel")
    assert_same(gpu_quantize(x.to(DEV), p, p)[:2], want[:2], "tile kernel")


def test_nvfp4_quantize_full_size_sampled():
    """The 70B layer's dY shape (16384 x 28672, Laplace with outliers), both
    orientations, round-up scales + SR + rotation as in the Wgrad recipe; the
    oracle checks sampled row bands of both outputs."""
    import gemm_pt_block_gb300 as mx

    rows, cols = 16384, 28672
    x = synth.dev_laplace(rows, cols, 1e-3, 8, DEV, outlier_frac=1e-3, outlier_mult=100.0)
    k = _k(x)
    p = oracle.Params(block=oracle.BLOCK_1X16, scale_mode=oracle.SCALE_ROUNDUP,
                      rounding=oracle.ROUND_SR, wht=True, wht_sign_mask=0x2468ACE1, seed=4,
                      sr_stream=1, tensor_exp=k)
    qr, sr_, qc, sc = mx.mxfp4_quantize(x, cuda_params(p, 1), cuda_params(p, 1))
    torch.cuda.synchronize()
    xs = oracle_input(x[:256].cpu())
    q, s = oracle.quantize_rows(xs, p)
    assert np.array_equal(qr[:256].cpu().numpy(), q)
    s_mma = sr_.cpu().numpy()
    for r in (0, 77, 255):
        for b in (0, 1, 7, cols // 16 - 1):
            assert s_mma[oracle.mma_scale_offset(r, b, rows, cols // 16)] == s[r, b]
    # Column-wise output: the oracle sees a column slice, whose source indices
    # differ from the full tensor's, so this check uses nearest rounding.
    c0 = cols - 128
    xc = oracle_input(x[:, c0:].cpu().contiguous())
    pr = oracle.Params(block=oracle.BLOCK_1X16, scale_mode=oracle.SCALE_ROUNDUP, wht=True,
                       wht_sign_mask=0x2468ACE1, tensor_exp=k)
    _, _, qc2, sc2 = mx.mxfp4_quantize(x, None, cuda_params(pr, 0))
    q2, s2 = oracle.quantize_cols(xc, pr)
    assert np.array_equal(qc2[c0:].cpu().numpy(), q2) and np.array_equal(sc2[c0:].cpu().numpy(), s2)


# ------------------------------------------------------------------ GEMM ----

def _nv_operands(rows, K, seed, lo=40, hi=70):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    s = rng.integers(lo, hi, (rows, K // 16), dtype=np.uint8)
    return q, s


def _dev(*arrays):
    return [torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in arrays]


def test_nvfp4_gemm_all_ones_exact():
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 256, 256
    q = np.full((M, K // 2), 0x22, np.uint8)                    # E2M1 1.0
    s = oracle.scales_to_mma(np.full((M, K // 16), 0x38, np.uint8))   # E4M3 1.0
    c = mx.nvfp4_gemm(*_dev(q, s), 3, *_dev(q, s), -5, M, N, K)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert torch.all(c == K * 2.0 ** -2)


def test_nvfp4_gemm_per_block_scales_exact():
    """Unit scales except one 16-block per row / column (checks each scale's
    slot and the scale-per-16 grouping); every partial sum is exact in fp32."""
    import gemm_pt_block_gb300 as mx

    M, N, K = 256, 512, 1024
    qa, _ = _nv_operands(M, K, 1)
    qb, _ = _nv_operands(N, K, 2)
    sa = np.full((M, K // 16), 0x38, np.uint8)
    sb = np.full((N, K // 16), 0x38, np.uint8)
    rng = np.random.default_rng(3)
    sa[np.arange(M), rng.integers(0, K // 16, M)] = 0x40      # 2.0
    sb[np.arange(N), rng.integers(0, K // 16, N)] = 0x34      # 0.75
    sam, sbm = oracle.scales_to_mma(sa), oracle.scales_to_mma(sb)
    c = mx.nvfp4_gemm(*_dev(qa, sam), 0, *_dev(qb, sbm), 1, M, N, K)
    torch.cuda.synchronize()
    ref, _ = oracle.gemm_ref_nv(qa, sam, 0, qb, sbm, 1, M, N, K)
    assert np.array_equal(c.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (256, 512, 768), (512, 768, 2304),
                                   (1024, 1280, 4096), (128, 128, 128), (128, 384, 384),
                                   (384, 640, 1152), (640, 384, 640)])
def test_nvfp4_gemm_random_within_tolerance(M, N, K):
    import gemm_pt_block_gb300 as mx

    qa, sa = _nv_operands(M, K, M + 1)
    qb, sb = _nv_operands(N, K, N + 2)
    sam, sbm = oracle.scales_to_mma(sa), oracle.scales_to_mma(sb)
    c = mx.nvfp4_gemm(*_dev(qa, sam), -7, *_dev(qb, sbm), 4, M, N, K)
    c16 = mx.nvfp4_gemm(*_dev(qa, sam), -7, *_dev(qb, sbm), 4, M, N, K, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    ref, absref = oracle.gemm_ref_nv(qa, sam, -7, qb, sbm, 4, M, N, K)
    gemm_tolerance_check(c.cpu().numpy(), ref, absref)
    gemm_tolerance_check_bf16(bf16_to_f64(c16), ref, absref)


def test_nvfp4_quantize_then_gemm_end_to_end():
    """X [512, 1024] t(4) and W [768, 1024] N(0, 0.02) quantized to NVFP4 with
    their own tensor factors (nearest scales, RTN), then Y = Xq Wq^T; operands
    against the oracle bit for bit, Y within tolerance, and close to X W^T."""
    import gemm_pt_block_gb300 as mx

    T, D, F = 512, 1024, 768
    x = synth.student_t(T, D, 4.0, 201)
    w = synth.normal(F, D, 0.02, 202)
    kx, kw = _k(x), _k(w)
    px = oracle.Params(block=oracle.BLOCK_1X16, tensor_exp=kx)
    pw = oracle.Params(block=oracle.BLOCK_1X16, tensor_exp=kw)
    qx, sx, _, _ = mx.mxfp4_quantize(x.to(DEV), cuda_params(px, 1))
    qw, sw, _, _ = mx.mxfp4_quantize(w.to(DEV), cuda_params(pw, 1))
    y = mx.nvfp4_gemm(qx, sx, kx, qw, sw, kw, T, F, D).cpu().numpy()
    rqx, rsx = oracle.quantize_rows(synth.bf16_bits(x), px)
    rqw, rsw = oracle.quantize_rows(synth.bf16_bits(w), pw)
    assert_same([qx.cpu().numpy(), sx.cpu().numpy(), qw.cpu().numpy(), sw.cpu().numpy()],
                [rqx, oracle.scales_to_mma(rsx), rqw, oracle.scales_to_mma(rsw)], "operands")
    ref, absref = oracle.gemm_ref_nv(rqx, oracle.scales_to_mma(rsx), kx, rqw,
                                     oracle.scales_to_mma(rsw), kw, T, F, D)
    gemm_tolerance_check(y, ref, absref)
    exact = x.double().numpy() @ w.double().numpy().T
    assert np.linalg.norm(y - exact) / np.linalg.norm(exact) < 0.15


@pytest.mark.parametrize("M,N,K", [(16384, 28672, 8192), (28672, 8192, 16384)])
def test_nvfp4_gemm_full_size_sampled(M, N, K):
    """70B-layer Fprop / Wgrad shapes in the benchmark's launch configuration;
    the oracle checks sampled outputs one by one."""
    import gemm_pt_block_gb300 as mx

    g = torch.Generator(device=DEV).manual_seed(M + N)
    qa = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    qb = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    sa = torch.randint(44, 64, (M * K // 16,), dtype=torch.uint8, device=DEV, generator=g)
    sb = torch.randint(44, 64, (N * K // 16,), dtype=torch.uint8, device=DEV, generator=g)
    c = mx.nvfp4_gemm(qa, sa, -2, qb, sb, 1, M, N, K)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    rows = np.array([0, 1, 127, 128, 255, M // 2 + 77, M - 1])
    ms = np.repeat(rows, 48)
    ns = np.tile(np.linspace(0, N - 1, 48).astype(np.int64), len(rows))
    ref, absref = oracle.gemm_pairs_nv(qa.cpu().numpy(), sa.cpu().numpy(), -2, qb.cpu().numpy(),
                                       sb.cpu().numpy(), 1, M, N, K, ms, ns)
    gemm_tolerance_check(c[torch.from_numpy(ms), torch.from_numpy(ns)].cpu().numpy(), ref, absref)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_nvfp4_mixed_with_other_block_types(dtype):
    """One orientation NVFP4, the other 1x32 / 32x32 / 64x64 MXFP4 (the general
    tile variant), both against the oracle."""
    rows, cols = 192, 320
    x = _input(rows, cols, dtype, seed=55)
    nv = oracle.Params(block=oracle.BLOCK_1X16, scale_mode=oracle.SCALE_FLOOR,
                       rounding=oracle.ROUND_SR, wht=True, wht_sign_mask=0x0F0F00FF, seed=3,
                       sr_stream=7, tensor_exp=_k(x))
    for blk in (oracle.BLOCK_1X32, oracle.BLOCK_32X32, oracle.BLOCK_64X64):
        mxp = oracle.Params(block=blk, scale_mode=oracle.SCALE_ROUNDUP, rounding=oracle.ROUND_SR,
                            seed=3, sr_stream=7)
        for prow, pcol in ((nv, mxp), (mxp, nv)):
            got = gpu_quantize(x.to(DEV), prow, pcol)
            want = oracle_quantize(oracle_input(x), prow, pcol)
            assert_same(got, want, f"mixed {blk}")


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8", "nvfp4"])
def test_dequantize_ex_every_format(fmt, layout):
    """GPU reconstruction of each format against the oracle's, bit for bit
    (every product is exact), over all code values and a spread of scales."""
    import gemm_pt_block_gb300 as mx

    rows, cols = 256, 384
    rng = np.random.default_rng(300 + layout)
    if fmt == "mxfp8":
        q = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] = 0x3F                      # no NaN codes
        s = rng.integers(100, 150, (rows, cols // 32), dtype=np.uint8)
        want = oracle.dequantize(q, s, rows, cols, f64=True, fmt=oracle.FORMAT_E4M3)
        p = mx.QuantParams(elem_format=mx.FORMAT_E4M3, scale_layout=layout)
    elif fmt == "nvfp4":
        q = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
        s = rng.integers(0, 127, (rows, cols // 16), dtype=np.uint8)
        want = oracle.dequantize_nv(q, s, rows, cols, tensor_exp=-9)
        p = mx.QuantParams(block=mx.BLOCK_1X16, tensor_exp=-9, scale_layout=layout)
    else:
        q = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
        s = rng.integers(90, 160, (rows, cols // 32), dtype=np.uint8)
        want = oracle.dequantize(q, s, rows, cols, f64=True)
        p = mx.QuantParams(scale_layout=layout)
    sd = oracle.scales_to_mma(s) if layout else s
    got = mx.mxfp4_dequantize(*_dev(q, sd), rows, cols, params=p)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().astype(np.float64), want)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (512, 768, 2304), (16384, 8192, 28672),
                                   (128, 384, 384), (384, 640, 1152)])
def test_nvfp4_gemm_scale_images_bit_identical(M, N, K):
    """nvfp4_gemm's workspace path (six 128x256b copies per K step instead of
    twelve) gives the same bits as without a workspace."""
    import gemm_pt_block_gb300 as mx

    g = torch.Generator(device=DEV).manual_seed(M + N + K)
    qa = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    qb = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=DEV, generator=g)
    sa = torch.randint(40, 70, (M * K // 16,), dtype=torch.uint8, device=DEV, generator=g)
    sb = torch.randint(40, 70, (N * K // 16,), dtype=torch.uint8, device=DEV, generator=g)
    plain = mx.nvfp4_gemm(qa, sa, -3, qb, sb, 2, M, N, K, workspace=False)
    img = mx.nvfp4_gemm(qa, sa, -3, qb, sb, 2, M, N, K)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert torch.equal(plain, img)
    if M <= 512:
        ref, absref = oracle.gemm_ref_nv(qa.cpu().numpy(), sa.cpu().numpy(), -3, qb.cpu().numpy(),
                                         sb.cpu().numpy(), 2, M, N, K)
        gemm_tolerance_check(img.cpu().numpy(), ref, absref)


def test_nvfp4_edge_cases():
    """Zeros (S = 0: signed-zero codes), a strided input, an empty tensor,
    tiny values under a large factor, and values that saturate the scale at 448."""
    import gemm_pt_block_gb300 as mx

    def both(x, p):
        got = gpu_quantize(x.to(DEV), p, p)
        want = oracle_quantize(oracle_input(x), p, p)
        assert_same(got, want, "nvfp4 edge")

    for mode in SCALES:
        z = torch.zeros(64, 96, dtype=torch.bfloat16)
        z[3, :16] = -0.0
        both(z, oracle.Params(block=oracle.BLOCK_1X16, scale_mode=mode))
        tiny = synth.normal(64, 96, 1e-30, 61).float()
        both(tiny, oracle.Params(block=oracle.BLOCK_1X16, scale_mode=mode, tensor_exp=40))
        big = synth.normal(64, 96, 1e4, 62).float()
        both(big, oracle.Params(block=oracle.BLOCK_1X16, scale_mode=mode, rounding=oracle.ROUND_SR,
                                seed=2, tensor_exp=-3))        # scales saturate at 448
    # strided input: a column slice of a wider tensor
    wide = _input(64, 160, "bf16", seed=63)
    view = wide.to(DEV)[:, 32:128]
    p = oracle.Params(block=oracle.BLOCK_1X16, scale_mode=oracle.SCALE_ROUNDUP, tensor_exp=_k(wide))
    got = gpu_quantize(view, p, p)
    want = oracle_quantize(oracle_input(wide[:, 32:128].contiguous()), p, p)
    assert_same(got, want, "nvfp4 strided")
    e = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    q, s, _, _ = mx.mxfp4_quantize(e, cuda_params(oracle.Params(block=oracle.BLOCK_1X16), 0))
    assert q.shape == (0, 32) and s.shape == (0, 4)


@pytest.mark.parametrize("rows_sr", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_nvfp4_dual_profiles(rows_sr, dtype):
    """NVFP4 dual calls with the activation / gradient recipes (rows without
    rotation, columns stochastic with rotation): the compile-time profiles."""
    x = _input(160, 352, dtype, seed=141)
    k = _k(x)
    prow = oracle.Params(block=oracle.BLOCK_1X16, scale_mode=oracle.SCALE_ROUNDUP,
                         rounding=oracle.ROUND_SR if rows_sr else oracle.ROUND_RTN, seed=12,
                         sr_stream=2, tensor_exp=k)
    pcol = oracle.Params(block=oracle.BLOCK_1X16, scale_mode=oracle.SCALE_ROUNDUP,
                         rounding=oracle.ROUND_SR, wht=True, wht_sign_mask=0x600DCAFE, seed=12,
                         sr_stream=2, tensor_exp=k)
    assert_same(gpu_quantize(x.to(DEV), prow, pcol), oracle_quantize(oracle_input(x), prow, pcol),
                "nvfp4 profile")
