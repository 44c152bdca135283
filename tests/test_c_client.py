"""The C ABI from C: `tests/c_client/mxfp4_client.c` links libmxfp4.so and the
CUDA runtime, with no Python or PyTorch in the loop. It compiles on any host;
on a GPU its quantized operands match the oracle bit for bit, its Fprop GEMM
is within the fp64 bound and equals the Python binding's result bit for bit."""
from __future__ import annotations

import os
import subprocess

import numpy as np
import pytest

import oracle
import synth
from _util import gemm_tolerance_check

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "mxfp4_client.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_client(out_dir: str) -> str:
    from gemm_pt_block_gb300 import build as b

    lib = b.build()
    libdir = os.path.dirname(lib)
    cudalib = os.path.join(CUDA, "lib64")
    exe = os.path.join(out_dir, "mxfp4_client")
    cmd = [os.environ.get("CC", "gcc"), "-std=c99", "-O2", "-Wall", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"), SRC,
           "-o", exe, "-L", libdir, "-lmxfp4", "-L", cudalib, "-lcudart",
           f"-Wl,-rpath,{libdir}:{cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    exe = build_client(str(tmp_path))
    assert os.access(exe, os.X_OK)


CASES = [
    # block, scale_mode, rounding, wht, sign-mask seed, SR seed
    (oracle.BLOCK_1X32, oracle.SCALE_FLOOR, oracle.ROUND_RTN, 0, None, 0),
    (oracle.BLOCK_32X32, oracle.SCALE_ROUNDUP, oracle.ROUND_SR, 1, 61, 7),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES)
def test_c_client_matches_oracle_and_binding(tmp_path, case):
    import torch

    import gemm_pt_block_gb300 as mx

    block, scale_mode, rounding, wht, mask_seed, seed = case
    mask = synth.sign_mask(mask_seed) if mask_seed is not None else 0
    T, D, F = 256, 512, 256
    x = synth.student_t(T, D, 4.0, 5100)
    w = synth.normal(F, D, 0.02, 5101)
    xb, wb = synth.bf16_bits(x), synth.bf16_bits(w)
    xb.tofile(str(tmp_path / "x.bin"))
    wb.tofile(str(tmp_path / "w.bin"))
    exe = build_client(str(tmp_path))
    prefix = str(tmp_path / "out")
    r = subprocess.run([exe, str(T), str(D), str(F), str(tmp_path / "x.bin"),
                        str(tmp_path / "w.bin"), prefix, str(block), str(scale_mode),
                        str(rounding), str(wht), str(mask), str(seed)],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    qx = np.fromfile(prefix + ".qx", dtype=np.uint8).reshape(T, D // 2)
    sx = np.fromfile(prefix + ".sx", dtype=np.uint8)
    qw = np.fromfile(prefix + ".qw", dtype=np.uint8).reshape(F, D // 2)
    sw = np.fromfile(prefix + ".sw", dtype=np.uint8)
    c = np.fromfile(prefix + ".c", dtype=np.float32).reshape(T, F)

    base = dict(block=block, scale_mode=scale_mode, rounding=rounding, wht=bool(wht),
                wht_sign_mask=mask, seed=seed)
    for q, s, src, stream in ((qx, sx, xb, 0), (qw, sw, wb, 1)):
        oq, os_ = oracle.quantize_rows(src, oracle.Params(**base, sr_stream=stream))
        assert np.array_equal(q, oq)
        assert np.array_equal(s, oracle.scales_to_mma(os_))

    ref, absref = oracle.gemm_ref(qx, sx, qw, sw, T, F, D)
    gemm_tolerance_check(c, ref, absref)

    dev = torch.device("cuda")
    cb = mx.mxfp4_gemm(torch.from_numpy(qx).to(dev), torch.from_numpy(sx).to(dev),
                       torch.from_numpy(qw).to(dev), torch.from_numpy(sw).to(dev), T, F, D)
    torch.cuda.synchronize()
    assert np.array_equal(cb.cpu().numpy().view(np.uint32), c.view(np.uint32))
