"""Calls from several host threads at once, each on its own CUDA stream (the
ABI's calls are thread-safe and re-entrant across streams): every thread's
quantized operands and GEMM result equal the same work run serially, bit for
bit. The check runs in a fresh process so that the concurrent calls are its
first ones and the per-device caches (kernel attributes, occupancy, the TMA
encoder) are filled under contention."""
from __future__ import annotations

import os
import subprocess
import sys
import threading

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _work(mx, torch, x, w, r, stream):
    with torch.cuda.stream(stream):
        xq, xs, xqc, xsc = mx.mxfp4_quantize(x, r.x_row, r.x_col)
        wq, ws, _, _ = mx.mxfp4_quantize(w, r.w_row, None)
        c = mx.mxfp4_gemm(xq, xs, wq, ws, x.shape[0], w.shape[0], x.shape[1])
        return [xq, xs, xqc, xsc, wq, ws, c]


def main() -> int:
    import torch

    import gemm_pt_block_gb300 as mx
    import synth

    n = 4
    T, D, F = 512, 1024, 768
    dev = torch.device("cuda")
    jobs = []
    for i in range(n):
        r = mx.recipe_2d_sr(synth.sign_mask(200 + i), seed=i)
        x = synth.student_t(T, D, 4.0, 6000 + i).to(dev)
        w = synth.normal(F, D, 0.02, 6100 + i).to(dev)
        jobs.append((x, w, r))
    torch.cuda.synchronize()

    results, errors = [None] * n, []
    start = threading.Barrier(n)

    def run(i):
        try:
            s = torch.cuda.Stream()
            start.wait()
            out = _work(mx, torch, *jobs[i], s)
            s.synchronize()
            results[i] = [t.clone() for t in out]
        except Exception as e:  # reported below
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=run, args=(i,)) for i in range(n)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    if errors:
        print("\n".join(errors))
        return 1
    for i in range(n):
        serial = _work(mx, torch, *jobs[i], torch.cuda.current_stream())
        torch.cuda.synchronize()
        for k, (a, b) in enumerate(zip(results[i], serial)):
            if not torch.equal(a, b):
                print(f"thread {i}, output {k} differs from the serial run")
                return 1
    print("OK")
    return 0


@pytest.mark.gpu
def test_concurrent_threads_match_serial():
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([ROOT, os.environ.get("PYTHONPATH", "")]))
    r = subprocess.run([sys.executable, os.path.abspath(__file__)], capture_output=True, text=True,
                       timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0 and "OK" in r.stdout, r.stdout + r.stderr


if __name__ == "__main__":
    sys.exit(main())
