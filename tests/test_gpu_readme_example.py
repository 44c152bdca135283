"""The Python usage example in README.md runs as written (on a GB300)."""
from __future__ import annotations

import os
import re

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs():
    import torch

    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "README.md has no python example"
    env: dict = {}
    exec(compile(blocks[0], "README.md example", "exec"), env)
    torch.cuda.synchronize()
    y, layer = env["y"], env["layer"]
    assert y.shape == (4096, 14336) and torch.isfinite(y).all()
    assert layer.weight.grad is not None and torch.isfinite(layer.weight.grad.float()).all()
