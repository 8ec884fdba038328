"""The usage example in README.md runs as written (sparse decode, paged decode
with a head sink, quantize-on-write, the staged prefill) and gives finite
outputs."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_runs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    with open(os.path.join(ROOT, "README.md")) as f:
        code = re.search(r"```python\n(.*?)```", f.read(), re.S).group(1)
    ns = {}
    exec(compile(code, "README.md", "exec"), ns)
    torch.cuda.synchronize()
    assert ns["out"].shape == (16, 32, 128)
    assert bool(torch.isfinite(ns["out"].float()).all())
    assert ns["out_p"].shape == (2048, 24, 256)
    assert bool(torch.isfinite(ns["out_p"].float()).all())
