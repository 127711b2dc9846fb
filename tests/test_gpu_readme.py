"""The usage example in README.md runs as written and its output is finite."""

import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_runs(lib):
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "README.md has no python example"
    env = {}
    exec(compile(blocks[0], "README.md example", "exec"), env)
    out = env["out"]
    torch.cuda.synchronize()
    assert out.shape == (2, 8, 128) and torch.isfinite(out).all()
    lens = env["lens"]
    assert list(lens) == [101, 101]
