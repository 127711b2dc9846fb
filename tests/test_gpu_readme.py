"""The usage example (paged_kv_cache_317_gb300/examples/readme_example.py, shown in
the README) runs as written and its output is finite."""

import os
import runpy

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EXAMPLE = os.path.join(ROOT, "paged_kv_cache_317_gb300", "examples", "readme_example.py")


def test_readme_example_runs(lib):
    env = runpy.run_path(EXAMPLE, run_name="readme_example")
    out = env["out"]
    torch.cuda.synchronize()
    assert out.shape == (2, 8, 128) and torch.isfinite(out).all()
    assert list(env["lens"]) == [101, 101]
