"""The README's quick start runs as written on the GPU (so the documented
calls and argument names stay those of the binding), and its results are
finite."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_quick_start_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    scope = {}
    exec(compile(code, "README.md", "exec"), scope)
    torch.cuda.synchronize()
    for name in ("out", "o1", "state", "caps"):
        assert torch.isfinite(scope[name]).all(), name
    assert scope["out"].shape == (318, 48, 128) and scope["caps"].shape[:2] == (3, 4)
