"""The usage example in README.md runs as written and gives finite outputs."""

import os
import re

import pytest
import torch

from libbuild import ROOT, ensure_built

pytestmark = pytest.mark.gpu


def test_readme_example_runs():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    text = open(os.path.join(ROOT, "README.md")).read()
    code = re.search(r"```python\n(.*?)```", text, flags=re.S).group(1)
    env = {}
    exec(compile(code, "README.md", "exec"), env)
    torch.cuda.synchronize()
    out = env["out"][0]
    assert out.shape == (1, 32, 128) and torch.isfinite(out.float()).all()
    env["cache"].check()
