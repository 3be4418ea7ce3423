"""The usage example in README.md runs as written and gives finite results."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs():
    assert torch.cuda.is_available()
    text = open(os.path.join(ROOT, "README.md")).read()
    block = re.search(r"```python\n(.*?)```", text, flags=re.S).group(1)
    env = {}
    exec(compile(block, "README.md", "exec"), env)
    torch.cuda.synchronize()
    F, R = env["F"], env["R"]
    assert env["o"].shape == (F, 16, 128) and env["o_raw"].shape == (R, 16, 128)
    for name in ("o", "lse", "do", "dq", "dk", "dv", "o_p", "o_lo", "pq", "pk", "pv", "go", "dy", "gdg", "gdb", "dx",
                 "dcw"):
        assert torch.isfinite(env[name].float()).all(), name
    assert env["tok"].shape == (F,)
