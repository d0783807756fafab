"""The usage examples in README.md run as written (in order, one namespace)."""
import os
import re

import pytest

pytestmark = pytest.mark.gpu

README = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")


def test_readme_examples_run():
    import torch
    blocks = re.findall(r"```python\n(.*?)```", open(README).read(), re.S)
    assert len(blocks) >= 2
    ns = {}
    for code in blocks:
        exec(compile(code, "README.md", "exec"), ns)
    torch.cuda.synchronize()
    assert ns["err"].item() == 0
    assert torch.isfinite(ns["out"].float()).all() and torch.isfinite(ns["outd"].float()).all()
    assert torch.isfinite(ns["out_dec"].float()).all()
    assert torch.isfinite(ns["out_pre"].float()).all()
    assert tuple(ns["y"].shape) == (8, 4096) and torch.isfinite(ns["y"].float()).all()
