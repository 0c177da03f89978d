"""The usage example of the README runs as written (GPU)."""
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_readme_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert len(blocks) == 1
    scope = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)
    torch.cuda.synchronize()
    y, y1 = scope["y"], scope["y1"]
    assert y.shape == (2048, 4096) and y1.shape == (1, 4096)
    assert torch.isfinite(y.float()).all() and torch.isfinite(y1.float()).all()
    # the prefill wrote the 2048 positions of blocks 0-15 and the decode step position 2048
    k_pool = scope["k_pool"]
    assert bool((k_pool[:16].float().abs().sum(dim=(1, 2, 3)) > 0).all())
    assert float(k_pool[16, :, 0].float().abs().sum()) > 0
    assert float(k_pool[16, :, 1:].float().abs().sum()) == 0
