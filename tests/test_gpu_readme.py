"""The usage example in README.md runs as written and gives the merge and
sort results the oracle gives."""
import os
import re

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example(gpu):
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "README has no python example"
    ns = {}
    exec(compile(blocks[0], "README.md", "exec"), ns)
    torch.cuda.synchronize()
    assert gpu.device_error() == 0
    A, B, C = (ns[k].cpu().numpy() for k in ("A", "B", "C"))
    assert np.array_equal(C, oracle.merge_i32(A, B))
    assert ns["i"] == oracle.corank_count(12345, A, B)
    split = ns["split"].cpu().numpy()
    assert split.size == (A.size + B.size + 4095) // 4096 + 1
    for t in [0, 1, 2, split.size // 2, split.size - 1]:
        assert split[t] == oracle.corank_pages(min(t * 4096, A.size + B.size), A, B)
    X, Y, Z = (ns[k].cpu().numpy() for k in ("X", "Y", "Z"))
    assert np.array_equal(Z.view(np.uint64), oracle.merge_keys(X, Y, descending=True).view(np.uint64))
    keys, vals = ns["keys"].cpu().numpy().view(np.uint32), ns["vals"].cpu().numpy().view(np.uint32)
    assert np.all(keys[1:] >= keys[:-1])
    assert np.array_equal(np.sort(vals), np.arange(vals.size, dtype=np.uint32))
