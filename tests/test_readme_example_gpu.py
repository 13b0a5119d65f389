"""The Python example in README.md runs as written and its result matches the oracle."""
import os
import re

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_61_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    with open(os.path.join(ROOT, "README.md")) as f:
        text = f.read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert len(blocks) == 1, "README.md holds one Python example"
    env = {}
    exec(compile(blocks[0], "README.md", "exec"), env)
    torch.cuda.synchronize()

    def bits(t):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)

    k, v, q = bits(env["k"]), bits(env["v"]), bits(env["q"])
    tables, lens = env["tables"].cpu().numpy(), env["lens"].cpu().numpy()
    rows = [(b, h) for b in (0, 31, 63) for h in (0, 5, 31)]
    ref_out, ref_lse = oracle.paged_decode(q, k, v, tables, lens, env["D"] ** -0.5, env["P"],
                                           synth.FP16, rows=rows)
    out = env["out"].float().cpu().numpy()
    lse = env["lse"].cpu().numpy()
    for b, h in rows:
        assert np.abs(out[b, h] - ref_out[b, h]).max() <= 2e-3
        assert abs(lse[b, h] - ref_lse[b, h]) <= 1e-3
