"""The README's Python example runs as written and its output matches the
fp64 oracle (two of its 32 sequences, every head)."""
import pathlib
import re

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
TOL = 2e-3


def test_readme_example_matches_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    text = (pathlib.Path(__file__).resolve().parents[1] / "README.md").read_text()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    torch.manual_seed(20)
    ns = {}
    exec(compile(code, "README.md", "exec"), ns)
    torch.cuda.synchronize()
    q, k, v = ns["q"].cpu().numpy(), ns["k_cache"].cpu().numpy(), ns["v_cache"].cpu().numpy()
    bt, sl, out = ns["block_table"].cpu().numpy(), ns["seq_lens"].cpu().numpy(), ns["out"]
    for b in (0, 31):
        ref = oracle.decode_paged(q[b:b + 1], k, v, bt[b:b + 1], sl[b:b + 1], ns["D"] ** -0.5)
        got = out[b:b + 1].float().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - ref))) <= TOL
