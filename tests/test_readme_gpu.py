"""The Python example of the package's documentation, as a user would write
it: 32 sequences of the D=256 GQA 6:1 shape through one decode_paged call,
checked against the fp64 oracle (two of the sequences, every head)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
TOL = 2e-3


def test_usage_example_matches_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_split_decode_gb300 as pd

    torch.manual_seed(20)
    B, Hq, Hkv, D, bs = 32, 24, 4, 256, 16
    num_blocks, max_blocks = 8192, 256
    q = torch.randn(B, Hq, D, device="cuda").half()                 # [B*qlen, Hq, D]
    k_cache = torch.randn(num_blocks, bs, Hkv, D, device="cuda").half()
    v_cache = torch.randn_like(k_cache)
    block_table = torch.randperm(num_blocks, device="cuda")[:B * max_blocks].view(B, max_blocks).int()
    seq_lens = torch.full((B,), 4096, dtype=torch.int32, device="cuda")  # includes the qlen new tokens
    out = pd.decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale=D ** -0.5,
                          window=0, qlen=1, num_splits=0)            # 0 = automatic split
    torch.cuda.synchronize()

    qn, kn, vn = q.cpu().numpy(), k_cache.cpu().numpy(), v_cache.cpu().numpy()
    bt, sl = block_table.cpu().numpy(), seq_lens.cpu().numpy()
    for b in (0, 31):
        ref = oracle.decode_paged(qn[b:b + 1], kn, vn, bt[b:b + 1], sl[b:b + 1], D ** -0.5)
        got = out[b:b + 1].float().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - ref))) <= TOL
