"""Pins for the oracle's variable-query-count decode (decode_paged_varlen):

* equal counts reproduce the uniform decode bit for bit;
* tiny mixed batches match the dense numpy brute force (tests/ref_dense.py,
  written apart from the oracle) for fp16, fp8 and int8 KV, with and
  without a window, including sequences shorter than their query count;
* a sequence with no query token writes nothing and changes nothing else.
"""
import numpy as np
import pytest

import ref_dense
from paged_split_decode_gb300 import inputs


def run_varlen(oracle, w):
    return oracle.decode_paged_varlen(w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(),
                                      w.block_table.numpy(), w.seq_lens.numpy(), w.q_start.numpy(),
                                      w.scale, window=w.window, k_scale=w.k_scale,
                                      v_scale=w.v_scale, kv_fp8=w.kv_fp8, kv_int8=w.kv_int8)


def run_dense(w):
    return ref_dense.attention(w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(),
                               w.block_table.numpy(), w.seq_lens.numpy(), w.scale, w.window,
                               1, w.kv_fp8, w.k_scale, w.v_scale, w.kv_int8,
                               q_start=w.q_start.numpy())


def test_equal_counts_match_uniform_decode(oracle_lib):
    w = inputs.make_workload(B=3, Hq=8, Hkv=2, D=64, qlen=3, seq_lens=[40, 2, 100], seed=4,
                             window=30)
    uni = oracle_lib.decode_paged(w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(),
                                  w.block_table.numpy(), w.seq_lens.numpy(), w.scale, w.window, 3)
    qs = np.arange(0, 10, 3, dtype=np.int32)
    var = oracle_lib.decode_paged_varlen(w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(),
                                         w.block_table.numpy(), w.seq_lens.numpy(), qs, w.scale,
                                         window=w.window)
    assert np.array_equal(uni, var)


CASES = [
    dict(qlens=[1, 4, 2, 0, 3], seq_lens=[30, 45, 1, 17, 3], kv="f16"),
    dict(qlens=[2, 1, 5], seq_lens=[100, 0, 64], kv="fp8", window=20),
    dict(qlens=[3, 3, 1, 2], seq_lens=[2, 90, 33, 16], kv="int8", window=7),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_varlen_matches_dense_bruteforce(oracle_lib, ci):
    c = dict(CASES[ci])
    qlens = c.pop("qlens")
    B = len(qlens)
    w = inputs.make_varlen_workload(qlens=qlens, B=B, Hq=6, Hkv=2, D=32, seed=10 + ci, **c)
    got = run_varlen(oracle_lib, w)
    want = run_dense(w)
    assert np.allclose(got, want, rtol=0, atol=1e-12)


def test_zero_query_sequence_writes_nothing(oracle_lib):
    w = inputs.make_varlen_workload(qlens=[2, 0, 3], B=3, Hq=4, Hkv=2, D=32, seq_lens=[50, 70, 20],
                                    seed=3)
    got = run_varlen(oracle_lib, w)
    # the same batch without sequence 1: identical rows
    keep = [0, 2]
    w2 = inputs.make_varlen_workload(qlens=[2, 3], B=2, Hq=4, Hkv=2, D=32, seq_lens=[50, 20],
                                     seed=3)
    w2.q = w.q
    w2.q_start = w.q_start[[0, 1, 3]].contiguous()
    w2.k_cache, w2.v_cache = w.k_cache, w.v_cache
    w2.block_table = w.block_table[keep].contiguous()
    w2.scale = w.scale
    assert np.array_equal(run_varlen(oracle_lib, w2), got)
    assert got.shape[0] == 5
