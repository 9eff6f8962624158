"""GPU parity of the bfloat16 path (q, both caches and out in bfloat16;
products on bfloat16 tensor-core operands) against the fp64 oracle on the same
bfloat16 inputs.

Tolerance, derived from the arithmetic rather than the fp16 figure: the
kernel rounds each softmax weight p_j to bfloat16 before P.V (relative error
<= 2^-8) and rounds the output to bfloat16 (<= 2^-8 |out|); everything else is
fp32 (scores, online softmax, accumulation). So for every element

    |gpu - ref| <= 2^-8 (|ref| + sum_j w_j |v_j| / sum_j w_j) + 1e-4,

where the middle term is the oracle run on |V| (the sign bits of the bfloat16
V cache cleared) and 1e-4 covers the fp32 parts. Rows with no visible key
must be exact zeros.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from paged_split_decode_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def pd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_split_decode_gb300 as pd
    pd.load()
    return pd


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def oracle_pair(w):
    """(ref, ref over |V|) from the oracle on the bfloat16 bit patterns."""
    args = (w.scale, w.window, w.qlen)
    q, k, v = bits(w.q), bits(w.k_cache), bits(w.v_cache)
    bt, sl = w.block_table.numpy(), w.seq_lens.numpy()
    ref = oracle.decode_paged(q, k, v, bt, sl, *args, bf16=True)
    vabs = v & np.uint16(0x7FFF)
    ref_abs = oracle.decode_paged(q, k, vabs, bt, sl, *args, bf16=True)
    return ref, ref_abs


def check(w, got, ref, ref_abs):
    g = got.float().cpu().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{w.name}: non-finite output"
    bound = 2.0 ** -8 * (np.abs(ref) + ref_abs) + 1e-4
    excess = np.abs(g - ref) / bound
    assert excess.max() <= 1.0, f"{w.name}: error {excess.max():.2f}x the bound"
    empty = np.all(ref == 0.0, axis=-1)
    assert np.all(g[empty] == 0.0), f"{w.name}: empty rows not zero"
    return float(excess.max())


def run(pd, w, S, out=None, flag=None):
    res = pd.decode_paged(w.q.to(DEV), w.k_cache.to(DEV), w.v_cache.to(DEV), w.block_table.to(DEV),
                          w.seq_lens.to(DEV), w.scale, w.window, w.qlen, S, out=out,
                          error_flag=flag)
    torch.cuda.synchronize()
    return res


CASES = [
    ("tiny_d128", dict(B=2, Hq=8, Hkv=2, D=128, seq_lens=[100, 0], pool_blocks=16,
                       max_blocks_per_seq=8)),
    ("gqa6_d256_head_groups", dict(B=3, Hq=24, Hkv=4, D=256, seq_lens=[4096, 1000, 17])),
    ("gqa4_d128_head_groups_ragged", dict(B=6, Hq=32, Hkv=8, D=128,
                                          seq_lens=[512, 3000, 1, 7000, 0, 1500])),
    ("gqa6_d256_per_head", dict(B=2, Hq=12, Hkv=2, D=256, seq_lens=[2500, 300])),
    ("verify_q3_window", dict(B=3, Hq=24, Hkv=4, D=256, qlen=3, window=700,
                              seq_lens=[2, 2000, 800])),
    ("rows_32_d128", dict(B=2, Hq=16, Hkv=2, D=128, qlen=4, seq_lens=[900, 33])),
    ("stale_nan_tails", dict(B=3, Hq=24, Hkv=4, D=256, seq_lens=[17, 1001, 250], stale="nan")),
    # two long sequences on a large table: many pieces per unit
    ("two_long_sequences", dict(B=2, Hq=24, Hkv=4, D=256, seq_lens=[9000, 9000], max_blocks_per_seq=1024)),
]


@pytest.mark.parametrize("S", [0, 1, 5, 12])
@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_bf16_matches_oracle(pd, name, kw, S):
    w = inputs.make_workload(kv="bf16", seed=zlib.crc32(name.encode()) % 10000, name=name, **kw)
    ref, ref_abs = oracle_pair(w)
    check(w, run(pd, w, S), ref, ref_abs)


def test_bf16_output_type_and_untouched_padding(pd):
    w = inputs.make_workload(kv="bf16", B=2, Hq=8, Hkv=2, D=128, seq_lens=[300, 5], seed=3)
    out = torch.full(w.q.shape, 3.0, dtype=torch.bfloat16, device=DEV)
    got = run(pd, w, 0, out=out)
    assert got.dtype == torch.bfloat16 and got.data_ptr() == out.data_ptr()
    ref, ref_abs = oracle_pair(w)
    check(w, got, ref, ref_abs)


def test_bf16_rejects_fp16_query(pd):
    w = inputs.make_workload(kv="bf16", B=1, Hq=8, Hkv=2, D=128, seq_lens=[64], seed=4)
    with pytest.raises(TypeError):
        pd.decode_paged(w.q.to(torch.float16).to(DEV), w.k_cache.to(DEV), w.v_cache.to(DEV),
                        w.block_table.to(DEV), w.seq_lens.to(DEV), w.scale)


def test_bf16_variable_query_count(pd):
    w = inputs.make_varlen_workload(qlens=[1, 3, 0, 2], kv="bf16", B=4, Hq=24, Hkv=4, D=256,
                                    seq_lens=[3000, 400, 90, 1200], seed=9)
    out = pd.decode_paged_varlen(w.q.to(DEV), w.k_cache.to(DEV), w.v_cache.to(DEV),
                                 w.block_table.to(DEV), w.seq_lens.to(DEV), w.q_start.to(DEV),
                                 w.qlen, w.scale)
    torch.cuda.synchronize()
    q, k, v = bits(w.q), bits(w.k_cache), bits(w.v_cache)
    args = (w.block_table.numpy(), w.seq_lens.numpy(), w.q_start.numpy(), w.scale)
    ref = oracle.decode_paged_varlen(q, k, v, *args, bf16=True)
    ref_abs = oracle.decode_paged_varlen(q, k, v & np.uint16(0x7FFF), *args, bf16=True)
    check(w, out, ref, ref_abs)


def test_bf16_writer_then_decode(pd):
    """bfloat16 tokens through the writer (bit copy, byte-compared with the
    oracle's writer), then decoded."""
    Hq, Hkv, D, bs, L = 8, 2, 128, 16, 77
    nb = 12
    g = torch.Generator().manual_seed(21)
    k_tok = torch.randn((L, Hkv, D), generator=g).to(torch.bfloat16)
    v_tok = torch.randn((L, Hkv, D), generator=g).to(torch.bfloat16)
    table = torch.randperm(nb, generator=g)[:5].to(torch.int32)
    slots = torch.tensor([int(table[j // bs]) * bs + j % bs for j in range(L)], dtype=torch.int64)
    kc = torch.zeros((nb, bs, Hkv, D), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    pd.write_kv_cache(k_tok.to(DEV), v_tok.to(DEV), slots.to(DEV), kc, vc)
    torch.cuda.synchronize()
    ko = np.zeros((nb, bs, Hkv, D), dtype=np.uint16)
    vo = np.zeros_like(ko)
    oracle.write_kv_cache(bits(k_tok), bits(v_tok), slots.numpy(), ko, vo, bf16=True)
    assert np.array_equal(bits(kc.cpu()), ko) and np.array_equal(bits(vc.cpu()), vo)
    q = torch.randn((1, Hq, D), generator=g).to(torch.bfloat16)
    sl = torch.tensor([L], dtype=torch.int32)
    out = pd.decode_paged(q.to(DEV), kc, vc, table[None].to(DEV), sl.to(DEV), 0.1)
    torch.cuda.synchronize()
    ref = oracle.decode_paged(bits(q), ko, vo, table[None].numpy(), sl.numpy(), 0.1, bf16=True)
    ref_abs = oracle.decode_paged(bits(q), ko, vo & np.uint16(0x7FFF), table[None].numpy(),
                                  sl.numpy(), 0.1, bf16=True)
    w = inputs.Workload(name="bf16_writer", q=q, k_cache=kc, v_cache=vc, block_table=table[None],
                        seq_lens=sl, scale=0.1)
    check(w, out, ref, ref_abs)
