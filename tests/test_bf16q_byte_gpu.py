"""GPU parity of e4m3fn and int8 caches under a bfloat16 q and out
(PD_KV_FP8_E4M3_BF16, PD_KV_INT8_BF16) against the fp64 oracle on the same
inputs: the bfloat16 q bits, the cache codes and their scales.

Tolerance: the kernels compute as for an fp16 q -- each q row is scaled by a
power of two into fp16, exactly -- so the byte kinds' 2e-3 holds for the
result before the output is rounded to bfloat16 (<= 2^-9 |out|, taken as
2^-8):

    |gpu - ref| <= 2^-8 |ref| + 2e-3.

Rows with no visible key must be exact zeros. The q rows scaled by 2^30 or
2^-30 (with the scale compensating) lie outside fp16's range and pass only
through the per-row scaling. The writer takes bfloat16 new tokens for these
caches and must store the oracle's codes byte for byte.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from paged_split_decode_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KINDS = ["fp8_bf16q", "int8_bf16q"]


@pytest.fixture(scope="module")
def pd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_split_decode_gb300 as pd
    pd.load()
    return pd


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def ref_run(w):
    return oracle.decode_paged(bits(w.q), w.k_cache.numpy(), w.v_cache.numpy(), w.block_table.numpy(),
                               w.seq_lens.numpy(), w.scale, w.window, w.qlen, w.k_scale, w.v_scale,
                               w.kv_fp8, kv_int8=w.kv_int8, bf16=True)


def gpu_run(pd, w, S):
    k, v = w.k_cache.to(DEV), w.v_cache.to(DEV)
    if w.kv_int8:
        k, v = k.view(torch.int8), v.view(torch.int8)
    out = pd.decode_paged(w.q.to(DEV), k, v, w.block_table.to(DEV), w.seq_lens.to(DEV), w.scale, w.window,
                          w.qlen, S, k_scale=w.k_scale, v_scale=w.v_scale)
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16
    return out


def check(w, got, ref):
    g = got.float().cpu().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{w.name}: non-finite output"
    bound = 2.0 ** -8 * np.abs(ref) + 2e-3
    excess = np.abs(g - ref) / bound
    assert excess.max() <= 1.0, f"{w.name}: error {excess.max():.2f}x the bound"
    empty = np.all(ref == 0.0, axis=-1)
    assert np.all(g[empty] == 0.0), f"{w.name}: empty rows not zero"


CASES = [
    ("gqa6_d256_head_groups", dict(B=3, Hq=24, Hkv=4, D=256, seq_lens=[4096, 1000, 17])),
    ("gqa6_d128_per_head_kg2", dict(B=3, Hq=12, Hkv=2, D=128, seq_lens=[2500, 300, 1])),
    # four heads per tile with D split over two warps: each warp loads its q
    # rows whole for the row exponents
    ("gqa4_d128_head_groups_dsplit", dict(B=3, Hq=16, Hkv=4, D=128, seq_lens=[3000, 200, 1])),
    ("rows_12_d256", dict(B=3, Hq=12, Hkv=2, D=256, qlen=2, seq_lens=[5, 1000, 64])),
    ("verify_q3_d256", dict(B=3, Hq=24, Hkv=4, D=256, qlen=3, seq_lens=[2, 2000, 800])),
    ("rows_32_window_d128", dict(B=2, Hq=16, Hkv=2, D=128, qlen=4, window=300, seq_lens=[1500, 40])),
    ("verify_q3_d128_empty", dict(B=3, Hq=24, Hkv=4, D=128, qlen=3, seq_lens=[0, 700, 1])),
]


@pytest.mark.parametrize("S", [0, 1, 3])
@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("kv", KINDS)
def test_byte_caches_under_bf16_q_match_oracle(pd, kv, name, kw, S):
    w = inputs.make_workload(kv=kv, seed=zlib.crc32((kv + name).encode()) % 10000, name=name, **kw)
    check(w, gpu_run(pd, w, S), ref_run(w))


@pytest.mark.parametrize("shift", [30, -30])
@pytest.mark.parametrize("qlen", [1, 3])
@pytest.mark.parametrize("kv", KINDS)
def test_q_beyond_fp16_range(pd, kv, qlen, shift):
    """q * 2^shift with the scale * 2^-shift: the scores are unchanged, the q
    values lie outside fp16's range (or below its subnormals)."""
    w = inputs.make_workload(B=2, Hq=24, Hkv=4, D=256, qlen=qlen, seq_lens=[900, 33], kv=kv,
                             seed=77 + qlen, name=f"q_shift_{shift}")
    w.q = (w.q.to(torch.float64) * 2.0 ** shift).to(torch.bfloat16)
    w.scale = w.scale * 2.0 ** -shift
    check(w, gpu_run(pd, w, 0), ref_run(w))


@pytest.mark.parametrize("kind", ["fp8", "int8"])
def test_writer_takes_bf16_tokens(pd, kind):
    T, Hkv, D, nb, bs = 300, 4, 256, 40, 16
    g = torch.Generator().manual_seed(5)
    k_new = (torch.randn((T, Hkv, D), generator=g) * 2).to(torch.bfloat16)
    v_new = (torch.randn((T, Hkv, D), generator=g) * 3).to(torch.bfloat16)
    slots = torch.randperm(nb * bs, generator=g)[:T].to(torch.int64)
    slots[::9] = -1
    ks, vs = 1.0 / 40, 1.0 / 30
    kc = torch.full((nb, bs, Hkv, D), 0x5A, dtype=torch.uint8)
    kd, vd = kc.to(DEV), kc.to(DEV)
    if kind == "int8":
        kd, vd = kd.view(torch.int8), vd.view(torch.int8)
    pd.write_kv_cache(k_new.to(DEV), v_new.to(DEV), slots.to(DEV), kd, vd, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    ko, vo = kc.numpy().copy(), kc.numpy().copy()
    assert oracle.write_kv_cache(bits(k_new), bits(v_new), slots.numpy(), ko, vo, k_scale=ks, v_scale=vs,
                                 kv_fp8=kind == "fp8", kv_int8=kind == "int8", bf16=True)
    assert np.array_equal(kd.view(torch.uint8).cpu().numpy(), ko)
    assert np.array_equal(vd.view(torch.uint8).cpu().numpy(), vo)


@pytest.mark.parametrize("kv", KINDS)
def test_varlen_under_bf16_q_matches_oracle(pd, kv):
    """A query count per sequence (decode_paged_varlen) over byte caches with
    a bfloat16 q: rows outside every sequence's range are left as they were."""
    qlens = [1, 3, 0, 2, 4, 1]
    w = inputs.make_varlen_workload(qlens=qlens, B=len(qlens), Hq=16, Hkv=4, D=256, kv=kv,
                                    seq_lens=[500, 2000, 7, 1, 900, 0], seed=31)
    k, v = w.k_cache.to(DEV), w.v_cache.to(DEV)
    if w.kv_int8:
        k, v = k.view(torch.int8), v.view(torch.int8)
    got = pd.decode_paged_varlen(w.q.to(DEV), k, v, w.block_table.to(DEV), w.seq_lens.to(DEV),
                                 w.q_start.to(DEV), w.qlen, w.scale, w.window, 0, k_scale=w.k_scale,
                                 v_scale=w.v_scale)
    torch.cuda.synchronize()
    ref = oracle.decode_paged_varlen(bits(w.q), w.k_cache.numpy(), w.v_cache.numpy(),
                                     w.block_table.numpy(), w.seq_lens.numpy(), w.q_start.numpy(),
                                     w.scale, w.window, w.k_scale, w.v_scale, w.kv_fp8, w.kv_int8,
                                     bf16=True)
    check(w, got, ref)
