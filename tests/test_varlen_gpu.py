"""GPU parity of decode_paged_varlen (a different number of query tokens per
sequence) against the oracle's decode_paged_varlen, through the C ABI.
Tolerance as for the uniform decode: max abs error <= 2e-3, exact zeros for
rows that see no key; rows outside every sequence's range are never written.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_split_decode_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 2e-3


@pytest.fixture(scope="module")
def pd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_split_decode_gb300 as pd
    pd.load()
    return pd


def kv_dev(w):
    k, v = w.k_cache.to(DEV), w.v_cache.to(DEV)
    if w.kv_int8:
        k, v = k.view(torch.int8), v.view(torch.int8)
    return k, v


def gpu_varlen(pd, w, S, out=None, flag=None, q_start=None):
    k, v = kv_dev(w)
    qs = (w.q_start if q_start is None else q_start).to(DEV)
    res = pd.decode_paged_varlen(w.q.to(DEV), k, v, w.block_table.to(DEV), w.seq_lens.to(DEV), qs,
                                 w.qlen, w.scale, w.window, S, out=out, k_scale=w.k_scale,
                                 v_scale=w.v_scale, error_flag=flag)
    torch.cuda.synchronize()
    return res


def ref_varlen(w):
    return oracle.decode_paged_varlen(w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(),
                                      w.block_table.numpy(), w.seq_lens.numpy(), w.q_start.numpy(),
                                      w.scale, w.window, w.k_scale, w.v_scale, w.kv_fp8,
                                      w.kv_int8)


def check(got, ref):
    g = got.float().cpu().numpy()
    assert np.all(np.isfinite(g))
    err = float(np.max(np.abs(g - ref))) if g.size else 0.0
    assert err <= TOL, f"max abs err {err:.3e}"
    zero = np.all(ref == 0.0, axis=-1)
    assert np.all(g[zero] == 0.0)


CASES = [
    ("f16_d128_mixed", dict(qlens=[1, 4, 2, 0, 3, 1], Hq=16, Hkv=2, D=128,
                            seq_lens=[300, 45, 1, 17, 2000, 0])),
    ("f16_d256_gqa6", dict(qlens=[1, 2, 3, 4, 1, 1, 2], Hq=24, Hkv=4, D=256,
                           seq_lens=[4096, 100, 3, 2500, 17, 1, 800])),
    ("f16_window", dict(qlens=[5, 1, 8, 2], Hq=8, Hkv=2, D=128, window=37,
                        seq_lens=[500, 90, 1200, 4])),
    ("fp8_d256", dict(qlens=[3, 1, 2, 0], Hq=24, Hkv=4, D=256, kv="fp8",
                      seq_lens=[1000, 4000, 31, 50])),
    ("fp8_d128_rows_32", dict(qlens=[4, 1, 3], Hq=16, Hkv=2, D=128, kv="fp8", window=100,
                              seq_lens=[700, 2, 1500])),
    ("int8_d256", dict(qlens=[2, 2, 1, 4], Hq=8, Hkv=1, D=256, kv="int8",
                       seq_lens=[900, 64, 3000, 3])),
    ("mha_many", dict(qlens=[(i % 4) for i in range(40)], Hq=4, Hkv=4, D=128,
                      seq_lens=[17 * i + 1 for i in range(40)])),
    # more sequences than the balanced split's prefix holds (1024)
    ("beyond_balanced_split_batch", dict(qlens=[(i % 3) + 1 for i in range(1050)], Hq=8, Hkv=2, D=128,
                                         seq_lens=[(11 * i) % 151 + 3 for i in range(1050)])),
]


@pytest.mark.parametrize("S", [0, 1, 3])
@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_varlen_matches_oracle(pd, name, kw, S):
    kw = dict(kw)
    qlens = kw.pop("qlens")
    w = inputs.make_varlen_workload(qlens=qlens, B=len(qlens), seed=len(name) * 31 + S, name=name,
                                    **kw)
    check(gpu_varlen(pd, w, S), ref_varlen(w))


@pytest.mark.parametrize("S", [0, 1, 4])
def test_equal_counts_are_bitwise_the_uniform_decode(pd, S):
    w = inputs.make_workload(B=5, Hq=24, Hkv=4, D=256, qlen=3, seq_lens=[800, 3, 4000, 0, 77],
                             seed=8)
    w.q_start = torch.arange(0, 16, 3, dtype=torch.int32)
    k, v = kv_dev(w)
    uni = pd.decode_paged(w.q.to(DEV), k, v, w.block_table.to(DEV), w.seq_lens.to(DEV), w.scale,
                          0, 3, S)
    var = gpu_varlen(pd, w, S)
    assert torch.equal(uni, var)


def test_rows_outside_every_sequence_are_untouched(pd):
    w = inputs.make_varlen_workload(qlens=[2, 3, 1], B=3, Hq=8, Hkv=2, D=128,
                                    seq_lens=[100, 40, 7], seed=2)
    # rows 0..1 and 8..9 belong to no sequence: shift every start by 2, add 2 spare rows
    T = int(w.q_start[-1])
    q = torch.zeros((T + 4, 8, 128), dtype=torch.float16)
    q[2:2 + T] = w.q
    w.q = q
    w.q_start = w.q_start + 2
    out = torch.full((T + 4, 8, 128), 7.0, dtype=torch.float16, device=DEV)
    got = gpu_varlen(pd, w, 0, out=out)
    ref = ref_varlen(w)
    g = got.float().cpu().numpy()
    assert np.all(g[:2] == 7.0) and np.all(g[2 + T:] == 7.0)
    assert float(np.max(np.abs(g[2:2 + T] - ref[2:2 + T]))) <= TOL


@pytest.mark.parametrize("S", [0, 3])
def test_malformed_query_ranges_are_flagged_and_skipped(pd, S):
    w = inputs.make_varlen_workload(qlens=[2, 3, 1, 2], B=4, Hq=8, Hkv=2, D=128,
                                    seq_lens=[100, 40, 70, 33], seed=6)
    T = int(w.q_start[-1])
    good = w.q_start.clone()
    bad = good.clone()
    bad[2] = 1        # sequence 1: start 2, end 1 -> negative count; sequence 2 becomes 1..6
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((T, 8, 128), 5.0, dtype=torch.float16, device=DEV)
    w.qlen = 3
    got = gpu_varlen(pd, w, S, out=out, flag=flag, q_start=bad)
    assert int(flag.item()) & pd.DEVERR_QUERY_START
    # sequence 2 (5 tokens > max 3) is skipped too; sequences 0 and 3 are intact
    ref = ref_varlen(w)
    g = got.float().cpu().numpy()
    for b in (0, 3):
        a, e = int(good[b]), int(good[b + 1])
        assert float(np.max(np.abs(g[a:e] - ref[a:e]))) <= TOL


def test_varlen_gqa6_batch32_full_size(pd):
    """The decode benchmark's geometry (D=256, Hq=24, Hkv=4, L=4096, B=32) with
    1 to 4 query tokens per sequence (rows per unit up to 24)."""
    g = torch.Generator().manual_seed(12)
    qlens = torch.randint(1, 5, (32,), generator=g).tolist()
    w = inputs.make_varlen_workload(qlens=qlens, B=32, Hq=24, Hkv=4, D=256, seq_lens=[4096] * 32,
                                    seed=12)
    check(gpu_varlen(pd, w, 0), ref_varlen(w))


def test_writer_and_varlen_decode_in_one_cuda_graph(pd):
    """The serving step -- write the new tokens' K/V, then decode a batch with a
    query count per sequence -- captured once into a CUDA graph and replayed
    after new values are written into the same buffers."""
    Hq, Hkv, D, bs = 24, 4, 256, 16
    qlens = [1, 3, 2]
    lens = [700, 45, 1300]
    B = len(lens)
    nb = sum((L + bs - 1) // bs for L in lens) + 4
    g = torch.Generator().manual_seed(90)
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    mb = max((L + bs - 1) // bs for L in lens)
    table = torch.full((B, mb), -1, dtype=torch.int32)
    used = 0
    for b, L in enumerate(lens):
        n = (L + bs - 1) // bs
        table[b, :n] = perm[used:used + n]
        used += n
    # the new tokens are the last qlen_b keys of each sequence
    slots = torch.tensor([int(table[b, j // bs]) * bs + j % bs
                          for b, L in enumerate(lens) for j in range(L - qlens[b], L)],
                         dtype=torch.int64)
    starts = torch.tensor([0, 1, 4, 6], dtype=torch.int32)
    T = int(starts[-1])
    kc = (torch.randn((nb, bs, Hkv, D), generator=g)).half().to(DEV)
    vc = (torch.randn((nb, bs, Hkv, D), generator=g)).half().to(DEV)
    q = torch.empty((T, Hq, D), dtype=torch.float16, device=DEV)
    kn = torch.empty((T, Hkv, D), dtype=torch.float16, device=DEV)
    vn = torch.empty_like(kn)
    out = torch.empty_like(q)
    bt, sl, qs, sm = table.to(DEV), torch.tensor(lens, dtype=torch.int32, device=DEV), \
        starts.to(DEV), slots.to(DEV)
    dims = pd.dims_of(q, kc, bt, max(qlens))
    ws = torch.empty(max(pd.workspace_bytes(dims, max(qlens), 0), 1), dtype=torch.uint8, device=DEV)
    stream = torch.cuda.Stream()

    def step():
        pd.write_kv_cache(kn, vn, sm, kc, vc)
        pd.decode_paged_varlen(q, kc, vc, bt, sl, qs, max(qlens), 0.0625, out=out, workspace=ws)

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for seed in (1, 2):
        gg = torch.Generator().manual_seed(seed)
        q.copy_(torch.randn((T, Hq, D), generator=gg).half())
        kn.copy_(torch.randn((T, Hkv, D), generator=gg).half())
        vn.copy_(torch.randn((T, Hkv, D), generator=gg).half())
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ko, vo = kc.cpu().numpy(), vc.cpu().numpy()
        # the new tokens landed where the table says
        for t, s_ in enumerate(slots.tolist()):
            assert np.array_equal(ko[s_ // bs, s_ % bs], kn[t].cpu().numpy())
        ref = oracle.decode_paged_varlen(q.cpu().numpy(), ko, vo, table.numpy(),
                                         np.array(lens, np.int32), starts.numpy(), 0.0625)
        g_ = out.float().cpu().numpy()
        assert float(np.max(np.abs(g_ - ref))) <= TOL
