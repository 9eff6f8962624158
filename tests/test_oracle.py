"""Pins for the fp64 oracle, independent of the oracle's own code.

* decoders: every fp16 bit pattern against numpy, every e4m3fn code against
  torch and the OCP code points in tests/golden;
* closed forms: the hand-derived cases in tests/golden/closed_forms.json and
  single-key / two-key / constant-V / scale-0 / empty-row identities;
* brute force: a dense numpy softmax (tests/ref_dense.py) and torch's fp64
  scaled_dot_product_attention on tiny paged inputs;
* invariants: split count, physical block permutation, window = truncation.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import ref_dense
from paged_split_decode_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    if isinstance(t, torch.Tensor):
        if t.dtype == torch.bfloat16:  # numpy has no bfloat16: hand over the bit patterns
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    return t


def run_oracle(oracle, w, split=None, **kw):
    args = dict(scale=w.scale, window=w.window, qlen=w.qlen, k_scale=w.k_scale,
                v_scale=w.v_scale, kv_fp8=w.kv_fp8, kv_int8=w.kv_int8, bf16=w.bf16)
    args.update(kw)
    if split is None:
        return oracle.decode_paged(_np(w.q), _np(w.k_cache), _np(w.v_cache), _np(w.block_table),
                                   _np(w.seq_lens), **args)
    return oracle.decode_paged_split(_np(w.q), _np(w.k_cache), _np(w.v_cache), _np(w.block_table),
                                     _np(w.seq_lens), num_splits=split, **args)


def run_dense(w):
    return ref_dense.attention(_np(w.q), _np(w.k_cache), _np(w.v_cache), _np(w.block_table),
                               _np(w.seq_lens), w.scale, w.window, w.qlen, w.kv_fp8, w.k_scale,
                               w.v_scale, w.kv_int8, bf16=w.bf16)


# ---- element decoders ----------------------------------------------------------

def test_f16_decoder_every_pattern(oracle_lib):
    bits = np.arange(65536, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_e4m3fn_decoder_every_code(oracle_lib):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle_lib.e4m3fn_to_f64(c) for c in range(256)])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_decoder_every_pattern(oracle_lib):
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    want = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_lib.bf16_to_f64(b) for b in range(65536)])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_int8_decoder_every_code(oracle_lib):
    want = np.arange(256, dtype=np.uint8).view(np.int8).astype(np.float64)
    got = np.array([oracle_lib.i8_to_f64(c) for c in range(256)])
    assert np.array_equal(got, want)
    assert oracle_lib.i8_to_f64(0x80) == -128.0 and oracle_lib.i8_to_f64(0x7F) == 127.0


def test_e4m3fn_spec_points(oracle_lib):
    pts = json.load(open(os.path.join(GOLDEN, "e4m3fn_points.json")))["points"]
    for p in pts:
        got = oracle_lib.e4m3fn_to_f64(p["code"])
        if p["value"] == "nan":
            assert math.isnan(got), p
        else:
            want = float(eval(p["value"]))
            assert got == want and math.copysign(1, got) == math.copysign(1, want), p


# ---- hand-derived closed forms ---------------------------------------------------

def _golden_workload(case):
    B, Hq, Hkv, D = case["B"], case["Hq"], case["Hkv"], case["D"]
    bs, qlen = case["block_size"], case["qlen"]
    lens = case["seq_lens"]
    fp8 = case.get("kv") in ("fp8", "int8")
    need = [(L + bs - 1) // bs for L in lens]
    pool = sum(need) + 1
    maxb = max(need + [1])
    table = np.full((B, maxb), -1, dtype=np.int32)
    # hand the blocks out in reverse pool order so that paging is exercised
    nxt = pool - 1
    for b in range(B):
        for lb in range(need[b]):
            table[b, lb] = nxt
            nxt -= 1
    dt = np.uint8 if fp8 else np.float16
    K = np.zeros((pool, bs, Hkv, D), dtype=dt)
    V = np.zeros((pool, bs, Hkv, D), dtype=dt)
    for b in range(B):
        for kh in range(Hkv):
            for j, (kr, vr) in enumerate(zip(case["keys"][b][kh], case["values"][b][kh])):
                K[table[b, j // bs], j % bs, kh] = kr
                V[table[b, j // bs], j % bs, kh] = vr
    q = np.array(case["q"], dtype=np.float16).reshape(B * qlen, Hq, D)
    return q, K, V, table, np.array(lens, dtype=np.int32)


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "closed_forms.json")))["cases"],
                         ids=lambda c: c["name"])
def test_golden_closed_forms(oracle_lib, case):
    q, K, V, table, lens = _golden_workload(case)
    fp8 = case.get("kv") == "fp8"
    kw = dict(scale=case["scale"], window=case["window"], qlen=case["qlen"], kv_fp8=fp8,
              kv_int8=case.get("kv") == "int8",
              k_scale=case.get("k_scale", 1.0), v_scale=case.get("v_scale", 1.0))
    env = {"e": math.e, "exp": math.exp, "sqrt": math.sqrt}
    want = np.array([[eval(x, env) for x in row] for row in case["expected"]])
    got = oracle_lib.decode_paged(q, K, V, table, lens, **kw).reshape(want.shape)
    assert np.allclose(got, want, rtol=1e-14, atol=1e-15), (got, want)
    for S in (1, 2, 3):
        got_s = oracle_lib.decode_paged_split(q, K, V, table, lens, num_splits=S, **kw)
        assert np.allclose(got_s.reshape(want.shape), want, rtol=1e-14, atol=1e-15)
    # rows that must be empty are exact zeros, not merely small
    empty = (want == 0).all(axis=1)
    assert np.all(got.reshape(want.shape)[empty] == 0.0)


# ---- brute force on tiny paged inputs -------------------------------------------------

TINY = [
    dict(B=1, Hq=1, Hkv=1, D=4, qlen=1, lens=[1], bs=1, window=0),
    dict(B=2, Hq=2, Hkv=1, D=8, qlen=1, lens=[5, 17], bs=4, window=0),
    dict(B=3, Hq=6, Hkv=2, D=8, qlen=2, lens=[9, 0, 33], bs=4, window=0),
    dict(B=3, Hq=4, Hkv=4, D=4, qlen=3, lens=[2, 3, 40], bs=16, window=5),
    dict(B=2, Hq=6, Hkv=1, D=128, qlen=1, lens=[70, 31], bs=16, window=20),
    dict(B=2, Hq=8, Hkv=2, D=128, qlen=3, lens=[100, 48], bs=16, window=0),
    dict(B=1, Hq=3, Hkv=1, D=8, qlen=1, lens=[16], bs=16, window=16),
    dict(B=2, Hq=2, Hkv=2, D=8, qlen=2, lens=[1, 2], bs=4, window=1),
]


def _tiny(c, kv="f16", seed=7, layout="permuted", scale=None):
    return inputs.make_workload(B=c["B"], Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"], qlen=c["qlen"],
                                seq_lens=c["lens"], block_size=c["bs"], window=c["window"],
                                kv=kv, seed=seed, layout=layout, scale=scale,
                                pool_blocks=sum((L + c["bs"] - 1) // c["bs"] for L in c["lens"]) + 3)


KV_KINDS = ["f16", "fp8", "int8", "bf16", "fp8_bf16q", "int8_bf16q"]


@pytest.mark.parametrize("kv", KV_KINDS)
@pytest.mark.parametrize("ci", range(len(TINY)))
def test_oracle_matches_dense_bruteforce(oracle_lib, ci, kv):
    w = _tiny(TINY[ci], kv=kv, seed=100 + ci)
    got = run_oracle(oracle_lib, w)
    want = run_dense(w)
    assert np.max(np.abs(got - want)) <= 1e-12


@pytest.mark.parametrize("kv", ["fp8", "int8"])
@pytest.mark.parametrize("ci", [1, 4, 5])
def test_bf16_q_over_byte_caches_equals_f16_q(oracle_lib, ci, kv):
    """A q whose values are exact in both fp16 and bfloat16 gives the same
    fp64 output, bit for bit, over the same byte caches whichever type it
    arrives in."""
    w = _tiny(TINY[ci], kv=kv, seed=300 + ci)
    g = torch.Generator().manual_seed(ci)
    # 8 significant bits and a modest exponent: exact in both types
    qv = (torch.randint(-255, 256, w.q.shape, generator=g).to(torch.float64) *
          torch.pow(2.0, torch.randint(-9, -3, w.q.shape, generator=g).to(torch.float64)))
    w.q = qv.to(torch.float16)
    assert torch.equal(w.q.to(torch.float64), qv)
    f16 = run_oracle(oracle_lib, w)
    w.q, w.bf16 = qv.to(torch.bfloat16), True
    assert torch.equal(w.q.to(torch.float64), qv)
    b16 = run_oracle(oracle_lib, w)
    assert np.array_equal(f16, b16)


@pytest.mark.parametrize("kv", ["f16", "bf16"])
@pytest.mark.parametrize("ci", [1, 2, 4, 5])
def test_oracle_matches_torch_sdpa(oracle_lib, ci, kv):
    """Dense fp64 torch scaled_dot_product_attention with a boolean mask per token."""
    w = _tiny(TINY[ci], kv=kv, seed=200 + ci)
    got = run_oracle(oracle_lib, w)
    Kc = w.k_cache.to(torch.float64)
    Vc = w.v_cache.to(torch.float64)
    G = w.Hq // w.Hkv
    for b in range(w.B):
        L = int(w.seq_lens[b])
        rows = slice(b * w.qlen, (b + 1) * w.qlen)
        if L == 0:
            assert np.all(got[rows] == 0)
            continue
        idx = [(int(w.block_table[b, j // w.block_size]), j % w.block_size) for j in range(L)]
        Kd = torch.stack([Kc[blk, s] for blk, s in idx]).repeat_interleave(G, dim=1)  # [L,Hq,D]
        Vd = torch.stack([Vc[blk, s] for blk, s in idx]).repeat_interleave(G, dim=1)
        qb = w.q[rows].to(torch.float64)                      # [qlen,Hq,D]
        mask = torch.from_numpy(ref_dense.visibility(L, w.qlen, w.window))  # [qlen,L]
        o = torch.nn.functional.scaled_dot_product_attention(
            qb.transpose(0, 1), Kd.transpose(0, 1), Vd.transpose(0, 1),
            attn_mask=mask[None], scale=w.scale)               # [Hq,qlen,D]
        o = o.transpose(0, 1).numpy()
        seen = mask.any(dim=1).numpy()
        assert np.max(np.abs(got[rows][seen] - o[seen])) <= 1e-12
        assert np.all(got[rows][~seen] == 0)


# ---- identities -------------------------------------------------------------------------

def test_constant_v_returns_v(oracle_lib):
    w = _tiny(TINY[5], seed=11)
    c = torch.linspace(-2, 2, w.D).to(torch.float16)
    w.v_cache[:] = c
    got = run_oracle(oracle_lib, w)
    for b in range(w.B):
        rows = got[b * w.qlen:(b + 1) * w.qlen]
        assert np.allclose(rows, c.double().numpy()[None, None, :], rtol=0, atol=1e-14)


def test_scale_zero_gives_mean_of_visible_v(oracle_lib):
    w = _tiny(TINY[3], seed=12, scale=0.0)
    got = run_oracle(oracle_lib, w)
    Vc = w.v_cache.double()
    G = w.Hq // w.Hkv
    for b in range(w.B):
        L = int(w.seq_lens[b])
        vis = ref_dense.visibility(L, w.qlen, w.window)
        for i in range(w.qlen):
            for h in range(w.Hq):
                js = np.nonzero(vis[i])[0]
                o = got[b * w.qlen + i, h]
                if len(js) == 0:
                    assert np.all(o == 0)
                    continue
                rows = [Vc[int(w.block_table[b, j // w.block_size]), j % w.block_size, h // G]
                        for j in js]
                assert np.allclose(o, torch.stack(rows).mean(0).numpy(), rtol=0, atol=1e-14)


def test_two_keys_is_a_sigmoid_mix(oracle_lib):
    w = inputs.make_workload(B=1, Hq=1, Hkv=1, D=8, seq_lens=[2], block_size=1, seed=13)
    got = run_oracle(oracle_lib, w)[0, 0]
    q = w.q[0, 0].double()
    k = [w.k_cache[int(w.block_table[0, j]), 0, 0].double() for j in range(2)]
    v = [w.v_cache[int(w.block_table[0, j]), 0, 0].double() for j in range(2)]
    s1, s2 = (w.scale * float(q @ k[0])), (w.scale * float(q @ k[1]))
    sig = 1.0 / (1.0 + math.exp(-(s1 - s2)))
    want = (sig * v[0] + (1 - sig) * v[1]).numpy()
    assert np.allclose(got, want, rtol=0, atol=1e-14)


def test_empty_rows_are_exact_zero(oracle_lib):
    w = inputs.tiny()
    got = run_oracle(oracle_lib, w)
    assert np.all(got[1] == 0.0)
    assert np.all(np.abs(got[0]) > 0)


# ---- invariants ------------------------------------------------------------------------

@pytest.mark.parametrize("kv", ["f16", "fp8", "int8", "bf16"])
@pytest.mark.parametrize("ci", [1, 2, 3, 4, 5, 7])
def test_split_mode_matches_one_shot(oracle_lib, ci, kv):
    w = _tiny(TINY[ci], kv=kv, seed=300 + ci)
    one = run_oracle(oracle_lib, w)
    for S in (1, 3, 8, 17):
        got = run_oracle(oracle_lib, w, split=S)
        assert np.max(np.abs(got - one)) <= 1e-12, S


def test_split_partials_recombine(oracle_lib):
    w = _tiny(TINY[5], seed=31)
    out, m, l, O = oracle_lib.decode_paged_split(
        _np(w.q), _np(w.k_cache), _np(w.v_cache), _np(w.block_table), _np(w.seq_lens), w.scale,
        num_splits=3, qlen=w.qlen, return_partials=True)
    again = oracle_lib.combine(m, l, O).reshape(out.shape)
    assert np.array_equal(again, out)
    # one-chunk partials are (max, sum of weights, weighted sum): O/l is the one-shot row
    _, m1, l1, O1 = oracle_lib.decode_paged_split(
        _np(w.q), _np(w.k_cache), _np(w.v_cache), _np(w.block_table), _np(w.seq_lens), w.scale,
        num_splits=1, qlen=w.qlen, return_partials=True)
    one = run_oracle(oracle_lib, w).reshape(-1, w.D)
    ok = l1[:, 0] > 0
    assert np.max(np.abs(O1[ok, 0] / l1[ok, 0, None] - one[ok])) <= 1e-12


def test_combine_edge_cases(oracle_lib):
    D = 4
    m = np.array([[-np.inf, -np.inf], [0.5, -np.inf], [1.0, 1.0 + math.log(3.0)]])
    l = np.array([[0.0, 0.0], [2.0, 0.0], [1.0, 1.0]])
    O = np.zeros((3, 2, D))
    O[1, 0] = [2, 4, 6, 8]
    O[2, 0] = [1, 0, 0, 0]
    O[2, 1] = [0, 1, 0, 0]
    out = oracle_lib.combine(m, l, O)
    assert np.all(out[0] == 0)
    assert np.allclose(out[1], [1, 2, 3, 4], atol=1e-15)
    # weights 1 and 3 (the second chunk's max is larger by log 3)
    assert np.allclose(out[2], [0.25, 0.75, 0, 0], atol=1e-15)


def test_block_permutation_is_bitwise_invariant(oracle_lib):
    w = _tiny(TINY[5], seed=41)
    base = run_oracle(oracle_lib, w)
    pool = w.k_cache.shape[0]
    perm = torch.randperm(pool, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(pool)
    k2 = w.k_cache[perm]
    v2 = w.v_cache[perm]
    t2 = w.block_table.clone()
    ok = t2 >= 0
    t2[ok] = inv[t2[ok].long()].to(torch.int32)
    got = oracle_lib.decode_paged(_np(w.q), _np(k2), _np(v2), _np(t2), _np(w.seq_lens), w.scale,
                                  qlen=w.qlen)
    assert np.array_equal(got, base)


@pytest.mark.parametrize("W", [1, 5, 16, 33])
def test_window_equals_truncation(oracle_lib, W):
    L, bs = 70, 16
    w = inputs.make_workload(B=1, Hq=6, Hkv=2, D=16, seq_lens=[L], block_size=bs, window=W, seed=51)
    got = run_oracle(oracle_lib, w)
    # the last W keys copied into a fresh cache, dense from slot 0
    n = min(W, L)
    nb = (n + bs - 1) // bs
    K = torch.zeros((nb, bs, w.Hkv, w.D), dtype=torch.float16)
    V = torch.zeros_like(K)
    for t, j in enumerate(range(L - n, L)):
        src = (int(w.block_table[0, j // bs]), j % bs)
        K[t // bs, t % bs] = w.k_cache[src]
        V[t // bs, t % bs] = w.v_cache[src]
    table = torch.arange(nb, dtype=torch.int32)[None]
    trunc = oracle_lib.decode_paged(_np(w.q), _np(K), _np(V), _np(table),
                                    np.array([n], dtype=np.int32), w.scale)
    assert np.max(np.abs(got - trunc)) <= 1e-14


def test_mha_special_case_matches_per_head_softmax(oracle_lib):
    w = inputs.make_workload(B=2, Hq=3, Hkv=3, D=8, seq_lens=[20, 9], block_size=4, seed=61)
    got = run_oracle(oracle_lib, w)
    for b in range(2):
        L = int(w.seq_lens[b])
        for h in range(3):
            ks = torch.stack([w.k_cache[int(w.block_table[b, j // 4]), j % 4, h] for j in range(L)]).double()
            vs = torch.stack([w.v_cache[int(w.block_table[b, j // 4]), j % 4, h] for j in range(L)]).double()
            p = torch.softmax(w.scale * (ks @ w.q[b, h].double()), dim=0)
            assert np.allclose(got[b, h], (p @ vs).numpy(), rtol=0, atol=1e-14)


def test_errors_are_reported(oracle_lib):
    w = _tiny(TINY[1], seed=71)
    bad = w.block_table.clone()
    bad[0, 0] = 10_000
    with pytest.raises(ValueError, match="block id"):
        oracle_lib.decode_paged(_np(w.q), _np(w.k_cache), _np(w.v_cache), _np(bad),
                                _np(w.seq_lens), w.scale)
    long = w.seq_lens.clone()
    long[0] = 10_000
    with pytest.raises(ValueError, match="seq_len"):
        oracle_lib.decode_paged(_np(w.q), _np(w.k_cache), _np(w.v_cache), _np(w.block_table),
                                _np(long), w.scale)
