"""Pins for the oracle's paged KV-cache writer and its quantisers, independent
of the oracle's own code.

* quantisers: hand-derived code points (tests/golden/quantiser_points.json),
  every finite e4m3fn code round-trips, torch's float8_e4m3fn cast (round to
  nearest even) on in-range values, numpy's rint + clip for int8;
* writer: every token lands at block slot // block_size, offset slot %
  block_size (numpy fancy indexing), padding tokens and untouched slots keep
  their sentinel bytes, fp8 / int8 codes equal the library quantisers of
  fp32(x) / fp32(scale), an out-of-range slot is reported and skipped, and the
  decode of what was written stays within half a code step of the input.
"""
import json
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _points():
    return json.load(open(os.path.join(GOLDEN, "quantiser_points.json")))


# ---- quantisers --------------------------------------------------------------

def test_e4m3fn_encoder_golden_points(oracle_lib):
    for c in _points()["e4m3fn"]:
        assert oracle_lib.e4m3fn_encode(float(c["t"])) == c["code"], c


def test_i8_encoder_golden_points(oracle_lib):
    for c in _points()["int8"]:
        assert oracle_lib.i8_encode(float(c["t"])) == c["code"], c


def test_e4m3fn_encoder_roundtrips_every_code(oracle_lib):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    for c, v in enumerate(vals):
        if np.isnan(v):
            continue
        assert oracle_lib.e4m3fn_encode(float(v)) == c, (c, v)


def _e4m3_midpoints():
    codes = torch.arange(0, 0x7F, dtype=torch.int32).to(torch.uint8)
    v = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mids = (v[:-1] + v[1:]) / 2  # exact in fp32 (at most 5 significant bits)
    return np.concatenate([mids, -mids]).astype(np.float32)


def test_e4m3fn_encoder_matches_torch_cast(oracle_lib):
    g = np.random.default_rng(5)
    t = np.concatenate([
        _e4m3_midpoints(),
        np.nextafter(_e4m3_midpoints(), np.float32(np.inf)),
        np.nextafter(_e4m3_midpoints(), np.float32(-np.inf)),
        (g.standard_normal(3000) * 40).astype(np.float32),
        (g.standard_normal(1000) * 0.01).astype(np.float32),
        g.uniform(-448, 448, 1000).astype(np.float32),
    ]).astype(np.float32)
    t = t[np.abs(t) <= 448]
    want = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_lib.e4m3fn_encode(float(x)) for x in t], dtype=np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(t[i]), int(got[i]), int(want[i])) for i in bad[:5]]


def test_e4m3fn_encoder_saturates_beyond_range(oracle_lib):
    t = np.array([448.5, 463.9, 464.0, 479.0, 480.0, 1e4, 3e38], dtype=np.float32)
    for x in t:
        assert oracle_lib.e4m3fn_encode(float(x)) == 0x7E
        assert oracle_lib.e4m3fn_encode(float(-x)) == 0xFE


def test_i8_encoder_matches_numpy(oracle_lib):
    g = np.random.default_rng(6)
    t = np.concatenate([np.arange(-140, 140.5, 0.5), g.standard_normal(3000) * 60,
                        g.uniform(-1, 1, 500)]).astype(np.float32)
    want = np.clip(np.rint(t.astype(np.float64)), -127, 127).astype(np.int64)
    got = np.array([oracle_lib.i8_encode(float(x)) for x in t])
    assert np.array_equal(got, want)


# ---- writer ------------------------------------------------------------------

# 16-bit caches take the new tokens' bits (fp16, or bfloat16 for a bfloat16
# model); byte caches quantise fp16 new tokens, or bfloat16 ones under a
# bfloat16 model
KINDS = ("f16", "bf16", "fp8", "int8", "fp8_bf16q", "int8_bf16q")


def _bf16_tokens(kind):
    return kind == "bf16" or kind.endswith("bf16q")


def _bf16_bits(x):
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _tokens_f32(x, kind):
    """The new tokens' values (fp16 arrays, or bfloat16 bit patterns)."""
    if _bf16_tokens(kind):
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    return x.astype(np.float32)


def _writer_case(kind, seed=0, T=37, num_blocks=11, bs=16, Hkv=3, D=40):
    g = np.random.default_rng(seed)
    k_new = (g.standard_normal((T, Hkv, D)) * 2).astype(np.float16)
    v_new = (g.standard_normal((T, Hkv, D)) * 3).astype(np.float16)
    if _bf16_tokens(kind):
        k_new, v_new = _bf16_bits(k_new), _bf16_bits(v_new)
    slots = g.permutation(num_blocks * bs)[:T].astype(np.int64)
    slots[::7] = -1  # padding tokens
    if kind == "f16":
        kc = np.full((num_blocks, bs, Hkv, D), 0x7E01, dtype=np.uint16).view(np.float16)
    elif kind == "bf16":
        kc = np.full((num_blocks, bs, Hkv, D), 0x7FC1, dtype=np.uint16)
    else:
        kc = np.full((num_blocks, bs, Hkv, D), 0x5A, dtype=np.uint8)
    vc = kc.copy()
    return k_new, v_new, slots, kc, vc


def _flags(kind):
    return dict(kv_fp8=kind.startswith("fp8"), kv_int8=kind.startswith("int8"),
                bf16=_bf16_tokens(kind))


def _quantise_lib(x, scale, kind):
    t = torch.from_numpy(_tokens_f32(x, kind)) / torch.tensor(np.float32(scale))
    if kind.startswith("fp8"):
        return t.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return np.clip(np.rint(t.numpy().astype(np.float64)), -127, 127).astype(np.int8).view(np.uint8)


@pytest.mark.parametrize("kind", KINDS)
def test_writer_layout_and_codes(oracle_lib, kind):
    k_new, v_new, slots, kc, vc = _writer_case(kind, seed=KINDS.index(kind))
    ks, vs = np.float32(0.037), np.float32(0.051)
    kc0, vc0 = kc.copy(), vc.copy()
    assert oracle_lib.write_kv_cache(k_new, v_new, slots, kc, vc, k_scale=ks, v_scale=vs,
                                     **_flags(kind))
    bs = kc.shape[1]
    live = slots >= 0
    blk, off = slots[live] // bs, slots[live] % bs
    if kind in ("f16", "bf16"):
        # a 16-bit cache holds the new tokens' bit patterns, two bytes each
        assert kc.dtype.itemsize == 2
        want_k, want_v = k_new[live], v_new[live]
        assert np.array_equal(kc[blk, off].view(np.uint16), want_k.view(np.uint16))
        assert np.array_equal(vc[blk, off].view(np.uint16), want_v.view(np.uint16))
    else:
        assert np.array_equal(kc[blk, off], _quantise_lib(k_new[live], ks, kind))
        assert np.array_equal(vc[blk, off], _quantise_lib(v_new[live], vs, kind))
    # every other slot keeps its sentinel
    mask = np.ones(kc.shape[:2], dtype=bool)
    mask[blk, off] = False
    assert np.array_equal(kc[mask].view(np.uint8), kc0[mask].view(np.uint8))
    assert np.array_equal(vc[mask].view(np.uint8), vc0[mask].view(np.uint8))


@pytest.mark.parametrize("kind", KINDS)
def test_writer_bad_slot_is_reported_and_skipped(oracle_lib, kind):
    k_new, v_new, slots, kc, vc = _writer_case(kind, seed=9, T=8)
    cap = kc.shape[0] * kc.shape[1]
    slots = np.array([3, cap, 17, -5, cap + 100, 40, 0, 2 * cap], dtype=np.int64)
    with pytest.raises(ValueError):
        oracle_lib.write_kv_cache(k_new, v_new, slots, kc.copy(), vc.copy(), **_flags(kind))
    kc_a, vc_a = kc.copy(), vc.copy()
    assert not oracle_lib.write_kv_cache(k_new, v_new, slots, kc_a, vc_a, allow_bad_slots=True,
                                         **_flags(kind))
    good = np.array([0, 2, 5, 6])
    kc_b, vc_b = kc.copy(), vc.copy()
    assert oracle_lib.write_kv_cache(k_new[good], v_new[good], slots[good], kc_b, vc_b,
                                     **_flags(kind))
    assert np.array_equal(kc_a.view(np.uint8), kc_b.view(np.uint8))
    assert np.array_equal(vc_a.view(np.uint8), vc_b.view(np.uint8))


@pytest.mark.parametrize("kind", ("fp8", "int8"))
def test_writer_then_decode_is_within_half_a_step(oracle_lib, kind):
    """What the writer stores decodes (code * scale) to within half a code step
    of the fp32 input: the writer and the decode read the same layout and
    agree on the scale's direction."""
    k_new, v_new, slots, kc, vc = _writer_case(kind, seed=21)
    scale = np.float32(0.02)
    oracle_lib.write_kv_cache(k_new, v_new, slots, kc, vc, k_scale=scale, v_scale=scale,
                              **_flags(kind))
    bs = kc.shape[1]
    live = slots >= 0
    codes = kc[slots[live] // bs, slots[live] % bs]
    dec = (oracle_lib.e4m3fn_to_f64 if kind == "fp8" else oracle_lib.i8_to_f64)
    lut = np.array([dec(c) for c in range(256)])
    x = k_new[live].astype(np.float64) / float(scale)
    y = lut[codes]
    fp32_div = np.abs(x) * 2.0 ** -23  # the quotient is rounded to fp32 first
    if kind == "int8":
        assert np.all(np.abs(y - np.clip(x, -127, 127)) <= 0.5 + fp32_div)
    else:
        # e4m3: the step at magnitude |x| is 2^(floor(log2|x|) - 3), subnormal step 2^-9
        ax = np.minimum(np.abs(x), 448)
        e = np.floor(np.log2(np.maximum(ax, 2.0 ** -6)))
        step = 2.0 ** (e - 3)
        assert np.all(np.abs(y - np.clip(x, -448, 448)) <= step / 2 + fp32_div)


def test_writer_f16_then_oracle_decode_reads_the_tokens(oracle_lib):
    """A sequence assembled by the writer decodes like the same keys laid out
    by the input generator: the writer's layout is the decode's layout."""
    g = np.random.default_rng(3)
    Hq, Hkv, D, bs, L = 4, 2, 32, 16, 45
    nb = 8
    k_tok = (g.standard_normal((L, Hkv, D))).astype(np.float16)
    v_tok = (g.standard_normal((L, Hkv, D))).astype(np.float16)
    table = g.permutation(nb)[:4].astype(np.int32)
    slots = np.array([table[j // bs] * bs + j % bs for j in range(L)], dtype=np.int64)
    kc = np.zeros((nb, bs, Hkv, D), dtype=np.float16)
    vc = np.zeros_like(kc)
    oracle_lib.write_kv_cache(k_tok, v_tok, slots, kc, vc)
    q = (g.standard_normal((1, Hq, D))).astype(np.float16)
    out = oracle_lib.decode_paged(q, kc, vc, table[None, :], np.array([L], np.int32), 0.2)
    # dense statement: softmax over all L keys of the matching KV head
    G = Hq // Hkv
    for h in range(Hq):
        s = 0.2 * (k_tok[:, h // G].astype(np.float64) @ q[0, h].astype(np.float64))
        w = np.exp(s - s.max())
        want = (w[:, None] * v_tok[:, h // G].astype(np.float64)).sum(0) / w.sum()
        assert np.allclose(out[0, h], want, rtol=0, atol=1e-12)
