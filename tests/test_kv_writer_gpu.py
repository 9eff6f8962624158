"""GPU parity of the paged KV-cache writer (write_kv_cache through the C ABI)
against the oracle's writer: the caches must agree byte for byte (fp16 bit
copies, e4m3fn and int8 codes), on sentinel-filled caches so that stray or
missing writes show. Then the decode reads what the writer stored, as the
writer-layout cell of opengfx1030/vllm-rdna pull request #33 ("Test Plan")
does.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_split_decode_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KINDS = ("f16", "fp8", "int8")


@pytest.fixture(scope="module")
def pd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_split_decode_gb300 as pd
    pd.load()
    return pd


def sentinel_caches(kind, num_blocks, bs, Hkv, D):
    shape = (num_blocks, bs, Hkv, D)
    if kind == "f16":
        k = torch.full(shape, 0x7E01, dtype=torch.int32).to(torch.int16).view(torch.float16)
    else:
        k = torch.full(shape, 0x5A, dtype=torch.uint8)
    return k, k.clone()


def dev_cache(kind, c):
    c = c.to(DEV)
    return c.view(torch.int8) if kind == "int8" else c


def run_both(pd, kind, w, k_scale=1.0, v_scale=1.0, flag=None):
    """Write w through the GPU and through the oracle; returns the four caches
    as uint8 numpy arrays and the oracle's all-slots-in-range verdict."""
    D, Hkv = w.k_new.shape[2], w.k_new.shape[1]
    kc, vc = sentinel_caches(kind, w.num_blocks, w.block_size, Hkv, D)
    kd, vd = dev_cache(kind, kc), dev_cache(kind, vc)
    pd.write_kv_cache(w.k_new.to(DEV), w.v_new.to(DEV), w.slot_mapping.to(DEV), kd, vd,
                      k_scale=k_scale, v_scale=v_scale, error_flag=flag)
    torch.cuda.synchronize()
    ko, vo = kc.numpy().copy(), vc.numpy().copy()
    ok = oracle.write_kv_cache(w.k_new.numpy(), w.v_new.numpy(), w.slot_mapping.numpy(), ko, vo,
                               k_scale=k_scale, v_scale=v_scale, kv_fp8=kind == "fp8",
                               kv_int8=kind == "int8", allow_bad_slots=True)
    as_u8 = lambda t: t.cpu().contiguous().view(torch.uint8).numpy()
    return as_u8(kd), as_u8(vd), ko.view(np.uint8), vo.view(np.uint8), ok


def assert_same_bytes(got, want, what):
    bad = np.nonzero(got.reshape(-1) != want.reshape(-1))[0]
    assert bad.size == 0, f"{what}: {bad.size} bytes differ, first at {bad[:4]}"


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("T,Hkv,D,num_blocks,bs", [
    (1, 1, 8, 1, 16), (37, 3, 40, 11, 16), (300, 4, 256, 40, 16), (1000, 8, 128, 70, 16),
    (129, 2, 256, 17, 32),
])
def test_writer_matches_oracle_bytes(pd, kind, T, Hkv, D, num_blocks, bs):
    w = inputs.make_writer_inputs(T, Hkv, D, num_blocks, bs, seed=T + D, pad_every=7,
                                  specials=True)
    ks, vs = (0.037, 0.051) if kind != "f16" else (1.0, 1.0)
    kg, vg, ko, vo, ok = run_both(pd, kind, w, ks, vs)
    assert ok
    assert_same_bytes(kg, ko, "k_cache")
    assert_same_bytes(vg, vo, "v_cache")


@pytest.mark.parametrize("kind", ("fp8", "int8"))
@pytest.mark.parametrize("scale", (1.0, 0.037, 3.0, 1.0 / 448, 1e-3, 250.0))
def test_writer_every_f16_pattern(pd, kind, scale):
    """All 65536 fp16 inputs through the quantiser at several scales: the fp32
    division, the rounding ties, saturation, subnormals, infinities and NaN."""
    x = inputs.all_f16_patterns(Hkv=1, D=256)
    T = x.shape[0]
    w = inputs.WriterInputs(x, x.flip(0).contiguous(), torch.arange(T, dtype=torch.int64), T, 1)
    kg, vg, ko, vo, ok = run_both(pd, kind, w, scale, scale * 0.5)
    assert ok
    assert_same_bytes(kg, ko, "k_cache")
    assert_same_bytes(vg, vo, "v_cache")


def test_writer_every_f16_pattern_copy(pd):
    x = inputs.all_f16_patterns(Hkv=2, D=128)
    T = x.shape[0]
    w = inputs.WriterInputs(x, x.flip(0).contiguous(), torch.arange(T, dtype=torch.int64), T, 1)
    kg, vg, ko, vo, ok = run_both(pd, "f16", w)
    assert_same_bytes(kg, ko, "k_cache")
    assert_same_bytes(vg, vo, "v_cache")


@pytest.mark.parametrize("kind", KINDS)
def test_writer_bad_slots_flagged_and_skipped(pd, kind):
    w = inputs.make_writer_inputs(16, 2, 64, 5, seed=3)
    cap = w.num_blocks * w.block_size
    w.slot_mapping[:] = torch.tensor([3, cap, 17, -5, cap + 100, 40, 0, 2 * cap, 1, 2, 4, 5, 6, 7,
                                      8, -1], dtype=torch.int64)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    kg, vg, ko, vo, ok = run_both(pd, kind, w, 0.02, 0.03, flag=flag)
    assert not ok
    assert int(flag.item()) == pd.DEVERR_SLOT
    assert_same_bytes(kg, ko, "k_cache")
    assert_same_bytes(vg, vo, "v_cache")


@pytest.mark.parametrize("kind", KINDS)
def test_writer_no_tokens_is_a_no_op(pd, kind):
    kc, vc = sentinel_caches(kind, 3, 16, 2, 64)
    kd, vd = dev_cache(kind, kc), dev_cache(kind, vc)
    e = torch.empty((0, 2, 64), dtype=torch.float16, device=DEV)
    pd.write_kv_cache(e, e, torch.empty(0, dtype=torch.int64, device=DEV), kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu().view(torch.uint8), kc.view(torch.uint8))


def test_writer_rejects_bad_arguments(pd):
    kc = torch.zeros((2, 16, 2, 64), dtype=torch.float16, device=DEV)
    x = torch.zeros((4, 2, 64), dtype=torch.float16, device=DEV)
    with pytest.raises(ValueError):
        pd.write_kv_cache(x, x, torch.zeros(3, dtype=torch.int64, device=DEV), kc, kc.clone())
    with pytest.raises(TypeError):
        pd.write_kv_cache(x, x, torch.zeros(4, dtype=torch.int32, device=DEV), kc, kc.clone())
    odd = torch.zeros((2, 16, 2, 12), dtype=torch.float16, device=DEV)
    y = torch.zeros((4, 2, 12), dtype=torch.float16, device=DEV)
    with pytest.raises(pd.DecodeError):  # D not a multiple of 8
        pd.write_kv_cache(y, y, torch.zeros(4, dtype=torch.int64, device=DEV), odd, odd.clone())


@pytest.mark.parametrize("kind", KINDS)
def test_decode_reads_what_the_writer_wrote(pd, kind):
    """Fill a paged cache token by token with the writer (through a permuted
    block table), decode it, and compare with the oracle decoding the
    oracle-written cache (byte-identical, checked first)."""
    B, Hq, Hkv, D, bs = 3, 12, 2, 128, 16
    lens = [45, 0, 130]
    nb = sum((L + bs - 1) // bs for L in lens) + 3
    g = torch.Generator().manual_seed(11)
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    mb = max((L + bs - 1) // bs for L in lens)
    table = torch.full((B, mb), -1, dtype=torch.int32)
    slots, used = [], 0
    for b, L in enumerate(lens):
        n = (L + bs - 1) // bs
        table[b, :n] = perm[used:used + n]
        used += n
        slots += [int(table[b, j // bs]) * bs + j % bs for j in range(L)]
    T = len(slots)
    w = inputs.make_writer_inputs(T, Hkv, D, nb, bs, seed=5)
    w.slot_mapping = torch.tensor(slots, dtype=torch.int64)
    ks, vs = (0.02, 0.03) if kind != "f16" else (1.0, 1.0)
    kg, vg, ko, vo, ok = run_both(pd, kind, w, ks, vs)
    assert_same_bytes(kg, ko, "k_cache")
    assert_same_bytes(vg, vo, "v_cache")
    q = (torch.randn((B, Hq, D), generator=g)).half()
    sl = torch.tensor(lens, dtype=torch.int32)
    shape = (nb, bs, Hkv, D)
    dt = {"f16": torch.float16, "fp8": torch.uint8, "int8": torch.int8}[kind]
    kd = torch.from_numpy(kg).view(dt).reshape(shape).to(DEV)
    vd = torch.from_numpy(vg).view(dt).reshape(shape).to(DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pd.decode_paged(q.to(DEV), kd, vd, table.to(DEV), sl.to(DEV), 0.09, 0, 1, 0,
                          k_scale=ks, v_scale=vs, error_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    kview = ko.view(np.uint16).reshape(shape) if kind == "f16" else ko.reshape(shape)
    vview = vo.view(np.uint16).reshape(shape) if kind == "f16" else vo.reshape(shape)
    ref = oracle.decode_paged(q.numpy(), kview, vview, table.numpy(), sl.numpy(), 0.09,
                              k_scale=ks, v_scale=vs, kv_fp8=kind == "fp8", kv_int8=kind == "int8")
    got = out.float().cpu().numpy()
    assert np.max(np.abs(got - ref)) <= 2e-3
    assert np.all(got[1] == 0.0)


@pytest.mark.parametrize("kind", ("f16", "fp8"))
def test_writer_prefill_size_sampled(pd, kind):
    """A prefill-sized write (32768 tokens, 4 KV heads, D=256, as one long
    sequence of the decode benchmarks) checked on 512 sampled tokens."""
    T, Hkv, D, bs = 32768, 4, 256, 16
    nb = T // bs + 64
    w = inputs.make_writer_inputs(T, Hkv, D, nb, bs, seed=77, pad_every=1001)
    kc, vc = sentinel_caches(kind, nb, bs, Hkv, D)
    kd, vd = dev_cache(kind, kc), dev_cache(kind, vc)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    ks, vs = (0.011, 0.013) if kind == "fp8" else (1.0, 1.0)
    pd.write_kv_cache(w.k_new.to(DEV), w.v_new.to(DEV), w.slot_mapping.to(DEV), kd, vd,
                      k_scale=ks, v_scale=vs, error_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    g = torch.Generator().manual_seed(1)
    pick = torch.randperm(T, generator=g)[:512]
    sub = inputs.WriterInputs(w.k_new[pick].contiguous(), w.v_new[pick].contiguous(),
                              w.slot_mapping[pick].contiguous(), nb, bs)
    ko, vo = kc.numpy().copy(), vc.numpy().copy()
    oracle.write_kv_cache(sub.k_new.numpy(), sub.v_new.numpy(), sub.slot_mapping.numpy(), ko, vo,
                          k_scale=ks, v_scale=vs, kv_fp8=kind == "fp8")
    live = sub.slot_mapping[sub.slot_mapping >= 0]
    blk, off = (live // bs).numpy(), (live % bs).numpy()
    kgot = kd.cpu().view(torch.uint8).numpy()
    vgot = vd.cpu().view(torch.uint8).numpy()
    assert_same_bytes(kgot[blk, off], ko.view(np.uint8)[blk, off], "k_cache")
    assert_same_bytes(vgot[blk, off], vo.view(np.uint8)[blk, off], "v_cache")
    # padding tokens and unused slots keep the sentinel
    pad = torch.ones(nb * bs, dtype=torch.bool)
    pad[w.slot_mapping[w.slot_mapping >= 0]] = False
    idx = torch.nonzero(pad).squeeze(1)[:2000]
    sent = kc.view(torch.uint8).numpy()
    assert_same_bytes(kgot.reshape(nb * bs, -1)[idx.numpy()], sent.reshape(nb * bs, -1)[idx.numpy()],
                      "untouched slots")
