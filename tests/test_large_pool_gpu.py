"""Caches larger than 4 GiB. The blocks a decode call reads, and the slots
the writer stores, sit past the first 4 GiB of each cache tensor, so a 32-bit
byte offset anywhere (kernels, tensor maps, writer) would touch the wrong
place. The decode runs the head-group fp16 kernel and the tensor-memory int8
and fp8 kernels (three row tiles). The oracle sees the
same blocks gathered into a compact pool: the output does not depend on where
the blocks sit (the oracle's block-permutation invariance)."""
import numpy as np
import pytest
import torch

import oracle
from paged_split_decode_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 2e-3
CACHE_BYTES = 5 << 30  # per cache tensor


@pytest.fixture(scope="module")
def pd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_split_decode_gb300 as pd
    pd.load()
    return pd


def big_pool(compact: torch.Tensor, dev_dtype=None):
    """A device cache of about CACHE_BYTES whose top blocks hold `compact`;
    returns (cache, index of the first of those blocks)."""
    per_block = compact[0].numel() * compact.element_size()
    nb = CACHE_BYTES // per_block + compact.shape[0]
    base = nb - compact.shape[0]
    assert base * per_block >= 4 << 30
    big = torch.empty((nb,) + tuple(compact.shape[1:]), dtype=compact.dtype, device=DEV)
    big[base:] = compact.to(DEV)
    return (big.view(dev_dtype) if dev_dtype is not None else big), base


@pytest.mark.parametrize("kv,qlen", [("f16", 1), ("int8", 3), ("fp8", 3)])
def test_decode_reads_blocks_past_4gib(pd, kv, qlen):
    w = inputs.make_workload(B=3, Hq=24, Hkv=4, D=256, qlen=qlen, seq_lens=[1000, 37, 2049], kv=kv,
                             seed=4100 + qlen, name=f"large_pool_{kv}")
    ref = oracle.decode_paged(w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(),
                              w.block_table.numpy(), w.seq_lens.numpy(), w.scale, w.window, w.qlen,
                              w.k_scale, w.v_scale, w.kv_fp8, kv_int8=w.kv_int8)
    dt = torch.int8 if kv == "int8" else None
    k, base = big_pool(w.k_cache, dt)
    v, _ = big_pool(w.v_cache, dt)
    table = torch.where(w.block_table >= 0, w.block_table + base, w.block_table).to(DEV)
    for S in (0, 1, 3):
        out = pd.decode_paged(w.q.to(DEV), k, v, table, w.seq_lens.to(DEV), w.scale, w.window, w.qlen,
                              S, k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - ref))) <= TOL, f"{kv} S={S}"
    del k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kind", ["f16", "fp8", "int8"])
def test_writer_stores_slots_past_4gib(pd, kind):
    Hkv, D, bs, T = 4, 256, 16, 300
    elem = 2 if kind == "f16" else 1
    nb = CACHE_BYTES // (bs * Hkv * D * elem)
    nslots = nb * bs
    g = torch.Generator().manual_seed(4200)
    k_new = torch.randn((T, Hkv, D), generator=g).half()
    v_new = torch.randn((T, Hkv, D), generator=g).half()
    lo = nslots - 4096  # the written slots lie in the last 4096; guard slots around them
    slots = (lo + torch.randperm(4096, generator=g)[:T]).to(torch.int64)
    assert lo * Hkv * D * elem >= 4 << 30
    k_scale, v_scale = (1.0, 1.0) if kind == "f16" else (1.0 / 64, 1.0 / 48)

    # oracle: the T tokens into a compact pool, token i at slot i
    nbc = -(-T // bs)
    shape_c = (nbc, bs, Hkv, D)
    if kind == "f16":
        ko = np.zeros(shape_c, dtype=np.float16)
    else:
        ko = np.zeros(shape_c, dtype=np.uint8)
    vo = ko.copy()
    assert oracle.write_kv_cache(k_new.numpy(), v_new.numpy(), np.arange(T, dtype=np.int64), ko, vo,
                                 k_scale=k_scale, v_scale=v_scale, kv_fp8=kind == "fp8",
                                 kv_int8=kind == "int8")
    want_k = ko.reshape(nbc * bs, Hkv, D)[:T].view(np.uint8)
    want_v = vo.reshape(nbc * bs, Hkv, D)[:T].view(np.uint8)

    dt = {"f16": torch.float16, "fp8": torch.uint8, "int8": torch.int8}[kind]
    caches = []
    for _ in range(2):
        c = torch.empty((nb, bs, Hkv, D), dtype=dt, device=DEV)
        c.view(torch.uint8).view(nslots, -1)[lo - 64:] = 0x5A  # sentinel over the written region
        caches.append(c)
    kc, vc = caches
    pd.write_kv_cache(k_new.to(DEV), v_new.to(DEV), slots.to(DEV), kc, vc, k_scale=k_scale,
                      v_scale=v_scale)
    torch.cuda.synchronize()
    for c, want in ((kc, want_k), (vc, want_v)):
        region = c.view(torch.uint8).view(nslots, -1)[lo - 64:].cpu().numpy()
        got = region[(slots - (lo - 64)).numpy()]
        assert np.array_equal(got, want.reshape(T, -1))
        untouched = np.ones(region.shape[0], dtype=bool)
        untouched[(slots - (lo - 64)).numpy()] = False
        assert np.all(region[untouched] == 0x5A)
    del kc, vc, caches
    torch.cuda.empty_cache()
