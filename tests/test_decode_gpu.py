"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs. Tolerance: max abs error <= 2e-3 on every element for
fp16 KV, and for fp8 KV against the oracle run on the identically decoded
codes; rows with no visible key must be exact zeros.

Workloads follow the decode benchmarks and cells of opengfx1030/vllm-rdna pull
request #33 ("Test Plan", results comment): the tiny two-sequence case, D=256
GQA 6:1 at L=4096 over the batch sweep, D=128 with ragged lengths and dense or
permuted tables, L=32768 with and without a 4096-key window across split
counts, and qlen=3 speculative verify over e4m3 KV.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from paged_split_decode_gb300 import inputs

TOL = 2e-3

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_split_decode_gb300 as pd
    pd.load()  # raises when the library is missing: no fallback
    return pd


DEV = "cuda:0"


def kv_on_device(w):
    k, v = w.k_cache.to(DEV), w.v_cache.to(DEV)
    if w.kv_int8:
        k, v = k.view(torch.int8), v.view(torch.int8)
    return k, v


def gpu_run(pd, w, num_splits=None, out=None, flag=None, workspace=None):
    S = w.num_splits if num_splits is None else num_splits
    k, v = kv_on_device(w)
    res = pd.decode_paged(w.q.to(DEV), k, v, w.block_table.to(DEV),
                          w.seq_lens.to(DEV), w.scale, w.window, w.qlen, S, out=out,
                          k_scale=w.k_scale, v_scale=w.v_scale, error_flag=flag, workspace=workspace)
    torch.cuda.synchronize()
    return res


def ref_run(w):
    return oracle.decode_paged(w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(),
                               w.block_table.numpy(), w.seq_lens.numpy(), w.scale, w.window, w.qlen,
                               w.k_scale, w.v_scale, w.kv_fp8, kv_int8=w.kv_int8)


def empty_rows(w):
    """[B*qlen*Hq] bool: rows whose query token sees no key."""
    rows = []
    for b, L in enumerate(w.seq_lens.tolist()):
        for i in range(w.qlen):
            rows += [L - w.qlen + i < 0 or L == 0] * w.Hq
    return np.array(rows)


def check(w, got, ref, tol=TOL):
    g = got.float().cpu().numpy().reshape(-1, w.D)
    r = ref.reshape(-1, w.D)
    assert np.all(np.isfinite(g)), f"{w.name}: non-finite output"
    err = float(np.max(np.abs(g - r))) if g.size else 0.0
    assert err <= tol, f"{w.name}: max abs err {err:.3e}"
    e = empty_rows(w)
    assert np.all(g[e] == 0.0), f"{w.name}: empty rows not zero"
    return err


def test_tiny_two_sequences_one_empty(pd):
    w = inputs.tiny()
    ref = ref_run(w)
    for S in (1, 0, 2, 5):
        check(w, gpu_run(pd, w, S), ref)


@pytest.mark.parametrize("B", [1, 2, 3, 8, 32])
def test_gqa6_d256_batch_sweep_balanced(pd, B):
    w = inputs.gqa_d256(B)
    check(w, gpu_run(pd, w), ref_run(w))


@pytest.mark.parametrize("heads", [(32, 8), (28, 4)])
@pytest.mark.parametrize("layout", ["dense", "permuted"])
def test_d128_ragged_lengths(pd, heads, layout):
    w = inputs.gqa_d128(heads, layout)
    check(w, gpu_run(pd, w), ref_run(w))


@pytest.mark.parametrize("B", [1, 2])
@pytest.mark.parametrize("window", [4096, 0])
def test_long_context_window_across_splits(pd, B, window):
    w = inputs.long_window(B, window, 0)
    ref = ref_run(w)
    outs = []
    for S in (1, 3, 8, 0):
        got = gpu_run(pd, w, S)
        check(w, got, ref)
        outs.append(got.float().cpu())
    for o in outs[1:]:
        assert torch.max(torch.abs(o - outs[0])).item() <= TOL


def test_speculative_verify_int8(pd):
    """The int8 decode wrapper: the verify shape over int8 KV codes."""
    w = inputs.make_workload(B=8, Hq=24, Hkv=4, D=256, qlen=3, seq_lens=[8192] * 8, kv="int8",
                             seed=1240, name="verify3_int8_d256_L8192_b8")
    ref = ref_run(w)
    for S in (0, 1, 4):
        check(w, gpu_run(pd, w, S), ref)


def test_speculative_verify_fp8(pd):
    w = inputs.verify_fp8()
    ref = ref_run(w)
    for S in (0, 1, 4):
        check(w, gpu_run(pd, w, S), ref)


EDGE = [
    # (name, kwargs)
    ("ragged_tail_and_short", dict(B=4, Hq=8, Hkv=2, D=128, seq_lens=[1, 15, 17, 333])),
    ("seq_shorter_than_qlen", dict(B=3, Hq=8, Hkv=2, D=128, qlen=3, seq_lens=[1, 2, 40])),
    ("all_empty", dict(B=3, Hq=8, Hkv=2, D=256, seq_lens=[0, 0, 0], pool_blocks=2)),
    ("window_one_key", dict(B=2, Hq=6, Hkv=1, D=256, seq_lens=[100, 16], window=1)),
    ("window_inside_a_tile", dict(B=2, Hq=4, Hkv=2, D=128, seq_lens=[97, 300], window=5, qlen=2)),
    ("mha_g1", dict(B=3, Hq=4, Hkv=4, D=128, seq_lens=[50, 700, 1])),
    ("rows_32", dict(B=2, Hq=8, Hkv=1, D=256, qlen=4, seq_lens=[600, 35])),
    ("rows_7", dict(B=5, Hq=28, Hkv=4, D=128, seq_lens=[10, 2000, 0, 64, 65])),
    ("block_size_32", dict(B=3, Hq=24, Hkv=4, D=256, block_size=32, seq_lens=[31, 33, 1000])),
    ("block_size_64_fp8", dict(B=2, Hq=16, Hkv=2, D=128, block_size=64, kv="fp8", qlen=2,
                               seq_lens=[129, 700])),
    ("fp8_d128_rows_24", dict(B=3, Hq=8, Hkv=1, D=128, kv="fp8", qlen=3, seq_lens=[5, 300, 1500])),
    ("fp8_d256_rows_6", dict(B=2, Hq=24, Hkv=4, D=256, kv="fp8", seq_lens=[4000, 17])),
    ("many_sequences", dict(B=300, Hq=8, Hkv=2, D=128, seq_lens=list(range(0, 3000, 10)))),
    # more sequences than the balanced split's shared-memory prefix holds
    # (1024): the automatic split falls back to one piece per unit
    ("beyond_balanced_split_batch", dict(B=1100, Hq=8, Hkv=2, D=128,
                                         seq_lens=[(17 * i) % 211 for i in range(1100)])),
    ("beyond_balanced_split_batch_fp8_verify", dict(B=1030, Hq=24, Hkv=4, D=256, kv="fp8", qlen=3,
                                                    seq_lens=[(13 * i) % 97 for i in range(1030)])),
    ("int8_d256_rows_6", dict(B=3, Hq=24, Hkv=4, D=256, kv="int8", seq_lens=[4000, 17, 0])),
    ("int8_d128_rows_24_window", dict(B=2, Hq=8, Hkv=1, D=128, kv="int8", qlen=3, window=300,
                                      seq_lens=[1500, 40])),
    ("int8_d256_rows_32", dict(B=2, Hq=8, Hkv=1, D=256, kv="int8", qlen=4, seq_lens=[700, 90])),
    # int8 with two and three row tiles per head (the latter windowed)
    ("int8_d256_rows_12", dict(B=3, Hq=12, Hkv=2, D=256, kv="int8", qlen=2, seq_lens=[5, 1000, 64])),
    ("int8_d256_rows_18_window", dict(B=3, Hq=24, Hkv=4, D=256, kv="int8", qlen=3, window=100,
                                      seq_lens=[2, 333, 1029])),
    # per-head tiles with two key groups over long rings (Hkv not a multiple of 4)
    ("fp8_d128_per_head_kg2", dict(B=4, Hq=16, Hkv=2, D=128, kv="fp8",
                                   seq_lens=[5000, 3001, 17, 4096])),
    ("int8_d128_per_head_kg2", dict(B=3, Hq=8, Hkv=1, D=128, kv="int8", seq_lens=[6000, 2500, 1])),
    ("f16_d256_per_head_kg2", dict(B=3, Hq=12, Hkv=2, D=256, seq_lens=[4100, 900, 33])),
    # head-group tiles with two head groups per sequence (Hkv = 8)
    ("fp8_d128_two_head_groups", dict(B=3, Hq=32, Hkv=8, D=128, kv="fp8", seq_lens=[3000, 47, 800])),
    ("f16_d256_two_head_groups", dict(B=2, Hq=16, Hkv=8, D=256, seq_lens=[2049, 700])),
    # e4m3 units of 9..32 rows run on the tensor-memory kernel: 128-key blocks,
    # partial blocks at piece ends, windows across blocks, block sizes > 16
    ("fp8_d256_rows_32_window", dict(B=3, Hq=8, Hkv=1, D=256, kv="fp8", qlen=4, window=200,
                                     seq_lens=[1000, 129, 3])),
    ("fp8_d256_rows_16_bs64", dict(B=2, Hq=16, Hkv=2, D=256, kv="fp8", qlen=2, block_size=64,
                                   seq_lens=[2000, 65])),
    ("fp8_d128_rows_9_block_edges", dict(B=4, Hq=9, Hkv=1, D=128, kv="fp8",
                                         seq_lens=[1, 128, 129, 5000])),
]


@pytest.mark.parametrize("S", [0, 1, 3, 17])
@pytest.mark.parametrize("name,kw", EDGE, ids=[e[0] for e in EDGE])
def test_edge_cases(pd, name, kw, S):
    w = inputs.make_workload(seed=zlib.crc32(name.encode()) % 10000, name=name, **kw)
    check(w, gpu_run(pd, w, S), ref_run(w))


# Automatic plans with few units on large block tables (the balanced cut over
# every CTA, several pieces per unit): equal lengths, equal tile counts with
# unequal lengths, one longer sequence, windows, byte caches and two row tiles
# per head (a bfloat16 cache: test_bf16_gpu.py).
FEW_UNITS = [
    ("f16_d256_gqa6_b8", dict(B=8, Hq=24, Hkv=4, D=256, seq_lens=[1000] * 8, max_blocks_per_seq=512)),
    ("f16_d256_equal_tiles_unequal_lens", dict(B=8, Hq=24, Hkv=4, D=256, seq_lens=[1000] * 7 + [993],
                                               max_blocks_per_seq=512)),
    ("f16_d256_one_longer", dict(B=8, Hq=24, Hkv=4, D=256, seq_lens=[1000] * 7 + [1100],
                                 max_blocks_per_seq=512)),
    ("fp8_d256_gqa6_b16", dict(B=16, Hq=24, Hkv=4, D=256, kv="fp8", seq_lens=[600] * 16,
                               max_blocks_per_seq=512)),
    ("int8_d128_b8_window", dict(B=8, Hq=32, Hkv=8, D=128, kv="int8", window=4000, seq_lens=[6000] * 8,
                                 max_blocks_per_seq=512)),
    ("fp8_d256_gqa6_b32", dict(B=32, Hq=24, Hkv=4, D=256, kv="fp8", seq_lens=[600] * 32,
                               max_blocks_per_seq=256)),
    ("f16_d256_b2_long", dict(B=2, Hq=24, Hkv=4, D=256, seq_lens=[9000, 9000], max_blocks_per_seq=1024)),
    ("f16_d256_qlen2_b4", dict(B=4, Hq=24, Hkv=4, D=256, qlen=2, seq_lens=[3000] * 4, max_blocks_per_seq=512)),
]


@pytest.mark.parametrize("name,kw", FEW_UNITS, ids=[e[0] for e in FEW_UNITS])
def test_few_units_on_large_tables(pd, name, kw):
    w = inputs.make_workload(seed=zlib.crc32(name.encode()) % 10000 + 11, name=name, **kw)
    check(w, gpu_run(pd, w, 0), ref_run(w))


STALE = [
    ("f16_rows_6", dict(B=4, Hq=24, Hkv=4, D=256, seq_lens=[1, 17, 4001, 250])),
    ("f16_rows_18_window", dict(B=3, Hq=24, Hkv=4, D=256, qlen=3, window=100,
                                seq_lens=[2, 333, 1029])),
    ("f16_d128_rows_8", dict(B=3, Hq=32, Hkv=8, D=128, seq_lens=[7, 90, 700])),
    ("fp8_rows_6", dict(B=3, Hq=24, Hkv=4, D=256, kv="fp8", seq_lens=[3, 4001, 250])),
    ("fp8_d128_rows_24", dict(B=2, Hq=8, Hkv=1, D=128, kv="fp8", qlen=3, seq_lens=[5, 301])),
    ("fp8_d256_rows_18", dict(B=3, Hq=24, Hkv=4, D=256, kv="fp8", qlen=3, seq_lens=[3, 4001, 250])),
    ("int8_rows_32", dict(B=2, Hq=8, Hkv=1, D=256, kv="int8", qlen=4, seq_lens=[700, 91])),
    ("int8_rows_18", dict(B=3, Hq=24, Hkv=4, D=256, kv="int8", qlen=3, seq_lens=[3, 4001, 250])),
]


@pytest.mark.parametrize("S", [0, 1, 5])
@pytest.mark.parametrize("name,kw", STALE, ids=[e[0] for e in STALE])
def test_stale_block_tail_is_never_read(pd, name, kw, S):
    """The slots past each sequence's last key in its last block hold NaN
    patterns (the unwritten tail of a block may hold anything): the output
    must equal the oracle, which never reads them."""
    w = inputs.make_workload(seed=zlib.crc32(name.encode()) % 10000 + 7, name=name, stale="nan",
                             **kw)
    check(w, gpu_run(pd, w, S), ref_run(w))


def test_one_workspace_across_changing_shapes(pd):
    """One workspace buffer serves calls of different shapes back to back: every
    call writes the partials it reads."""
    import paged_split_decode_gb300 as P
    ws = torch.full((64 << 20,), 0xA5, dtype=torch.uint8, device=DEV)  # garbage start
    ws_list = [inputs.make_workload(B=2, Hq=8, Hkv=8, D=128, seq_lens=[5000, 16384], seed=21),
               inputs.make_workload(B=32, Hq=32, Hkv=8, D=128, seq_lens=[4096] * 32, seed=22),
               inputs.make_workload(B=3, Hq=24, Hkv=4, D=256, seq_lens=[9000, 1, 700], seed=23,
                                    qlen=3, kv="fp8"),
               inputs.make_workload(B=32, Hq=32, Hkv=8, D=256, seq_lens=[8192] * 32, seed=24)]
    refs = [ref_run(w) for w in ws_list]
    for rep in range(2):
        for w, r in zip(ws_list, refs):
            for S in (0, 3):
                check(w, gpu_run(pd, w, S, workspace=ws), r)


@pytest.mark.parametrize("S", [0, 9, 64, 100, 500])
def test_split_tree_with_many_pieces(pd, S):
    """One KV head, one long sequence: the balanced split cuts it into one piece
    per CTA (hundreds), a fixed split into S pieces; the combine tree (fan-out
    8) then has up to three levels."""
    w = inputs.make_workload(B=1, Hq=8, Hkv=1, D=128, seq_lens=[20000], seed=41, qlen=2)
    check(w, gpu_run(pd, w, S), ref_run(w))


@pytest.mark.parametrize("S", [0, 1, 3])
def test_cuda_graph_capture_and_replay(pd, S):
    """A call captured once into a CUDA graph (no host sync, no allocation, the
    split plan fixed by host-known shapes) replays correctly after new values
    are written into the same input buffers."""
    shape = dict(B=4, Hq=24, Hkv=4, D=256, pool_blocks=600, max_blocks_per_seq=256)
    w1 = inputs.make_workload(seq_lens=[3000, 17, 900, 0], seed=51, **shape)
    w2 = inputs.make_workload(seq_lens=[2999, 1, 4000, 64], seed=52, **shape)
    q, bt, sl = w1.q.to(DEV), w1.block_table.to(DEV), w1.seq_lens.to(DEV)
    k, v = kv_on_device(w1)
    out = torch.empty_like(q)
    dims = pd.dims_of(q, k, bt, 1)
    ws = torch.empty(max(pd.workspace_bytes(dims, 1, S), 1), dtype=torch.uint8, device=DEV)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        pd.decode_paged(q, k, v, bt, sl, w1.scale, 0, 1, S, out=out, workspace=ws)  # warm up
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        pd.decode_paged(q, k, v, bt, sl, w1.scale, 0, 1, S, out=out, workspace=ws)
    for w in (w1, w2):
        q.copy_(w.q.to(DEV)); bt.copy_(w.block_table.to(DEV)); sl.copy_(w.seq_lens.to(DEV))
        k2, v2 = kv_on_device(w)
        k.copy_(k2); v.copy_(v2)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        check(w, out, ref_run(w))


def test_custom_scale_writes_into_out_only(pd):
    """A caller-owned out is written in full; bytes around it are untouched."""
    w = inputs.make_workload(B=2, Hq=24, Hkv=4, D=256, seq_lens=[1000, 0], seed=5, scale=0.37)
    n = w.q.numel()
    buf = torch.full((n + 2 * 4096,), 7.0, dtype=torch.float16, device=DEV)
    out = buf[4096:4096 + n].view_as(w.q)
    gpu_run(pd, w, 0, out=out)
    check(w, out, ref_run(w))
    assert torch.all(buf[:4096] == 7.0) and torch.all(buf[4096 + n:] == 7.0)


def test_scale_zero_is_mean_of_v(pd):
    w = inputs.make_workload(B=2, Hq=8, Hkv=2, D=128, seq_lens=[333, 64], seed=6, scale=0.0)
    check(w, gpu_run(pd, w), ref_run(w))


def test_writer_layout_per_head_constants(pd):
    """V rows hold a constant per (KV head, dim): every query head must return
    the constant of the KV head h // G (the cache layout and GQA mapping)."""
    w = inputs.make_workload(B=3, Hq=24, Hkv=4, D=256, seq_lens=[77, 1000, 16], seed=8)
    c = torch.arange(4, dtype=torch.float32)[:, None] * 0.5 - 1 + torch.linspace(0, 0.25, 256)[None]
    w.v_cache[:] = c.to(torch.float16)[None, None]
    got = gpu_run(pd, w).float().cpu()
    for h in range(24):
        assert torch.max(torch.abs(got[:, h] - c.to(torch.float16).float()[h // 6])).item() <= 1e-3


def test_block_permutation_invariance_and_determinism(pd):
    w = inputs.gqa_d256(2)
    a = gpu_run(pd, w).clone()
    b = gpu_run(pd, w).clone()
    assert torch.equal(a, b), "same inputs, same workspace: results must be bitwise equal"
    pool = w.k_cache.shape[0]
    perm = torch.randperm(pool, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(pool)
    w2 = inputs.Workload(**{**w.__dict__})
    w2.k_cache = w.k_cache[perm].contiguous()
    w2.v_cache = w.v_cache[perm].contiguous()
    t = w.block_table.clone()
    ok = t >= 0
    t[ok] = inv[t[ok].long()].to(torch.int32)
    w2.block_table = t
    c = gpu_run(pd, w2)
    assert torch.equal(a, c), "a physical block permutation must not change the result"


def test_tensor_memory_kernel_determinism_and_permutation(pd):
    """The e4m3 units of 9..32 rows (tcgen05 kernel): run twice bitwise equal,
    and unchanged by a physical permutation of the cache blocks."""
    w = inputs.make_workload(B=3, Hq=24, Hkv=4, D=256, qlen=3, kv="fp8", seq_lens=[3000, 777, 40], seed=61,
                             name="tc8_det")
    for S in (0, 5):
        a = gpu_run(pd, w, S).clone()
        b = gpu_run(pd, w, S).clone()
        assert torch.equal(a, b), "same inputs, same workspace: results must be bitwise equal"
        pool = w.k_cache.shape[0]
        perm = torch.randperm(pool, generator=torch.Generator().manual_seed(4))
        inv = torch.empty_like(perm)
        inv[perm] = torch.arange(pool)
        w2 = inputs.Workload(**{**w.__dict__})
        w2.k_cache = w.k_cache[perm].contiguous()
        w2.v_cache = w.v_cache[perm].contiguous()
        t = w.block_table.clone()
        ok = t >= 0
        t[ok] = inv[t[ok].long()].to(torch.int32)
        w2.block_table = t
        assert torch.equal(a, gpu_run(pd, w2, S)), "a physical block permutation must not change the result"
        check(w, a, ref_run(w))


@pytest.mark.parametrize("S", [0, 3])
def test_tensor_memory_kernel_graph_replay(pd, S):
    """The tcgen05 e4m3 kernel captured once into a CUDA graph replays
    correctly on new inputs written into the same buffers."""
    shape = dict(B=3, Hq=16, Hkv=2, D=128, qlen=2, kv="fp8", pool_blocks=700, max_blocks_per_seq=300)
    w1 = inputs.make_workload(seq_lens=[4000, 33, 1500], seed=71, **shape)
    w2 = inputs.make_workload(seq_lens=[129, 4700, 0], seed=72, **shape)
    q, bt, sl = w1.q.to(DEV), w1.block_table.to(DEV), w1.seq_lens.to(DEV)
    k, v = kv_on_device(w1)
    out = torch.empty_like(q)
    dims = pd.dims_of(q, k, bt, 2, None)
    ws = torch.empty(max(pd.workspace_bytes(dims, 2, S), 1), dtype=torch.uint8, device=DEV)
    kw = dict(k_scale=w1.k_scale, v_scale=w1.v_scale, out=out, workspace=ws)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        pd.decode_paged(q, k, v, bt, sl, w1.scale, 0, 2, S, **kw)  # warm up
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        pd.decode_paged(q, k, v, bt, sl, w1.scale, 0, 2, S, **kw)
    for w in (w1, w2):
        # the scales are arguments of the captured call (w1's): the codes of w2
        # are read with them, and the reference does the same
        q.copy_(w.q.to(DEV)); bt.copy_(w.block_table.to(DEV)); sl.copy_(w.seq_lens.to(DEV))
        k2, v2 = kv_on_device(w)
        k.copy_(k2); v.copy_(v2)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        wref = inputs.Workload(**{**w.__dict__})
        wref.k_scale, wref.v_scale = w1.k_scale, w1.v_scale
        check(w, out, ref_run(wref))


def test_tensor_memory_kernel_long_pieces(pd):
    """Long sequences through the tcgen05 kernel: many 128-key blocks per
    piece, windows that start inside blocks, a sequence shorter than qlen."""
    w = inputs.make_workload(B=3, Hq=12, Hkv=1, D=256, qlen=2, kv="fp8", window=5000,
                             seq_lens=[20000, 1, 7777], seed=81, name="tc8_long")
    ref = ref_run(w)
    for S in (0, 1, 2, 9):
        check(w, gpu_run(pd, w, S), ref)


def test_device_errors_are_flagged_not_trapped(pd):
    w = inputs.make_workload(B=2, Hq=8, Hkv=2, D=128, seq_lens=[100, 50], seed=9)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    bad = inputs.Workload(**{**w.__dict__})
    bad.block_table = w.block_table.clone()
    bad.block_table[0, 2] = 1 << 20            # outside the pool
    gpu_run(pd, bad, 0, flag=flag)
    assert int(flag.item()) & 1
    flag.zero_()
    bad2 = inputs.Workload(**{**w.__dict__})
    bad2.seq_lens = torch.tensor([100, 10_000], dtype=torch.int32)  # above the table's capacity
    gpu_run(pd, bad2, 1, flag=flag)
    assert int(flag.item()) & 2
    flag.zero_()
    out = gpu_run(pd, w, 0, flag=flag)          # the context is still healthy
    assert int(flag.item()) == 0
    check(w, out, ref_run(w))


@pytest.mark.parametrize("shape", [dict(B=4, Hq=24, Hkv=4, D=256, qlen=1),
                                   dict(B=3, Hq=24, Hkv=4, D=256, qlen=3, kv="fp8"),
                                   dict(B=3, Hq=24, Hkv=4, D=256, qlen=3, kv="int8")],
                         ids=["rows_6", "rows_18_pairs", "rows_18_int8"])
def test_wait_that_nothing_completes_times_out_cleanly(pd, shape):
    """Failure detection without a GPU fault: with loads suppressed the ring's
    barriers never complete, every wait runs out after a short limit, the call
    sets PD_DEVERR_TIMEOUT and returns; the next normal call is correct."""
    from paged_split_decode_gb300 import binding
    w = inputs.make_workload(seq_lens=[700, 3000, 16, 0][:shape["B"]], seed=61, **shape)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.set_wait_limit_ns(20_000_000)   # 20 ms
    binding.set_fault_injection(1)
    try:
        gpu_run(pd, w, 0, flag=flag)
    finally:
        binding.set_fault_injection(0)
        binding.set_wait_limit_ns(0)
    assert int(flag.item()) & 4, "the timeout bit must be set"
    flag.zero_()
    check(w, gpu_run(pd, w, 0, flag=flag), ref_run(w))
    assert int(flag.item()) == 0


def test_combine_entry_point_matches_oracle(pd):
    w = inputs.make_workload(B=3, Hq=8, Hkv=2, D=128, seq_lens=[500, 0, 77], qlen=2, seed=10)
    _, m, l, O = oracle.decode_paged_split(w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(),
                                           w.block_table.numpy(), w.seq_lens.numpy(), w.scale,
                                           num_splits=5, qlen=w.qlen, return_partials=True)
    want = oracle.combine(m, l, O)
    mt = torch.tensor(m, dtype=torch.float32, device=DEV)
    lt = torch.tensor(l, dtype=torch.float32, device=DEV)
    Ot = torch.tensor(O, dtype=torch.float32, device=DEV)
    got = pd.decode_paged_combine(mt, lt, Ot)
    torch.cuda.synchronize()
    g = got.float().cpu().numpy()
    assert np.max(np.abs(g - want)) <= TOL
    assert np.all(g[np.all(want == 0, axis=1)] == 0)


def test_default_workspace_is_per_stream(pd):
    """Decodes on two streams with no workspace argument each get their own
    default buffer (their split partials would race in a shared one): every
    result matches the oracle."""
    ws = [inputs.gqa_d256(2),
          inputs.make_workload(B=2, Hq=24, Hkv=4, D=256, qlen=1, seq_lens=[4096, 3000], seed=77)]
    refs = [ref_run(w) for w in ws]
    dev_in = []
    for w in ws:
        k, v = kv_on_device(w)
        dev_in.append((w.q.to(DEV), k, v, w.block_table.to(DEV), w.seq_lens.to(DEV)))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in ws]
    outs = []
    for _ in range(4):  # back to back, so that the two streams' calls overlap
        for w, s, (q, k, v, bt, sl) in zip(ws, streams, dev_in):
            with torch.cuda.stream(s):
                outs.append((w, pd.decode_paged(q, k, v, bt, sl, w.scale, w.window, w.qlen, 0,
                                                k_scale=w.k_scale, v_scale=w.v_scale)))
    torch.cuda.synchronize()
    for w, got in outs:
        check(w, got, refs[ws.index(w)])


# Fixed splits of two to eight pieces on the tensor-memory kernels (e4m3 and
# int8 KV, 9-32 query rows per KV head): a unit's pieces run as one thread-block
# cluster and merge through distributed shared memory, with no split-combine
# launch. Sequences with fewer tiles than pieces leave CTAs of a cluster
# without a piece; empty sequences and tokens that see no key are zero rows.
CLUSTER = [
    ("rows18_d256", dict(B=4, Hq=24, Hkv=4, D=256, qlen=3, kv="fp8", seq_lens=[3000, 40, 0, 2])),
    ("rows16_d128", dict(B=3, Hq=16, Hkv=2, D=128, qlen=2, kv="fp8", seq_lens=[900, 17, 2500])),
    ("rows32_d256_window", dict(B=2, Hq=8, Hkv=1, D=256, qlen=4, kv="fp8", window=300,
                                seq_lens=[2000, 33])),
    ("rows24_d128_stale", dict(B=3, Hq=8, Hkv=1, D=128, qlen=3, kv="fp8", seq_lens=[5, 301, 4000],
                               stale="nan")),
    ("rows18_d256_int8", dict(B=4, Hq=24, Hkv=4, D=256, qlen=3, kv="int8", seq_lens=[3000, 40, 0, 2])),
    ("rows12_d128_int8_window", dict(B=3, Hq=8, Hkv=2, D=128, qlen=3, kv="int8", window=500,
                                     seq_lens=[2000, 33, 700])),
]


@pytest.mark.parametrize("S", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("name,kw", CLUSTER, ids=[c[0] for c in CLUSTER])
def test_tensor_memory_kernel_cluster_merge(pd, name, kw, S):
    w = inputs.make_workload(seed=zlib.crc32(name.encode()) % 10000 + 3, name=name, **kw)
    check(w, gpu_run(pd, w, S), ref_run(w))


# Fixed splits of 9 to 16 pieces on the mma.sync kernels: clusters beyond the
# portable eight CTAs (the merge reads each unit's partials back from L2 after
# one cluster barrier); units with fewer tiles than pieces, empty sequences,
# windows and a bfloat16 cache included.
WIDE_CLUSTER = [
    ("f16_d256_gqa6", dict(B=3, Hq=24, Hkv=4, D=256, seq_lens=[4096, 70, 0])),
    ("f16_d128_gqa4_window", dict(B=2, Hq=32, Hkv=8, D=128, window=900, seq_lens=[3000, 2200])),
    ("fp8_d256_gqa6", dict(B=2, Hq=24, Hkv=4, D=256, kv="fp8", seq_lens=[5000, 33])),
    ("int8_d256_q3", dict(B=2, Hq=24, Hkv=4, D=256, kv="int8", qlen=3, seq_lens=[2500, 3])),
]


@pytest.mark.parametrize("S", [9, 12, 16])
@pytest.mark.parametrize("name,kw", WIDE_CLUSTER, ids=[c[0] for c in WIDE_CLUSTER])
def test_wide_cluster_merge(pd, name, kw, S):
    w = inputs.make_workload(seed=zlib.crc32(name.encode()) % 10000 + 5, name=name, **kw)
    check(w, gpu_run(pd, w, S), ref_run(w))
