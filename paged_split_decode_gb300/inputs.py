"""Seeded synthetic inputs for paged decode attention.

This module only draws numbers and lays them out; it holds none of the
attention arithmetic, so the CUDA path and the fp64 oracle can both consume
its output. Everything is drawn on the CPU from a seeded ``torch.Generator``
and returned as CPU tensors.

Recipe (shapes follow the benchmark commands of opengfx1030/vllm-rdna pull
request #33, "Test Plan" step 3, and the geometry of its results comment):

* Q, K, V values are i.i.d. N(0, 1) drawn in fp32 and rounded to fp16 (or,
  for the bfloat16 kind, to bfloat16 -- q and both caches).
* fp8 KV: the N(0, 1) fp32 draw is divided by one per-cache scale
  ``amax / 448`` (448 is the largest finite e4m3fn value), clamped to
  [-448, 448] and rounded to e4m3fn by torch's CPU cast; the cache holds the
  code bytes and the scale is returned beside it.
* int8 KV: the same draw divided by ``amax / 127``, rounded half to even,
  clamped to [-127, 127]; the cache holds the two's-complement code bytes.
* Block tables: ``permuted`` draws a random permutation of the physical block
  pool and hands each sequence a slice of it; ``dense`` gives sequence b the
  contiguous run of blocks after sequence b-1's. Table entries past a
  sequence's last block are -1, so reading one is an error the kernel reports.
* Every slot of every pool block holds a drawn value, including the slots
  after a sequence's last key (the stale tail of a partly filled block);
  optionally that tail holds NaN patterns instead.
* KV-cache writer inputs: new K/V rows N(0, sigma) in fp16 for T tokens, a
  slot per token drawn without repetition from the cache's slots (a random
  permutation), every ``pad_every``-th token a padding token (slot -1), and
  optionally a sprinkle of special fp16 values (zeros of both signs,
  infinities, NaN, the largest finite and subnormal values).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BLOCK_SIZE = 16
E4M3_MAX = 448.0


@dataclass
class Workload:
    name: str
    q: torch.Tensor            # fp16 [B*qlen, Hq, D]
    k_cache: torch.Tensor      # fp16 or uint8 (e4m3fn codes) [num_blocks, bs, Hkv, D]
    v_cache: torch.Tensor
    block_table: torch.Tensor  # int32 [B, max_blocks_per_seq]
    seq_lens: torch.Tensor     # int32 [B]
    scale: float
    window: int = 0
    qlen: int = 1
    num_splits: int = 0
    kv_fp8: bool = False
    kv_int8: bool = False
    bf16: bool = False         # q and the output in bfloat16 (the caches too, unless byte codes)
    k_scale: float = 1.0
    v_scale: float = 1.0
    meta: dict = field(default_factory=dict)
    # per-sequence query counts: sequence b owns rows q_start[b]..q_start[b+1]-1
    # of q (int32 [B+1]); None = qlen rows each. qlen is then the largest count.
    q_start: torch.Tensor | None = None

    @property
    def B(self):
        return int(self.seq_lens.shape[0])

    @property
    def Hq(self):
        return int(self.q.shape[1])

    @property
    def Hkv(self):
        return int(self.k_cache.shape[2])

    @property
    def D(self):
        return int(self.q.shape[2])

    @property
    def block_size(self):
        return int(self.k_cache.shape[1])


def _normal(gen, shape):
    return torch.randn(*shape, generator=gen, dtype=torch.float32)


def _fp8_quantise(x: torch.Tensor):
    amax = float(x.abs().max()) if x.numel() else 1.0
    scale = torch.tensor(amax / E4M3_MAX if amax > 0 else 1.0, dtype=torch.float32)
    codes = (x / scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, float(scale)


def _int8_quantise(x: torch.Tensor):
    amax = float(x.abs().max()) if x.numel() else 1.0
    scale = torch.tensor(amax / 127.0 if amax > 0 else 1.0, dtype=torch.float32)
    codes = torch.round(x / scale).clamp(-127, 127).to(torch.int8).view(torch.uint8)
    return codes, float(scale)


def blocks_needed(seq_len: int, block_size: int = BLOCK_SIZE) -> int:
    return (int(seq_len) + block_size - 1) // block_size


def make_block_table(gen, seq_lens, max_blocks_per_seq, layout="permuted", pool_blocks=None,
                     block_size=BLOCK_SIZE, first_block=0):
    """Block table [B, max_blocks] over a pool; returns (table, pool_blocks)."""
    need = [blocks_needed(L, block_size) for L in seq_lens]
    total = sum(need)
    pool = pool_blocks if pool_blocks is not None else first_block + total
    if pool - first_block < total:
        raise ValueError("pool too small")
    table = torch.full((len(seq_lens), max_blocks_per_seq), -1, dtype=torch.int32)
    if layout == "permuted":
        ids = torch.randperm(pool - first_block, generator=gen)[:total].to(torch.int32) + first_block
    elif layout == "dense":
        ids = torch.arange(first_block, first_block + total, dtype=torch.int32)
    else:
        raise ValueError(layout)
    off = 0
    for b, n in enumerate(need):
        if n > max_blocks_per_seq:
            raise ValueError("sequence longer than the table")
        table[b, :n] = ids[off:off + n]
        off += n
    return table, pool


def make_workload(*, B, Hq, Hkv, D, seq_lens, qlen=1, block_size=BLOCK_SIZE, layout="permuted",
                  window=0, kv="f16", seed=0, scale=None, num_splits=0, max_blocks_per_seq=None,
                  pool_blocks=None, name="custom", stale="drawn") -> Workload:
    """``kv``: "f16", "bf16", "fp8", "int8", or "fp8_bf16q" / "int8_bf16q"
    (byte caches under a bfloat16 q). ``stale="nan"`` overwrites, in each
    sequence's last block, the slots past its last key with NaN bit patterns
    (the unwritten tail of a block may hold anything); int8 codes have no NaN,
    so they get -128 there."""
    kv_name = kv
    bq = kv in ("bf16", "fp8_bf16q", "int8_bf16q")
    kv = {"fp8_bf16q": "fp8", "int8_bf16q": "int8"}.get(kv, kv)
    gen = torch.Generator().manual_seed(int(seed))
    seq_lens = [int(x) for x in seq_lens]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max([blocks_needed(L, block_size) for L in seq_lens] + [1])
    table, pool = make_block_table(gen, seq_lens, max_blocks_per_seq, layout, pool_blocks, block_size)
    qf = _normal(gen, (B * qlen, Hq, D))
    q = qf.to(torch.bfloat16) if bq else qf.to(torch.float16)
    kf = _normal(gen, (pool, block_size, Hkv, D))
    vf = _normal(gen, (pool, block_size, Hkv, D))
    kv_fp8 = kv_int8 = False
    if kv == "fp8":
        k_cache, k_scale = _fp8_quantise(kf)
        v_cache, v_scale = _fp8_quantise(vf)
        kv_fp8 = True
    elif kv == "int8":
        k_cache, k_scale = _int8_quantise(kf)
        v_cache, v_scale = _int8_quantise(vf)
        kv_int8 = True
    elif kv == "f16":
        k_cache, v_cache = kf.to(torch.float16), vf.to(torch.float16)
        k_scale = v_scale = 1.0
    elif kv == "bf16":
        k_cache, v_cache = kf.to(torch.bfloat16), vf.to(torch.bfloat16)
        k_scale = v_scale = 1.0
    else:
        raise ValueError(kv)
    if stale == "nan":
        for b, L in enumerate(seq_lens):
            if L % block_size == 0 or L == 0:
                continue
            blk = int(table[b, (L - 1) // block_size])
            for c in (k_cache, v_cache):
                if c.dtype == torch.float16:
                    c.view(torch.int16)[blk, L % block_size:] = 0x7E00
                elif c.dtype == torch.bfloat16:
                    c.view(torch.int16)[blk, L % block_size:] = 0x7FC0
                elif kv == "fp8":
                    c[blk, L % block_size:] = 0x7F
                else:
                    c[blk, L % block_size:] = 0x80
    elif stale != "drawn":
        raise ValueError(stale)
    return Workload(name=name, q=q, k_cache=k_cache, v_cache=v_cache, block_table=table,
                    seq_lens=torch.tensor(seq_lens, dtype=torch.int32),
                    scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
                    window=int(window), qlen=int(qlen), num_splits=int(num_splits), kv_fp8=kv_fp8,
                    kv_int8=kv_int8, bf16=bq,
                    k_scale=k_scale, v_scale=v_scale,
                    meta=dict(layout=layout, seed=int(seed), kv=kv_name))


def make_varlen_workload(*, qlens, seed=0, name="varlen", **kw) -> Workload:
    """A batch whose sequences carry different numbers of query tokens: the
    caches and tables as make_workload draws them, Q redrawn as
    [sum(qlens), Hq, D] with sequence b owning the rows after sequence b-1's."""
    qlens = [int(x) for x in qlens]
    w = make_workload(seed=seed, name=name, qlen=1, **kw)
    assert len(qlens) == w.B
    gen = torch.Generator().manual_seed(int(seed) + 7919)
    starts = [0]
    for n in qlens:
        starts.append(starts[-1] + n)
    w.q = _normal(gen, (starts[-1], w.Hq, w.D)).to(torch.bfloat16 if w.bf16 else torch.float16)
    w.q_start = torch.tensor(starts, dtype=torch.int32)
    w.qlen = max(qlens + [1])
    w.meta["qlens"] = qlens
    return w


# ---- the five named workloads ------------------------------------------------

def tiny(seed=1235) -> Workload:
    """B=2, Hq=8, Hkv=2, D=128, seq_lens {100, 0}, a 16-block permuted pool, S=1."""
    return make_workload(B=2, Hq=8, Hkv=2, D=128, seq_lens=[100, 0], layout="permuted",
                         pool_blocks=16, max_blocks_per_seq=8, seed=seed, num_splits=1,
                         name="tiny_d128_b2")


def gqa_d256(B, seed=None, seq_len=4096, layout="permuted", num_splits=0) -> Workload:
    """Hq=24, Hkv=4 (6:1), D=256, qlen=1, L=4096 for every row, permuted table."""
    seed = 1236 * 1000 + B if seed is None else seed
    return make_workload(B=B, Hq=24, Hkv=4, D=256, seq_lens=[seq_len] * B, layout=layout,
                         seed=seed, num_splits=num_splits, name=f"gqa6_d256_L{seq_len}_b{B}")


def gqa_d128(heads=(32, 8), layout="dense", B=32, seed=None, lo=512, hi=16384) -> Workload:
    """D=128, B=32, seq_lens uniform integers in [512, 16384], dense or permuted table."""
    Hq, Hkv = heads
    seed = (1237 * 1000 + Hq * 10 + Hkv) * 2 + (layout == "permuted") if seed is None else seed
    gen = torch.Generator().manual_seed(seed)
    lens = torch.randint(lo, hi + 1, (B,), generator=gen).tolist()
    return make_workload(B=B, Hq=Hq, Hkv=Hkv, D=128, seq_lens=lens, layout=layout, seed=seed + 1,
                         max_blocks_per_seq=1024, name=f"gqa{Hq // Hkv}_d128_{layout}_b{B}")


def long_window(B, window, num_splits, seed=None, seq_len=32768) -> Workload:
    """Hq=24, Hkv=4, D=256, L=32768, window 4096 or none, a fixed split count."""
    seed = 1238 * 1000 + B if seed is None else seed
    return make_workload(B=B, Hq=24, Hkv=4, D=256, seq_lens=[seq_len] * B, window=window,
                         seed=seed, num_splits=num_splits,
                         name=f"long_d256_L{seq_len}_b{B}_w{window}_s{num_splits}")


def verify_fp8(B=8, seed=1239, seq_len=8192) -> Workload:
    """B=8, Hq=24, Hkv=4, D=256, qlen=3 causal, L=8192, e4m3fn KV with per-cache scales."""
    return make_workload(B=B, Hq=24, Hkv=4, D=256, seq_lens=[seq_len] * B, qlen=3, kv="fp8",
                         seed=seed, name=f"verify3_fp8_d256_L{seq_len}_b{B}")


@dataclass
class WriterInputs:
    k_new: torch.Tensor        # fp16 [T, Hkv, D]
    v_new: torch.Tensor        # fp16 [T, Hkv, D]
    slot_mapping: torch.Tensor  # int64 [T]; -1 = padding token
    num_blocks: int
    block_size: int


_SPECIAL_F16 = (0x0000, 0x8000, 0x7C00, 0xFC00, 0x7E00, 0x7BFF, 0xFBFF, 0x0001, 0x8001, 0x03FF,
                0x0400, 0x3C00, 0xBC00)


def make_writer_inputs(T, Hkv, D, num_blocks, block_size=BLOCK_SIZE, seed=0, sigma=1.0,
                       pad_every=0, specials=False) -> WriterInputs:
    """New tokens for the paged KV-cache writer (see the module recipe)."""
    g = torch.Generator().manual_seed(seed)
    k = (torch.randn((T, Hkv, D), generator=g) * sigma).half()
    v = (torch.randn((T, Hkv, D), generator=g) * sigma).half()
    if specials and T > 0:
        sp = torch.tensor(_SPECIAL_F16, dtype=torch.int32).to(torch.int16).view(torch.float16)
        for x in (k, v):
            flat = x.view(-1)
            idx = torch.randint(0, flat.numel(), (4 * len(_SPECIAL_F16),), generator=g)
            flat[idx] = sp.repeat(4)
    slots = torch.randperm(num_blocks * block_size, generator=g)[:T].to(torch.int64)
    assert slots.numel() == T, "more tokens than cache slots"
    if pad_every > 0:
        slots[::pad_every] = -1
    return WriterInputs(k, v, slots, num_blocks, block_size)


def all_f16_patterns(Hkv=1, D=256) -> torch.Tensor:
    """Every fp16 bit pattern once, as [65536 / (Hkv*D), Hkv, D] fp16."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    return bits.view(torch.float16).reshape(-1, Hkv, D).clone()
