"""Seeded synthetic inputs for paged decode attention.

This module only draws numbers and lays them out; it holds none of the
attention arithmetic, so the CUDA path and the fp64 oracle can both consume
its output. Everything is drawn on the CPU from a seeded ``torch.Generator``
and returned as CPU tensors.

Recipe (shapes follow the benchmark commands of opengfx1030/vllm-rdna pull
request #33, "Test Plan" step 3, and the geometry of its results comment):

* Q, K, V values are i.i.d. N(0, 1) drawn in fp32 and rounded to fp16.
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
  after a sequence's last key (the stale tail of a partly filled block).
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
    k_scale: float = 1.0
    v_scale: float = 1.0
    meta: dict = field(default_factory=dict)

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
                  pool_blocks=None, name="custom") -> Workload:
    gen = torch.Generator().manual_seed(int(seed))
    seq_lens = [int(x) for x in seq_lens]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max([blocks_needed(L, block_size) for L in seq_lens] + [1])
    table, pool = make_block_table(gen, seq_lens, max_blocks_per_seq, layout, pool_blocks, block_size)
    q = _normal(gen, (B * qlen, Hq, D)).to(torch.float16)
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
    else:
        raise ValueError(kv)
    return Workload(name=name, q=q, k_cache=k_cache, v_cache=v_cache, block_table=table,
                    seq_lens=torch.tensor(seq_lens, dtype=torch.int32),
                    scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
                    window=int(window), qlen=int(qlen), num_splits=int(num_splits), kv_fp8=kv_fp8,
                    kv_int8=kv_int8,
                    k_scale=k_scale, v_scale=v_scale,
                    meta=dict(layout=layout, seed=int(seed), kv=kv))


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
