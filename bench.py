#!/usr/bin/env python3
"""Benchmark: paged decode attention, KV-read HBM GB/s, D=256 GQA 6:1.

Workload (the decode benchmark of opengfx1030/vllm-rdna pull request #33,
"Test Plan" step 3, at the D=256 6:1 geometry of its results comment): Hq=24,
Hkv=4, D=256, qlen=1, fp16 Q/K/V ~ N(0,1), block_size 16, seq_len 4096 for
every sequence, random-permuted block tables, balanced split. The headline
step is one decode_paged call over B=32 sequences; the batch sweep B in
{1,2,3,8,32} is reported beside it.

One step = one call of the whole path (page translation, KV gather, scores,
masking, online softmax, P.V in the decode kernel; the split combine in a
second kernel launched behind it with programmatic dependent launch). KV bytes are
the algorithmic K+V bytes of the visible keys. Cold L2: every step reads its
KV through a different block table over a pool at least 4x the L2 size, so no
step finds the previous step's KV in L2. The K timed steps are captured in a
CUDA graph and replayed once between CUDA events on the launching stream
(removes host launch overhead only).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on the host cores instead (the
only other implementation available); under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_split_decode_gb300 import inputs  # noqa: E402

METRIC = "paged decode attn: KV-read HBM GB/s (% of GB300 peak), us/call, D=256 GQA 6:1"
UNIT = "GB/s"
HEADLINE_B = 32
SWEEP_B = (1, 2, 3, 8, 32)
HQ, HKV, D, SEQ_LEN, BS = 24, 4, 256, 4096, 16
KERNEL_SOURCES = ["paged_split_decode_gb300/csrc/decode_kernel.cuh",
                  "paged_split_decode_gb300/csrc/ptx.cuh",
                  "paged_split_decode_gb300/csrc/decode_f16_d256.cu",
                  "paged_split_decode_gb300/csrc/launch.h",
                  "paged_split_decode_gb300/csrc/pdecode_api.cu",
                  "paged_split_decode_gb300/csrc/split_combine.cu"]
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the headline decode kernel, from one ncu capture of
#   bench.py --workload gqa6_d256_L4096_b32 --steps 5 --warmup 3
# (-k regex:decode_paged_kernel -s 3 -c 1), with the hash of KERNEL_SOURCES
# it was taken on; reported as roofline.traffic only while the sources hash
# the same (null otherwise).
HEADLINE_TRAFFIC = {"kernel_source_hash": "02d13a5e8a62f2f3", "bytes_per_launch": 537374464 + 3144704}


def kv_bytes_of(seq_lens, qlen, window, Hkv, Dh, elem):
    """Algorithmic KV bytes: each visible key once per (sequence, KV head), K and V."""
    total = 0
    for L in seq_lens:
        if L <= 0:
            continue
        first = max(0, L - qlen - window + 1) if window > 0 else 0
        total += L - first
    return total * Hkv * Dh * elem * 2


def kernel_hash():
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_per_launch():
    """ncu's DRAM read+write bytes per headline decode launch, or None when no
    capture was taken on the current kernel sources."""
    if HEADLINE_TRAFFIC["bytes_per_launch"] is None or HEADLINE_TRAFFIC["kernel_source_hash"] != kernel_hash():
        return None
    return int(HEADLINE_TRAFFIC["bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock/throttle samples (every 50 ms) stamped on arrival; the
    summary keeps the samples that arrived during the timed region (plus 100 ms
    of slack for nvidia-smi's own reporting delay)."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.samples = []
        self.t0 = self.t1 = None

    def _reader(self):
        for ln in self.proc.stdout:
            if ln.strip():
                self.samples.append((time.monotonic(), ln.strip()))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._reader, daemon=True)
            self.th.start()
            t_wait = time.monotonic()
            while not self.samples and time.monotonic() - t_wait < 5:
                time.sleep(0.01)
        except (OSError, ValueError):
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.monotonic()

    def mark_end(self):
        self.t1 = time.monotonic()

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.th.join(timeout=2)

    def summary(self):
        sm, mx, reasons, n_in = [], None, set(), 0
        t0 = self.t0 or 0.0
        t1 = (self.t1 or t0) + 0.1
        rows = [(t, ln) for t, ln in self.samples if t0 <= t <= t1]
        if not rows and self.samples:  # region shorter than one period: nearest sample after it
            after = [(t, ln) for t, ln in self.samples if t >= t0]
            rows = after[:1]
        for _, ln in rows:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            n_in += 1
            for n, v in zip(self.NAMES, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": n_in, "region_ms": round(((self.t1 or t0) - t0) * 1e3, 2)}


def gpu_smi_id(device):
    props = torch.cuda.get_device_properties(device)
    u = getattr(props, "uuid", None)
    if u is not None:
        u = str(u)
        return u if u.startswith("GPU-") else "GPU-" + u
    return str(device.index or 0)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
class DeviceWorkload:
    """A workload resident in HBM with n_rot disjoint block tables over one
    pool at least 4x the L2 size, so consecutive steps never find their K/V in
    L2. Values: N(0,1) fp16 (or e4m3fn codes, NaN codes excluded) drawn on the
    device from a seeded generator; the timed path does not look at them."""

    def __init__(self, device, l2_bytes, seed, B, Hq, Hkv, Dh, seq_lens, qlen=1, window=0,
                 kv="f16", layout="permuted", bs=BS, max_blocks=None, qlens=None):
        # "fp8_bf16q" / "int8_bf16q": byte caches under a bfloat16 q and out
        q_bf16 = kv in ("bf16", "fp8_bf16q", "int8_bf16q")
        kv = {"fp8_bf16q": "fp8", "int8_bf16q": "int8"}.get(kv, kv)
        gen = torch.Generator().manual_seed(seed)
        need = [(L + bs - 1) // bs for L in seq_lens]
        self.max_blocks = max_blocks or max(need + [1])
        per_table = max(sum(need), 1)
        elem = 1 if kv in ("fp8", "int8") else 2
        footprint = per_table * bs * Hkv * Dh * elem * 2
        self.n_rot = min(1024, max(2, -(-4 * l2_bytes // footprint)))
        pool = self.n_rot * per_table
        ids = torch.randperm(pool, generator=gen).to(torch.int32) if layout == "permuted" \
            else torch.arange(pool, dtype=torch.int32)
        self.tables = []
        for r in range(self.n_rot):
            t = torch.full((B, self.max_blocks), -1, dtype=torch.int32)
            off = r * per_table
            for b, n in enumerate(need):
                t[b, :n] = ids[off:off + n]
                off += n
            self.tables.append(t.to(device))
        dg = torch.Generator(device=device).manual_seed(seed + 1)
        shape = (pool, bs, Hkv, Dh)
        if kv == "int8":
            def codes():
                return torch.randint(-127, 128, shape, generator=dg, device=device,
                                     dtype=torch.int32).to(torch.int8)
            self.k, self.v = codes(), codes()
            self.k_scale = self.v_scale = 1.0 / 64
        elif kv == "fp8":
            def codes():
                mag = torch.randint(0, 0x7E + 1, shape, generator=dg, device=device, dtype=torch.int32)
                sign = torch.randint(0, 2, shape, generator=dg, device=device, dtype=torch.int32)
                return (mag | (sign << 7)).to(torch.uint8)
            self.k, self.v = codes(), codes()
            self.k_scale = self.v_scale = 1.0 / 64
        else:
            dt = torch.bfloat16 if kv == "bf16" else torch.float16
            self.k = torch.randn(shape, generator=dg, device=device, dtype=torch.float32).to(dt)
            self.v = torch.randn(shape, generator=dg, device=device, dtype=torch.float32).to(dt)
            self.k_scale = self.v_scale = 1.0
        self.q_start = None
        if qlens is not None:  # a query count per sequence (rows q_start[b]..q_start[b+1]-1)
            starts = [0]
            for n in qlens:
                starts.append(starts[-1] + n)
            self.q_start = torch.tensor(starts, dtype=torch.int32, device=device)
            qlen = max(qlens)
            rows = starts[-1]
        else:
            rows = B * qlen
        self.q = torch.randn((rows, Hq, Dh), generator=dg, device=device,
                             dtype=torch.float32).to(torch.bfloat16 if q_bf16 else torch.float16)
        self.seq_lens = torch.tensor(seq_lens, dtype=torch.int32, device=device)
        self.out = torch.empty_like(self.q)
        self.B, self.qlen, self.window, self.Dh = B, qlen, window, Dh
        self.kv_bytes = kv_bytes_of(seq_lens, qlen, window, Hkv, Dh, elem)
        self.kv = kv
        self.scale = 1.0 / Dh ** 0.5


def time_workload(wl, num_splits, steps, warmup, device, world, sample_clocks=False):
    """K calls captured in one CUDA graph (table r % n_rot for call r), replayed
    once between CUDA events on the launching stream."""
    import paged_split_decode_gb300 as pd
    stream = torch.cuda.Stream(device)
    dims = pd.dims_of(wl.q, wl.k, wl.tables[0], wl.qlen, None, wl.k_scale, wl.v_scale)
    ws = pd.get_workspace(device, pd.workspace_bytes(dims, wl.qlen, num_splits))
    flag = torch.zeros(1, dtype=torch.int32, device=device)

    def call(r):
        if wl.q_start is not None:
            pd.decode_paged_varlen(wl.q, wl.k, wl.v, wl.tables[r % wl.n_rot], wl.seq_lens,
                                   wl.q_start, wl.qlen, wl.scale, wl.window, num_splits, out=wl.out,
                                   k_scale=wl.k_scale, v_scale=wl.v_scale, workspace=ws,
                                   error_flag=flag)
            return
        pd.decode_paged(wl.q, wl.k, wl.v, wl.tables[r % wl.n_rot], wl.seq_lens, wl.scale, wl.window,
                        wl.qlen, num_splits, out=wl.out, k_scale=wl.k_scale, v_scale=wl.v_scale,
                        workspace=ws, error_flag=flag)

    with torch.cuda.stream(stream):
        for r in range(warmup):
            call(r)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for r in range(steps):
            call(warmup + r)
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(device)
    clk = ClockSampler(gpu_smi_id(device)) if sample_clocks else None
    if clk:
        clk.__enter__()
    with torch.cuda.stream(stream):
        if clk:
            clk.mark_start()
        start.record(stream)
        graph.replay()  # launches on the current stream, i.e. `stream`
        end.record(stream)
        end.synchronize()
        if clk:
            clk.mark_end()
    if clk:
        clk.__exit__(None, None, None)
    torch.cuda.synchronize(device)
    barrier(world)
    ms = start.elapsed_time(end)
    if int(flag.item()) != 0:
        raise RuntimeError(f"device error flag {int(flag.item())}")
    del graph
    grid = pd.grid_ctas(dims, wl.qlen, num_splits)
    return ms, (clk.summary() if clk else None), grid


def gqa6_workload(B, device, l2, seed):
    return DeviceWorkload(device, l2, seed, B, HQ, HKV, D, [SEQ_LEN] * B)


def other_workloads(device, l2, seed, only=None):
    """The other workloads the metric covers, as (name, workload, num_splits);
    with `only`, just the one of that name (the others are not built)."""
    full = []

    def add(name, make, S):
        full.append((name, make, S))

    add("tiny_d128_b2_lens100_0", lambda: DeviceWorkload(device, l2, seed, 2, 8, 2, 128, [100, 0],
                                                          max_blocks=8), 1)
    g = torch.Generator().manual_seed(seed + 3)
    lens = torch.randint(512, 16385, (32,), generator=g).tolist()
    for (hq, hkv) in ((32, 8), (28, 4)):
        for layout in ("dense", "permuted"):
            add(f"gqa{hq // hkv}_d128_b32_ragged_{layout}",
                lambda hq=hq, hkv=hkv, layout=layout: DeviceWorkload(
                    device, l2, seed + hq, 32, hq, hkv, 128, lens, layout=layout, max_blocks=1024), 0)
    cache = {}
    for B in (1, 2):
        for window in (4096, 0):
            def mk(B=B, window=window):
                key = (B, window)
                if key not in cache:
                    cache.clear()
                    cache[key] = DeviceWorkload(device, l2, seed + 10 * B + window, B, 24, 4, 256,
                                                [32768] * B, window=window)
                return cache[key]
            for S in (1, 3, 8, 0):
                add(f"long_d256_L32768_b{B}_w{window or 'none'}_s{S or 'auto'}", mk, S)
    add("verify_q3_fp8_d256_L8192_b8",
        lambda: DeviceWorkload(device, l2, seed + 99, 8, 24, 4, 256, [8192] * 8, qlen=3, kv="fp8"), 0)
    add("verify_q3_f16_d256_L8192_b8",
        lambda: DeviceWorkload(device, l2, seed + 98, 8, 24, 4, 256, [8192] * 8, qlen=3), 0)
    add("verify_q3_int8_d256_L8192_b8",
        lambda: DeviceWorkload(device, l2, seed + 97, 8, 24, 4, 256, [8192] * 8, qlen=3, kv="int8"), 0)
    add("gqa6_d256_L4096_b32_fp8",
        lambda: DeviceWorkload(device, l2, seed + 96, 32, 24, 4, 256, [4096] * 32, kv="fp8"), 0)
    add("gqa6_d256_L4096_b32_int8",
        lambda: DeviceWorkload(device, l2, seed + 95, 32, 24, 4, 256, [4096] * 32, kv="int8"), 0)
    add("gqa6_d256_L4096_b32_bf16",
        lambda: DeviceWorkload(device, l2, seed + 93, 32, 24, 4, 256, [4096] * 32, kv="bf16"), 0)
    add("gqa6_d256_L4096_b32_fp8_bf16q",
        lambda: DeviceWorkload(device, l2, seed + 92, 32, 24, 4, 256, [4096] * 32, kv="fp8_bf16q"), 0)
    add("verify_q3_fp8_bf16q_d256_L8192_b8",
        lambda: DeviceWorkload(device, l2, seed + 91, 8, 24, 4, 256, [8192] * 8, qlen=3, kv="fp8_bf16q"), 0)
    gq = torch.Generator().manual_seed(seed + 94)
    qlens = torch.randint(1, 5, (32,), generator=gq).tolist()
    add("varlen_q1to4_d256_L4096_b32",
        lambda: DeviceWorkload(device, l2, seed + 94, 32, 24, 4, 256, [4096] * 32, qlens=qlens), 0)
    for name, make, S in full:
        if only is None or name == only:
            yield name, make(), S



class WriterWorkload:
    """The paged KV-cache writer storing T new tokens (fp16 [T, Hkv, D] K and
    V) into a cache pool at least 4x L2; each step takes the next of n_rot
    disjoint slot mappings and the next of two input sets, so the written
    lines and the read inputs are cold in L2."""

    def __init__(self, device, l2_bytes, seed, T, Hkv, Dh, kv="f16", bs=BS):
        gen = torch.Generator(device=device).manual_seed(seed)
        elem = 1 if kv in ("fp8", "int8") else 2
        row = Hkv * Dh
        self.n_rot = max(2, -(-4 * l2_bytes // (T * row * elem * 2)))
        slots = self.n_rot * T
        self.num_blocks = -(-slots // bs)
        shape = (self.num_blocks, bs, Hkv, Dh)
        dt = {"f16": torch.float16, "fp8": torch.uint8, "int8": torch.int8}[kv]
        self.k = torch.empty(shape, dtype=dt, device=device)
        self.v = torch.empty(shape, dtype=dt, device=device)
        perm = torch.randperm(self.num_blocks * bs, generator=gen, device=device)[:slots]
        self.maps = [perm[r * T:(r + 1) * T].to(torch.int64).contiguous() for r in range(self.n_rot)]
        self.inputs = [(torch.randn((T, Hkv, Dh), generator=gen, device=device).half(),
                        torch.randn((T, Hkv, Dh), generator=gen, device=device).half())
                       for _ in range(2)]
        self.scale = 1.0 if kv == "f16" else 1.0 / 64
        self.bytes = T * row * (2 * 2 + elem * 2)  # read K and V fp16, write both caches


def time_writer(wl, steps, warmup, device, world):
    import paged_split_decode_gb300 as pd
    stream = torch.cuda.Stream(device)
    flag = torch.zeros(1, dtype=torch.int32, device=device)

    def call(r):
        kn, vn = wl.inputs[r % 2]
        pd.write_kv_cache(kn, vn, wl.maps[r % wl.n_rot], wl.k, wl.v, k_scale=wl.scale,
                          v_scale=wl.scale, error_flag=flag)

    with torch.cuda.stream(stream):
        for r in range(warmup):
            call(r)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for r in range(steps):
            call(warmup + r)
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    with torch.cuda.stream(stream):
        start.record(stream)
        graph.replay()
        end.record(stream)
        end.synchronize()
    barrier(world)
    if int(flag.item()) != 0:
        raise RuntimeError(f"writer error flag {int(flag.item())}")
    del graph
    return start.elapsed_time(end)


def writer_workloads(device, l2, seed):
    """Prefill-sized writes: 32768 tokens of the D=256 GQA 6:1 geometry (Hkv=4)."""
    for kv in ("f16", "fp8", "int8"):
        yield f"kv_writer_{kv}_T32768_h4_d256", WriterWorkload(device, l2, seed, 32768, 4, 256, kv)


def time_e2e(B, steps, warmup, device, seed, world):
    """Public API with host buffers: H2D of the step's inputs (pinned), the
    call, D2H of the output, all inside the timed region."""
    import paged_split_decode_gb300 as pd
    gen = torch.Generator().manual_seed(seed)
    nblk = (SEQ_LEN + BS - 1) // BS
    pool = B * nblk
    table = torch.randperm(pool, generator=gen).to(torch.int32).view(B, nblk).pin_memory()
    k = torch.randn((pool, BS, HKV, D), generator=gen).to(torch.float16).pin_memory()
    v = torch.randn((pool, BS, HKV, D), generator=gen).to(torch.float16).pin_memory()
    q = torch.randn((B, HQ, D), generator=gen).to(torch.float16).pin_memory()
    lens = torch.full((B,), SEQ_LEN, dtype=torch.int32).pin_memory()
    out_h = torch.empty((B, HQ, D), dtype=torch.float16).pin_memory()
    dq, dk, dv = (torch.empty_like(x, device=device) for x in (q, k, v))
    dt, dl = torch.empty_like(table, device=device), torch.empty_like(lens, device=device)
    dout = torch.empty_like(dq)
    scale = 1.0 / D ** 0.5
    h2d = sum(x.numel() * x.element_size() for x in (q, k, v, table, lens))
    d2h = out_h.numel() * out_h.element_size()

    def step():
        for dst, src in ((dq, q), (dk, k), (dv, v), (dt, table), (dl, lens)):
            dst.copy_(src, non_blocking=True)
        pd.decode_paged(dq, dk, dv, dt, dl, scale, 0, 1, 0, out=dout)
        out_h.copy_(dout, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(device)
    barrier(world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        step()
    e.record()
    e.synchronize()
    barrier(world)
    return s.elapsed_time(e), h2d, d2h


def cpu_oracle_rate(B, budget_s=10.0, seed=777, max_seqs=None, threads=None):
    """Time the fp64 oracle on the host cores (all of them, or `threads`) over
    whole sequences of the workload; returns (GB/s of KV, cores, sample
    description, seconds/step)."""
    import oracle
    n = B if max_seqs is None else min(B, max_seqs)
    w = inputs.gqa_d256(n, seed=seed)
    args = (w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(), w.block_table.numpy(),
            w.seq_lens.numpy(), w.scale)
    cores = threads or oracle.default_threads()
    oracle.decode_paged(*args, threads=cores)  # warm (builds if needed)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.decode_paged(*args, threads=cores)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = (time.perf_counter() - t0) / reps
    kvb = kv_bytes_of(w.seq_lens.tolist(), 1, 0, HKV, D, 2)
    return kvb / dt / 1e9, cores, f"{n} of {B} sequences x all 24 heads, {reps} runs", dt


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    B = HEADLINE_B
    # bounded sample per step: 4 sequences of the B=32 batch
    nseq = 4
    w = inputs.gqa_d256(nseq, seed=4242)
    cores = oracle.default_threads()
    a = (w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(), w.block_table.numpy(),
         w.seq_lens.numpy(), w.scale)
    for _ in range(args.warmup):
        oracle.decode_paged(*a, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode_paged(*a, threads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    kvb = kv_bytes_of(w.seq_lens.tolist(), 1, 0, HKV, D, 2)
    val = kvb / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(B),
        "cpu_baseline": {"value": round(val, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{nseq} of {B} sequences x all 24 heads per step"},
        "e2e": {"value": round(val, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def short_name(name):
    """A workload's name in the compact per-workload summary."""
    for pat, rep in ((r"^gqa6_d256_L4096_b(\d+)$", r"b\1"), (r"^tiny_.*", "tiny"),
                     (r"^gqa(\d)_d128_b32_ragged_(dense|permuted)$", r"d128g\1_\2"),
                     (r"^long_d256_L32768_", "L32k_"), (r"_w4096_", "_w4k_"),
                     (r"^verify_q3_(\w+?)_d256_L8192_b8$", r"q3_\1"),
                     (r"^gqa6_d256_L4096_b32_", "b32_"), (r"^varlen_q1to4_.*", "varlen"),
                     (r"^kv_writer_(\w+?)_T32768_h4_d256$", r"wr_\1")):
        name = re.sub(pat, rep, name)
    return name


def workload_config(B):
    return {"workload": f"gqa6_d256_L{SEQ_LEN}_b{B}", "B": B, "Hq": HQ, "Hkv": HKV, "D": D,
            "qlen": 1, "seq_len": SEQ_LEN, "block_size": BS, "block_table": "random-permuted",
            "num_splits": "auto (balanced)", "kv_dtype": "fp16",
            "l2": "inputs larger than L2: each step reads its KV through a different block table "
                  "over a pool >= 4x L2", "launch": "CUDA graph of the K steps, replayed once",
            "parallelism": "replicas (one per GPU, no collective)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--workload", default=None,
                    help="time only this workload (a sweep name such as gqa6_d256_L4096_b8 or a "
                         "name from the configs list) and print its line; for profiling")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    from paged_split_decode_gb300 import build as pkg_build
    import paged_split_decode_gb300 as pd
    if rank == 0 or world == 1:
        pkg_build.build()
    barrier(world)
    pd.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    peak, peak_kind = measured_peaks()

    if args.workload and args.workload.startswith("kv_writer_"):
        for name, wwl in writer_workloads(device, l2, 7000):
            if name != args.workload:
                continue
            ms = time_writer(wwl, args.steps, args.warmup, device, world)
            per = ms / args.steps
            if rank == 0:
                print(json.dumps({"workload": name, "us_per_call": round(per * 1e3, 3),
                                  "hbm_gbs": round(wwl.bytes / (per * 1e-3) / 1e9, 1),
                                  "bytes": wwl.bytes, "steps": args.steps}), flush=True)
            return
        raise SystemExit(f"unknown workload {args.workload}")
    if args.workload:
        cands = [(f"gqa6_d256_L{SEQ_LEN}_b{B}", (lambda B=B: gqa6_workload(B, device, l2, 1000 + B)), 0)
                 for B in SWEEP_B]
        for name, wl, S in other_workloads(device, l2, 5000, only=args.workload):
            cands.append((name, (lambda wl=wl: wl), S))
        hit = [c for c in cands if c[0] == args.workload]
        if not hit:
            raise SystemExit(f"unknown workload {args.workload}; known: {[c[0] for c in cands]}")
        name, make, S = hit[0]
        wl = make()
        ms, clk, grid = time_workload(wl, S, args.steps, args.warmup, device, world, sample_clocks=True)
        per = ms / args.steps
        g = wl.kv_bytes / (per * 1e-3) / 1e9
        if rank == 0:
            print(json.dumps({"workload": name, "num_splits": S or "auto", "us_per_call": round(per * 1e3, 3),
                              "kv_gbs": round(g, 1), "frac_of_peak": round(g / peak, 4),
                              "kv_bytes": wl.kv_bytes, "grid_ctas": grid, "steps": args.steps,
                              "clocks": clk}), flush=True)
        return

    sweep = []
    Bs = [HEADLINE_B] if args.no_sweep else list(SWEEP_B)
    head = None
    small_steps = min(args.steps, 200)
    for B in Bs:
        wl = gqa6_workload(B, device, l2, 1000 + B + 17 * rank)
        steps = args.steps if B == HEADLINE_B else small_steps
        ms, clk, grid = time_workload(wl, 0, steps, args.warmup, device, world,
                                      sample_clocks=(B == HEADLINE_B))
        ms = max_over_ranks(ms, world, device)
        per = ms / steps
        gbs = wl.kv_bytes / (per * 1e-3) / 1e9
        sweep.append({"B": B, "us_per_call": round(per * 1e3, 3), "kv_gbs": round(gbs, 1),
                      "frac_of_peak": round(gbs / peak, 4), "kv_bytes": wl.kv_bytes,
                      "grid_ctas": grid, "steps": steps})
        if B == HEADLINE_B:
            head = (ms, per, wl.kv_bytes, gbs, clk)
        del wl
        torch.cuda.empty_cache()
    ms, per, kvb, gbs, clk = head
    total_bytes = kvb * world
    value = total_bytes / (ms / args.steps * 1e-3) / 1e9

    configs = []
    if not args.no_sweep:
        for name, wl, S in other_workloads(device, l2, 5000 + 17 * rank):
            cms, _, grid = time_workload(wl, S, small_steps, args.warmup, device, world)
            cms = max_over_ranks(cms, world, device)
            cper = cms / small_steps
            cg = wl.kv_bytes / (cper * 1e-3) / 1e9
            configs.append({"workload": name, "num_splits": S or "auto",
                            "us_per_call": round(cper * 1e3, 3), "kv_gbs": round(cg, 1),
                            "frac_of_peak": round(cg / peak, 4), "kv_bytes": wl.kv_bytes,
                            "grid_ctas": grid, "steps": small_steps})
            del wl
            torch.cuda.empty_cache()
        for name, wwl in writer_workloads(device, l2, 7000 + 17 * rank):
            wms = max_over_ranks(time_writer(wwl, small_steps, args.warmup, device, world), world,
                                 device)
            wper = wms / small_steps
            wg = wwl.bytes / (wper * 1e-3) / 1e9
            configs.append({"workload": name, "us_per_call": round(wper * 1e3, 3),
                            "hbm_gbs": round(wg, 1), "frac_of_peak": round(wg / peak, 4),
                            "bytes": wwl.bytes, "steps": small_steps,
                            "bytes_are": "K and V fp16 read + both caches written"})
            del wwl
            torch.cuda.empty_cache()

    e2e_steps = args.e2e_steps or max(3, min(args.steps, 10))
    e_ms, h2d, d2h = time_e2e(HEADLINE_B, e2e_steps, 2, device, 99 + rank, world)
    e_ms = max_over_ranks(e_ms, world, device)
    e2e_val = kvb * world / (e_ms / e2e_steps * 1e-3) / 1e9

    cpu = None
    if rank == 0 and not args.no_cpu:
        rate, cores, sample, _ = cpu_oracle_rate(HEADLINE_B, budget_s=10.0, max_seqs=4)
        rate1, _, sample1, _ = cpu_oracle_rate(HEADLINE_B, budget_s=5.0, max_seqs=1, threads=1)
        cpu = {"value": round(rate, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": sample + " (D=256 GQA 6:1, L=4096)",
               "one_core": {"value": round(rate1, 4), "unit": UNIT, "sample": sample1}}
    traffic = traffic_per_launch()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
            "us_per_call": round(per * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": workload_config(HEADLINE_B),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                         "traffic": traffic,
                         "algorithmic_bytes_per_launch": kvb,
                         "kernel": "decode_paged_kernel<D=256,f16,NT=1,HG=2,DS=2>",
                         "timed": "decode kernel + split-combine kernel per step (CUDA events around the graph of K steps)"},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_val, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": args.steps * 2,  # decode kernel + split-combine kernel per step
            "clocks": clk,
            "sweep": sweep,
            "configs": configs,
            # last, so that it ends the line: every workload as [us per call,
            # fraction of the measured copy peak]
            "workloads_fmt": "short name: [us_per_call, frac_of_peak]",
            "workloads": {short_name(f"gqa6_d256_L{SEQ_LEN}_b{r['B']}"): [r["us_per_call"], r["frac_of_peak"]]
                          for r in sweep} | {short_name(c["workload"]): [c["us_per_call"], c["frac_of_peak"]]
                                             for c in configs},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
