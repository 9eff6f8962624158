"""fp64 CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. The CUDA library never loads it
and shares no code with it.

The arithmetic lives in ``pd_oracle.c`` (plain C, fp64). This module compiles
it with the host C compiler when the shared object is missing or older than
the source, and wraps its three entry points for numpy arrays:

* :func:`decode_paged` -- the one-shot definition (softmax over the visible
  keys of each query token, weighted sum of V), which the "Test Result"
  section of opengfx1030/vllm-rdna pull request #33 calls the one-shot fp64
  reference;
* :func:`decode_paged_split` -- the same result reached through contiguous
  block chunks, online softmax inside each chunk and a split-K combine (the
  schedule model of the same section);
* :func:`combine` -- that combine on its own;
* :func:`decode_paged_varlen` -- a different query count per sequence, each
  sequence being the one-shot decode of itself alone;
* :func:`write_kv_cache` -- the paged KV-cache writer (new tokens into their
  slots, fp16 copied, fp8 / int8 quantised with the per-cache scale) whose
  layout the decode reads back, with its quantisers :func:`e4m3fn_encode` and
  :func:`i8_encode`.

Row ranges are spread over a thread pool; the C code runs without the GIL.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pd_oracle.c")
_LIB = os.path.join(_HERE, "libpdoracle.so")
_lock = threading.Lock()
_lib = None


class Dims(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("qlen", ctypes.c_int), ("Hq", ctypes.c_int),
        ("Hkv", ctypes.c_int), ("D", ctypes.c_int), ("block_size", ctypes.c_int),
        ("num_blocks", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int),
        ("kv_kind", ctypes.c_int), ("k_scale", ctypes.c_double), ("v_scale", ctypes.c_double),
    ]


_ERRORS = {-1: "bad arguments", -2: "block id out of range", -3: "seq_len out of range",
           -4: "out of memory"}


def build(force: bool = False) -> str:
    """Compile pd_oracle.c into libpdoracle.so next to it (portable C, -O2)."""
    with _lock:
        fresh = os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)
        if force or not fresh:
            tmp = _LIB + f".tmp{os.getpid()}"
            cc = os.environ.get("CC", "gcc")
            subprocess.check_call([cc, "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        lib.pdo_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.pdo_f16_to_f64.restype = ctypes.c_double
        lib.pdo_e4m3fn_to_f64.argtypes = [ctypes.c_uint8]
        lib.pdo_e4m3fn_to_f64.restype = ctypes.c_double
        lib.pdo_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.pdo_bf16_to_f64.restype = ctypes.c_double
        lib.pdo_i8_to_f64.argtypes = [ctypes.c_uint8]
        lib.pdo_i8_to_f64.restype = ctypes.c_double
        lib.pdo_decode_paged.argtypes = [ctypes.POINTER(Dims), P, P, P, P, P, ctypes.c_double,
                                         ctypes.c_int, ctypes.c_long, ctypes.c_long, P]
        lib.pdo_decode_paged.restype = ctypes.c_int
        lib.pdo_decode_paged_split.argtypes = [ctypes.POINTER(Dims), P, P, P, P, P, ctypes.c_double,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_long,
                                               ctypes.c_long, P, P, P, P]
        lib.pdo_decode_paged_split.restype = ctypes.c_int
        lib.pdo_combine.argtypes = [ctypes.c_long, ctypes.c_int, ctypes.c_int, P, P, P, P]
        lib.pdo_combine.restype = ctypes.c_int
        lib.pdo_e4m3fn_encode.argtypes = [ctypes.c_float]
        lib.pdo_e4m3fn_encode.restype = ctypes.c_uint8
        lib.pdo_i8_encode.argtypes = [ctypes.c_float]
        lib.pdo_i8_encode.restype = ctypes.c_int8
        lib.pdo_write_kv_cache.argtypes = [ctypes.POINTER(Dims), P, P, P, ctypes.c_long, P, P]
        lib.pdo_write_kv_cache.restype = ctypes.c_int
        _lib = lib
    return _lib


def f16_to_f64(bits: int) -> float:
    return _load().pdo_f16_to_f64(bits)


def e4m3fn_to_f64(code: int) -> float:
    return _load().pdo_e4m3fn_to_f64(code)


def bf16_to_f64(bits: int) -> float:
    return _load().pdo_bf16_to_f64(bits)


def i8_to_f64(code: int) -> float:
    return _load().pdo_i8_to_f64(code)


def e4m3fn_encode(t: float) -> int:
    """e4m3fn code nearest to the fp32 value t (ties to even, saturating)."""
    return int(_load().pdo_e4m3fn_encode(float(np.float32(t))))


def i8_encode(t: float) -> int:
    """Nearest integer to the fp32 value t (ties to even), clamped to +-127."""
    return int(_load().pdo_i8_encode(float(np.float32(t))))


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_bits(a, dtype):
    a = np.ascontiguousarray(np.asarray(a))
    if a.dtype == np.float16 and dtype == np.uint16:
        return a.view(np.uint16)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype} bit patterns, got {a.dtype}")
    return a


def _kv_kind(kv_fp8, kv_int8, bf16):
    """0 fp16, 1 e4m3fn, 2 int8 caches with fp16 q; with bf16: 3 bfloat16
    caches, 4 e4m3fn and 5 int8 caches, q (and new tokens) in bfloat16."""
    if bf16:
        return 4 if kv_fp8 else (5 if kv_int8 else 3)
    return 2 if kv_int8 else int(bool(kv_fp8))


def _prepare(q, k_cache, v_cache, block_table, seq_lens, qlen, k_scale, v_scale, kv_fp8,
             kv_int8=False, bf16=False):
    q = _as_bits(q, np.uint16)
    kdt = np.uint8 if (kv_fp8 or kv_int8) else np.uint16
    k = _as_bits(k_cache, kdt)
    v = _as_bits(v_cache, kdt)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    num_blocks, bs, Hkv, D = k.shape
    assert v.shape == k.shape
    B = sl.shape[0]
    assert bt.ndim == 2 and bt.shape[0] == B
    assert q.shape[0] == B * qlen and q.shape[2] == D
    Hq = q.shape[1]
    dims = Dims(B, qlen, Hq, Hkv, D, bs, num_blocks, bt.shape[1], _kv_kind(kv_fp8, kv_int8, bf16),
                float(k_scale), float(v_scale))
    return dims, q, k, v, bt, sl


def _run_rows(n_rows, threads, fn):
    threads = max(1, min(threads or default_threads(), n_rows or 1))
    bounds = np.linspace(0, n_rows, threads + 1).astype(np.int64)
    if threads == 1:
        rcs = [fn(0, n_rows)]
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            rcs = list(ex.map(lambda k: fn(int(bounds[k]), int(bounds[k + 1])), range(threads)))
    for rc in rcs:
        if rc != 0:
            raise ValueError(f"oracle: {_ERRORS.get(rc, rc)}")


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale, window=0, qlen=1,
                 k_scale=1.0, v_scale=1.0, kv_fp8=False, threads=None, rows=None, kv_int8=False,
                 bf16=False):
    """One-shot fp64 paged decode. Returns float64 [B*qlen, Hq, D].

    q: fp16 [B*qlen, Hq, D]; caches: fp16 (or uint8 e4m3fn codes with
    kv_fp8=True, or int8 codes as uint8 with kv_int8=True)
    [num_blocks, block_size, Hkv, D]; with bf16=True q holds bfloat16 bit
    patterns (uint16), over byte caches as given or else over caches of
    bfloat16 bit patterns. block_table int32 [B, max_blocks];
    seq_lens int32 [B]. ``rows`` = (begin, end) restricts the computed output
    rows (flattened (token, head) index); the others stay 0.
    """
    lib = _load()
    dims, q, k, v, bt, sl = _prepare(q, k_cache, v_cache, block_table, seq_lens, qlen,
                                     k_scale, v_scale, kv_fp8, kv_int8, bf16)
    out = np.zeros((q.shape[0], q.shape[1], q.shape[2]), dtype=np.float64)
    r0, r1 = rows if rows is not None else (0, q.shape[0] * q.shape[1])
    fn = lambda a, b: lib.pdo_decode_paged(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(bt),
                                           _ptr(sl), float(scale), int(window), r0 + a, r0 + b,
                                           _ptr(out))
    _run_rows(r1 - r0, threads, fn)
    return out


def decode_paged_split(q, k_cache, v_cache, block_table, seq_lens, scale, num_splits, window=0,
                       qlen=1, k_scale=1.0, v_scale=1.0, kv_fp8=False, threads=None,
                       return_partials=False, kv_int8=False, bf16=False):
    """Split-mode fp64 paged decode (chunks + online softmax + combine).

    Returns out, or (out, m, l, O) with m/l [rows, S] and O [rows, S, D] when
    ``return_partials`` (rows = B*qlen*Hq, m in natural-log units)."""
    lib = _load()
    dims, q, k, v, bt, sl = _prepare(q, k_cache, v_cache, block_table, seq_lens, qlen,
                                     k_scale, v_scale, kv_fp8, kv_int8, bf16)
    S = int(num_splits)
    n_rows = q.shape[0] * q.shape[1]
    D = q.shape[2]
    out = np.zeros((q.shape[0], q.shape[1], D), dtype=np.float64)
    m = l = O = None
    if return_partials:
        m = np.zeros((n_rows, S)); l = np.zeros((n_rows, S)); O = np.zeros((n_rows, S, D))
    fn = lambda a, b: lib.pdo_decode_paged_split(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v),
                                                 _ptr(bt), _ptr(sl), float(scale), int(window), S,
                                                 a, b, _ptr(out), _ptr(m), _ptr(l), _ptr(O))
    _run_rows(n_rows, threads, fn)
    return (out, m, l, O) if return_partials else out


def decode_paged_varlen(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, scale,
                        window=0, k_scale=1.0, v_scale=1.0, kv_fp8=False, kv_int8=False,
                        threads=None, bf16=False):
    """fp64 paged decode with a query count per sequence: sequence b owns rows
    query_start_loc[b] .. query_start_loc[b+1]-1 of q, and is the one-shot
    decode of that single sequence with qlen = the row count. Rows outside
    every sequence stay 0. Returns float64 [T, Hq, D]."""
    qs = np.asarray(query_start_loc, dtype=np.int64)
    q = np.asarray(q)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(sl.shape[0]):
        a, e = int(qs[b]), int(qs[b + 1])
        if e <= a:
            continue
        out[a:e] = decode_paged(q[a:e], k_cache, v_cache, bt[b:b + 1], sl[b:b + 1], scale,
                                window=window, qlen=e - a, k_scale=k_scale, v_scale=v_scale,
                                kv_fp8=kv_fp8, kv_int8=kv_int8, threads=threads, bf16=bf16)
    return out


def combine(m, l, O):
    """fp64 split-K combine: m, l [rows, S] (natural-log m), O [rows, S, D] -> [rows, D]."""
    lib = _load()
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    O = np.ascontiguousarray(O, dtype=np.float64)
    rows, S, D = O.shape
    out = np.zeros((rows, D), dtype=np.float64)
    rc = lib.pdo_combine(rows, S, D, _ptr(m), _ptr(l), _ptr(O), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle: {_ERRORS.get(rc, rc)}")
    return out


def write_kv_cache(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale=1.0, v_scale=1.0,
                   kv_fp8=False, kv_int8=False, allow_bad_slots=False, bf16=False):
    """Paged KV-cache writer, in place on the numpy caches.

    k_new/v_new: fp16 [T, Hkv, D] (bfloat16 bits with bf16=True: written to
    bfloat16 caches as they are, quantised into byte caches); slot_mapping: int64 [T] (negative = padding
    token, skipped); caches [num_blocks, block_size, Hkv, D] fp16, or uint8
    holding e4m3fn codes (kv_fp8) or int8 codes (kv_int8). A slot beyond the
    cache raises ValueError, or with ``allow_bad_slots`` is skipped and the
    call returns False. Returns True when every slot was in range."""
    lib = _load()
    kdt = np.uint8 if (kv_fp8 or kv_int8) else np.uint16
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("caches must be C-contiguous (they are written in place)")
    kc = k_cache.view(kdt) if k_cache.dtype != kdt else k_cache
    vc = v_cache.view(kdt) if v_cache.dtype != kdt else v_cache
    kn = _as_bits(k_new, np.uint16)
    vn = _as_bits(v_new, np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    num_blocks, bs, Hkv, D = kc.shape
    T = sm.shape[0]
    assert kn.shape == (T, Hkv, D) and vn.shape == kn.shape and vc.shape == kc.shape
    dims = Dims(0, 1, Hkv, Hkv, D, bs, num_blocks, 0, _kv_kind(kv_fp8, kv_int8, bf16),
                float(np.float32(k_scale)), float(np.float32(v_scale)))
    rc = lib.pdo_write_kv_cache(ctypes.byref(dims), _ptr(kn), _ptr(vn), _ptr(sm), T, _ptr(kc),
                                _ptr(vc))
    if rc == -2 and allow_bad_slots:
        return False
    if rc != 0:
        raise ValueError(f"oracle: {_ERRORS.get(rc, rc)}")
    return True


__all__ = ["build", "decode_paged", "decode_paged_split", "decode_paged_varlen", "combine",
           "write_kv_cache",
           "f16_to_f64", "bf16_to_f64", "e4m3fn_to_f64", "i8_to_f64", "e4m3fn_encode", "i8_encode",
           "default_threads"]

if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
