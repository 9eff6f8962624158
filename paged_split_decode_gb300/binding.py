"""Thin ctypes binding over libpdecode (C ABI in include/pdecode.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the launch stream, a status other than PD_OK becomes an
exception. Every step of the computation runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpdecode.so")
_lib = None
_lock = threading.Lock()

PD_KV_F16 = 0
PD_KV_FP8_E4M3 = 1
PD_KV_INT8 = 2
PD_KV_BF16 = 3
PD_KV_FP8_E4M3_BF16 = 4  # e4m3fn caches under a bfloat16 q and out
PD_KV_INT8_BF16 = 5      # int8 caches under a bfloat16 q and out
_BF16_IO = (PD_KV_BF16, PD_KV_FP8_E4M3_BF16, PD_KV_INT8_BF16)
DEVERR_BLOCK_ID = 1
DEVERR_SEQ_LEN = 2
DEVERR_TIMEOUT = 4
DEVERR_SLOT = 8
DEVERR_QUERY_START = 16

EXPORTS = ("decode_paged", "decode_paged_varlen", "decode_paged_combine", "decode_paged_static_scratch",
           "write_kv_cache", "pd_workspace_bytes", "pd_grid_ctas", "pd_status_str", "pd_set_wait_limit_ns",
           "pd_set_fault_injection")


class PdDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("D", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float)]


class DecodeError(RuntimeError):
    pass


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libpdecode.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"{_LIB_PATH} is missing: build it first "
                                   "(paged_split_decode_gb300.build.build())")
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            lib.pd_status_str.argtypes = [ctypes.c_int]
            lib.pd_status_str.restype = ctypes.c_char_p
            lib.pd_workspace_bytes.argtypes = [ctypes.POINTER(PdDims), ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int]
            lib.pd_workspace_bytes.restype = ctypes.c_size_t
            lib.pd_grid_ctas.argtypes = [ctypes.POINTER(PdDims), ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int]
            lib.pd_grid_ctas.restype = ctypes.c_int
            lib.decode_paged.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, P, ctypes.POINTER(PdDims), P,
                                         ctypes.c_size_t, P, P]
            lib.decode_paged.restype = ctypes.c_int
            lib.decode_paged_varlen.argtypes = [P, P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_float, ctypes.c_int, ctypes.c_int, P,
                                                ctypes.POINTER(PdDims), P, ctypes.c_size_t, P, P]
            lib.decode_paged_varlen.restype = ctypes.c_int
            lib.decode_paged_combine.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 P, P]
            lib.decode_paged_combine.restype = ctypes.c_int
            lib.write_kv_cache.argtypes = [P, P, P, ctypes.c_int, P, P, ctypes.POINTER(PdDims), P, P]
            lib.write_kv_cache.restype = ctypes.c_int
            lib.pd_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
            lib.pd_set_wait_limit_ns.restype = None
            lib.pd_set_fault_injection.argtypes = [ctypes.c_int]
            lib.pd_set_fault_injection.restype = None
            _lib = lib
    return _lib


def set_wait_limit_ns(ns: int) -> None:
    """Wall-time limit of the decode kernel's pipeline waits (0: default 2 s)."""
    load().pd_set_wait_limit_ns(int(ns))


def set_fault_injection(mode: int) -> None:
    """1: the decode kernel's producer issues no loads (waits run out); 0: off."""
    load().pd_set_fault_injection(int(mode))


def status_str(code: int) -> str:
    return load().pd_status_str(code).decode()


def _check(code: int, what: str):
    if code != 0:
        raise DecodeError(f"{what}: {status_str(code)} (status {code})")


def make_dims(B, Hq, Hkv, D, block_size, num_blocks, max_blocks_per_seq, kv_fp8=False,
              k_scale=1.0, v_scale=1.0, kv_int8=False, kv_bf16=False, q_bf16=False) -> PdDims:
    """``q_bf16``: a bfloat16 q (and out, and new tokens) over fp8 / int8 caches."""
    kind = (PD_KV_BF16 if kv_bf16 else PD_KV_INT8 if kv_int8
            else PD_KV_FP8_E4M3 if kv_fp8 else PD_KV_F16)
    if q_bf16 and kind in (PD_KV_FP8_E4M3, PD_KV_INT8):
        kind += 3
    elif q_bf16 and kind == PD_KV_F16:
        raise TypeError("a bfloat16 q needs bfloat16, fp8 or int8 caches")
    return PdDims(int(B), int(Hq), int(Hkv), int(D), int(block_size), int(num_blocks),
                  int(max_blocks_per_seq), kind, float(k_scale), float(v_scale))


def kv_kind_of(k_cache, act_dtype=None) -> int:
    """fp16 caches -> PD_KV_F16; bfloat16 -> PD_KV_BF16; torch.int8 ->
    PD_KV_INT8; uint8 or float8_e4m3fn -> PD_KV_FP8_E4M3; the byte kinds with
    a bfloat16 ``act_dtype`` (q, or a writer's new tokens) -> PD_KV_INT8_BF16,
    PD_KV_FP8_E4M3_BF16."""
    if k_cache.dtype == torch.float16:
        kind = PD_KV_F16
    elif k_cache.dtype == torch.bfloat16:
        kind = PD_KV_BF16
    elif k_cache.dtype == torch.int8:
        kind = PD_KV_INT8
    elif k_cache.dtype in (torch.uint8, torch.float8_e4m3fn):
        kind = PD_KV_FP8_E4M3
    else:
        raise TypeError(f"unsupported KV cache dtype {k_cache.dtype}")
    if act_dtype == torch.bfloat16 and kind in (PD_KV_FP8_E4M3, PD_KV_INT8):
        kind += 3
    return kind


def _dtypes(kind):
    """(cache dtype(s), q / out / new-token dtype) of a kind."""
    base = {PD_KV_FP8_E4M3_BF16: PD_KV_FP8_E4M3, PD_KV_INT8_BF16: PD_KV_INT8}.get(kind, kind)
    kv_dt = {PD_KV_F16: torch.float16, PD_KV_INT8: torch.int8, PD_KV_BF16: torch.bfloat16,
             PD_KV_FP8_E4M3: (torch.uint8, torch.float8_e4m3fn)}[base]
    return kv_dt, torch.bfloat16 if kind in _BF16_IO else torch.float16


def _dims_for(kind, B, Hq, Hkv, D, bs, num_blocks, max_blocks, k_scale, v_scale) -> PdDims:
    return PdDims(int(B), int(Hq), int(Hkv), int(D), int(bs), int(num_blocks), int(max_blocks), int(kind),
                  float(k_scale), float(v_scale))


def dims_of(q, k_cache, block_table, qlen, kv_fp8=None, k_scale=1.0, v_scale=1.0) -> PdDims:
    num_blocks, bs, Hkv, D = k_cache.shape
    return _dims_for(kv_kind_of(k_cache, q.dtype), block_table.shape[0], q.shape[1], Hkv, D, bs,
                     num_blocks, block_table.shape[1], k_scale, v_scale)


def workspace_bytes(dims: PdDims, qlen: int, num_splits: int, sm_count: int = 0) -> int:
    return int(load().pd_workspace_bytes(ctypes.byref(dims), int(qlen), int(num_splits),
                                         int(sm_count)))


def grid_ctas(dims: PdDims, qlen: int, num_splits: int, sm_count: int = 0) -> int:
    return int(load().pd_grid_ctas(ctypes.byref(dims), int(qlen), int(num_splits), int(sm_count)))


_workspaces: dict = {}


def get_workspace(device: torch.device, nbytes: int, stream: int | None = None) -> torch.Tensor | None:
    """A reusable workspace per (device, stream), grown on demand.

    Every call writes what it reads, so one buffer serves every call made on
    one stream in turn; calls on different streams (which may overlap on the
    GPU) get different buffers. ``stream`` is the raw cudaStream_t handle the
    call launches on (default: torch's current stream on ``device``); the
    buffer is allocated on that stream, so torch's allocator reuses it, once
    it is outgrown, only in that stream's order."""
    if nbytes == 0:
        return None
    cur = torch.cuda.current_stream(device)
    handle = cur.cuda_stream if stream is None else int(stream)
    key = (device.type, device.index, handle)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        size = max(nbytes, 1 << 20)
        if handle == cur.cuda_stream:
            ws = torch.empty(size, dtype=torch.uint8, device=device)
        else:
            with torch.cuda.stream(torch.cuda.ExternalStream(handle, device=device)):
                ws = torch.empty(size, dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def _dev_ptr(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return t.data_ptr()


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale, window=0, qlen=1,
                 num_splits=0, out=None, *, k_scale=1.0, v_scale=1.0, workspace=None,
                 error_flag=None, stream=None):
    """Paged decode attention on the GPU; returns ``out`` (fp16 [B*qlen, Hq, D]).

    ``k_cache``/``v_cache`` are fp16, uint8 / float8_e4m3fn holding e4m3fn
    codes, or int8 codes (then ``k_scale``/``v_scale`` apply). ``num_splits``
    0 = balanced.
    """
    lib = load()
    kind = kv_kind_of(k_cache, q.dtype)
    kv_dt, q_dt = _dtypes(kind)
    dims = dims_of(q, k_cache, block_table, qlen, None, k_scale, v_scale)
    if out is None:
        out = torch.empty_like(q)
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype:
        raise ValueError("v_cache must match k_cache in shape and dtype")
    if q.dim() != 3 or q.shape[0] != block_table.shape[0] * qlen or seq_lens.numel() != block_table.shape[0]:
        raise ValueError("q must be [B*qlen, Hq, D] with B = rows of block_table and seq_lens")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    need = workspace_bytes(dims, qlen, num_splits)
    if workspace is None:
        workspace = get_workspace(q.device, need, stream)
    ws_ptr = 0 if workspace is None else _dev_ptr(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    flag_ptr = None if error_flag is None else _dev_ptr(error_flag, "error_flag", (torch.int32, torch.uint32))
    rc = lib.decode_paged(_dev_ptr(q, "q", q_dt), _dev_ptr(k_cache, "k_cache", kv_dt),
                          _dev_ptr(v_cache, "v_cache", kv_dt),
                          _dev_ptr(block_table, "block_table", torch.int32),
                          _dev_ptr(seq_lens, "seq_lens", torch.int32), float(scale), int(window),
                          int(qlen), int(num_splits), _dev_ptr(out, "out", q_dt),
                          ctypes.byref(dims), ws_ptr or None, ws_bytes, flag_ptr, stream)
    _check(rc, "decode_paged")
    return out


def decode_paged_varlen(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, max_qlen,
                        scale, window=0, num_splits=0, out=None, *, k_scale=1.0, v_scale=1.0,
                        workspace=None, error_flag=None, stream=None):
    """Paged decode with qlen_b = query_start_loc[b+1] - query_start_loc[b]
    query tokens for sequence b (rows query_start_loc[b].. of q and out);
    returns ``out`` (fp16 [T, Hq, D]; rows outside every sequence's range are
    left as they were)."""
    lib = load()
    kind = kv_kind_of(k_cache, q.dtype)
    kv_dt, q_dt = _dtypes(kind)
    dims = dims_of(q, k_cache, block_table, max_qlen, None, k_scale, v_scale)
    if out is None:
        out = torch.zeros_like(q)
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype:
        raise ValueError("v_cache must match k_cache in shape and dtype")
    B = block_table.shape[0]
    if q.dim() != 3 or seq_lens.numel() != B or query_start_loc.numel() != B + 1:
        raise ValueError("q must be [T, Hq, D]; seq_lens [B]; query_start_loc [B+1]")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    need = workspace_bytes(dims, max_qlen, num_splits)
    if workspace is None:
        workspace = get_workspace(q.device, need, stream)
    ws_ptr = 0 if workspace is None else _dev_ptr(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    flag_ptr = None if error_flag is None else _dev_ptr(error_flag, "error_flag", (torch.int32, torch.uint32))
    rc = lib.decode_paged_varlen(_dev_ptr(q, "q", q_dt), _dev_ptr(k_cache, "k_cache", kv_dt),
                                 _dev_ptr(v_cache, "v_cache", kv_dt),
                                 _dev_ptr(block_table, "block_table", torch.int32),
                                 _dev_ptr(seq_lens, "seq_lens", torch.int32),
                                 _dev_ptr(query_start_loc, "query_start_loc", torch.int32),
                                 int(q.shape[0]), int(max_qlen), float(scale), int(window),
                                 int(num_splits), _dev_ptr(out, "out", q_dt),
                                 ctypes.byref(dims), ws_ptr or None, ws_bytes, flag_ptr, stream)
    _check(rc, "decode_paged_varlen")
    return out


def decode_paged_combine(part_m, part_l, part_o, out=None, *, stream=None):
    """Split-K combine: part_m/part_l fp32 [rows, S] (natural-log m), part_o fp32
    [rows, S, D] -> fp16 [rows, D]."""
    lib = load()
    rows, S, D = part_o.shape
    if out is None:
        out = torch.empty((rows, D), dtype=torch.float16, device=part_o.device)
    if stream is None:
        stream = torch.cuda.current_stream(part_o.device).cuda_stream
    rc = lib.decode_paged_combine(_dev_ptr(part_m, "part_m", torch.float32),
                                  _dev_ptr(part_l, "part_l", torch.float32),
                                  _dev_ptr(part_o, "part_o", torch.float32), int(rows), int(S),
                                  int(D), _dev_ptr(out, "out", torch.float16), stream)
    _check(rc, "decode_paged_combine")
    return out


def write_kv_cache(k_new, v_new, slot_mapping, k_cache, v_cache, *, k_scale=1.0, v_scale=1.0,
                   error_flag=None, stream=None):
    """Store new tokens' K/V rows in the paged caches, in place.

    k_new/v_new: fp16 or bfloat16 [T, Hkv, D]; slot_mapping: int64 [T]
    (negative = padding); caches [num_blocks, block_size, Hkv, D] of the
    tokens' type, or uint8 / float8_e4m3fn (e4m3fn codes) or int8 (codes),
    quantised with ``k_scale``/``v_scale``."""
    lib = load()
    kind = kv_kind_of(k_cache, k_new.dtype)
    kv_dt, q_dt = _dtypes(kind)
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype:
        raise ValueError("v_cache must match k_cache in shape and dtype")
    num_blocks, bs, Hkv, D = k_cache.shape
    T = slot_mapping.numel()
    if k_new.shape != (T, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [T, Hkv, D] with T = len(slot_mapping)")
    dims = _dims_for(kind, 0, Hkv, Hkv, D, bs, num_blocks, 0, k_scale, v_scale)
    if stream is None:
        stream = torch.cuda.current_stream(k_cache.device).cuda_stream
    flag_ptr = None if error_flag is None else _dev_ptr(error_flag, "error_flag", (torch.int32, torch.uint32))
    rc = lib.write_kv_cache(_dev_ptr(k_new, "k_new", q_dt),
                            _dev_ptr(v_new, "v_new", q_dt),
                            _dev_ptr(slot_mapping, "slot_mapping", torch.int64), int(T),
                            _dev_ptr(k_cache, "k_cache", kv_dt), _dev_ptr(v_cache, "v_cache", kv_dt),
                            ctypes.byref(dims), flag_ptr, stream)
    _check(rc, "write_kv_cache")
