"""Dense brute-force attention in numpy/torch, written apart from the oracle.

It materialises each sequence's keys into a dense [L, Hkv, D] array through
the block table, builds the boolean visibility matrix from the rules stated in
the oracle's header (causal position L - qlen + i, optional window of W keys
ending at that position), and applies a masked softmax with whole-array numpy
operations. Element decoding uses library routines (numpy's float16, torch's
float8_e4m3fn), not the oracle's own decoders, so the two pin each other.
"""
import numpy as np
import torch


def _bf16_to_f64(x):
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def decode_cache(cache, fp8, scale, int8=False, bf16=False):
    """Byte codes (with a bfloat16 q or not), else bfloat16 or fp16 values."""
    if int8:
        return np.ascontiguousarray(cache).view(np.int8).astype(np.float64) * float(scale)
    if fp8:
        t = torch.from_numpy(np.ascontiguousarray(cache)).view(torch.float8_e4m3fn)
        return t.to(torch.float64).numpy() * float(scale)
    if bf16:
        return _bf16_to_f64(cache)
    return np.asarray(cache).astype(np.float16).astype(np.float64)


def dense_kv(cache_f64, block_table, b, L):
    bs = cache_f64.shape[1]
    idx = [(int(block_table[b][j // bs]), j % bs) for j in range(L)]
    if not idx:
        return np.zeros((0,) + cache_f64.shape[2:])
    return np.stack([cache_f64[blk, slot] for blk, slot in idx])  # [L, Hkv, D]


def visibility(L, qlen, window):
    """[qlen, L] boolean: token i sees key j."""
    j = np.arange(L)[None, :]
    p = (L - qlen + np.arange(qlen))[:, None]
    vis = j <= p
    if window > 0:
        vis &= j >= p - window + 1
    return vis


def attention(q, k_cache, v_cache, block_table, seq_lens, scale, window=0, qlen=1,
              kv_fp8=False, k_scale=1.0, v_scale=1.0, kv_int8=False, q_start=None, bf16=False):
    """q_start (optional, [B+1]): sequence b owns rows q_start[b]..q_start[b+1]-1
    and has that many query tokens; otherwise every sequence has qlen."""
    qf = _bf16_to_f64(q) if bf16 else np.asarray(q).astype(np.float16).astype(np.float64)
    Kc = decode_cache(k_cache, kv_fp8, k_scale, kv_int8, bf16)
    Vc = decode_cache(v_cache, kv_fp8, v_scale, kv_int8, bf16)
    B = len(seq_lens)
    Hq, D = qf.shape[1], qf.shape[2]
    Hkv = Kc.shape[2]
    G = Hq // Hkv
    out = np.zeros_like(qf)
    for b in range(B):
        L = int(seq_lens[b])
        r0, n = (b * qlen, qlen) if q_start is None else (int(q_start[b]), int(q_start[b + 1]) - int(q_start[b]))
        if L <= 0 or n <= 0:
            continue
        Kd = dense_kv(Kc, block_table, b, L)  # [L, Hkv, D]
        Vd = dense_kv(Vc, block_table, b, L)
        Kh = np.repeat(Kd, G, axis=1)           # [L, Hq, D]
        Vh = np.repeat(Vd, G, axis=1)
        vis = visibility(L, n, window)          # [n, L]
        qb = qf[r0:r0 + n]                      # [n, Hq, D]
        s = scale * np.einsum("ihd,jhd->ihj", qb, Kh)
        s = np.where(vis[:, None, :], s, -np.inf)
        m = s.max(axis=-1, keepdims=True)
        seen = np.isfinite(m)
        w = np.where(seen, np.exp(s - np.where(seen, m, 0.0)), 0.0)
        den = w.sum(axis=-1, keepdims=True)
        o = np.einsum("ihj,jhd->ihd", w, Vh) / np.where(den > 0, den, 1.0)
        out[r0:r0 + n] = np.where(seen, o, 0.0)
    return out
