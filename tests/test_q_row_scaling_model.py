"""The per-row scaling that carries a bfloat16 q into fp16 for the byte
caches' fp16 products, modelled on the CPU: with m the row's largest |q|,
e = clamp(141 - biased_exponent(m), -113, 126) puts m * 2^e in [2^14, 2^15)
(fp16's top binade below 65504) whenever the clamp allows. Then every
element x gives x * 2^e exactly in fp16 (bfloat16 has 8 significant bits,
fp16 11) unless it falls below fp16's normal range, where the error is at
most 2^-25 after scaling: about 2^-39 of the row's largest value. The score
factor 2^-e undoes the scaling exactly. Checked over random rows spanning
bfloat16's exponent range, with numpy's float16 as the reference rounding.
"""
import numpy as np
import torch


def row_exponent(m):
    """The kernels' exponent for a row whose largest |value| is m (float32)."""
    if not m > 0:
        return 0
    eb = int((np.float32(m).view(np.uint32) >> 23) & 255)
    return max(-113, min(126, 141 - eb))


def bf16_row(rng, n, center_exp):
    x = rng.standard_normal(n) * 2.0 ** center_exp
    x[rng.integers(0, n, n // 8)] *= 2.0 ** rng.integers(-30, 1, n // 8)  # small elements too
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float32).numpy()


def test_scaled_rows_are_exact_in_fp16():
    rng = np.random.default_rng(7)
    for center in list(range(-120, 121, 7)) + [-126, -5, 0, 5, 120]:
        for _ in range(4):
            x = bf16_row(rng, 256, center)
            m = float(np.max(np.abs(x)))
            e = row_exponent(m)
            up = np.float32(2.0 ** e)
            y = (x * up).astype(np.float32)
            h = y.astype(np.float16).astype(np.float32)
            if 2.0 ** -113 <= m and m < 2.0 ** 127:  # the clamp does not bind
                assert 2.0 ** 14 <= m * 2.0 ** e < 2.0 ** 15
            assert np.all(np.isfinite(h))          # never past fp16's range
            normal = np.abs(y) >= 2.0 ** -14
            assert np.array_equal(h[normal], y[normal])
            assert np.all(np.abs(h - y) <= 2.0 ** -25)
            # the score factor undoes the scaling exactly
            assert np.array_equal((h[normal] * np.float32(2.0 ** -e)), x[normal])


def test_all_zero_row_keeps_exponent_zero():
    assert row_exponent(0.0) == 0
