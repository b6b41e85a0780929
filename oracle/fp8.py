"""FP8 (E4M3) draft-head quantisation (TEST INFRASTRUCTURE ONLY).

[DMTP] "DMTP: A Better First Token for Block Drafting via MTP", §6.5 names quantising the
head on the drafting side as a way to cut the vocabulary matrix's traffic, with the
target's verification left as it is: the heads that only produce drafts (T1 from MTP,
T2..T7 from the drafter) may read a quantised copy of the vocabulary matrix; the verify
head stays exact, so the committed tokens do not change.

Reading (the page names no format): E4M3 ("e4m3fn": 4 exponent bits with bias 7, 3
mantissa bits, subnormals, no infinities, largest finite value 448), one power-of-two
scale per row of each operand: s = 2^e with e the smallest integer such that
max|row| <= 448 s, and q = round-to-nearest-even(row / s) on the E4M3 grid. Both the head
rows (once) and each head input row (the RMS-normalised hidden) are quantised; the draft
logits are s_x s_v (q_x . q_v). Power-of-two scales keep row / s exact, so the only
rounding is the E4M3 one.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_grid() -> np.ndarray:
    """The non-negative finite E4M3 values in code order (codes 0..126; code 127 is NaN):
    code = 8 e + m, value m 2^-9 for e = 0 (subnormals), (1 + m/8) 2^(e-7) otherwise."""
    vals = []
    for code in range(127):
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


_GRID = e4m3_grid()


def round_e4m3(x) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to the even code (float64 in and out);
    |x| must not exceed 448 (the scales below guarantee it)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    if np.any(a > E4M3_MAX):
        raise ValueError("value outside the E4M3 range")
    hi = np.searchsorted(_GRID, a, side="left")          # first grid value >= a
    hi = np.minimum(hi, len(_GRID) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _GRID[lo], _GRID[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(a == _GRID[hi], hi, np.where(pick_hi, hi, lo))
    return np.sign(x) * _GRID[code]


def pow2_scale(amax: float) -> float:
    """2^e for the smallest integer e with amax <= 448 * 2^e (1 for an all-zero row)."""
    amax = float(amax)
    if amax == 0.0:
        return 1.0
    e = int(np.ceil(np.log2(amax / E4M3_MAX)))
    while amax > E4M3_MAX * 2.0 ** e:
        e += 1
    while amax <= E4M3_MAX * 2.0 ** (e - 1):
        e -= 1
    return 2.0 ** e


def quantize_rows(X: np.ndarray):
    """(q, s): per-row power-of-two scales s [rows] and E4M3 values q with X ~ q * s."""
    X = np.atleast_2d(np.asarray(X, dtype=np.float64))
    s = np.array([pow2_scale(np.max(np.abs(r))) for r in X])
    q = round_e4m3(X / s[:, None])
    return q, s


def fp8_logits(Y: np.ndarray, Hq: np.ndarray, Hs: np.ndarray) -> np.ndarray:
    """Draft logits of the quantised head: s_y s_v (q_y . q_v) for every row of Y."""
    qy, sy = quantize_rows(Y)
    return (qy @ Hq.T) * sy[:, None] * Hs[None, :]


def fp8_logit_bounds(Y: np.ndarray, Hq: np.ndarray, Hs: np.ndarray, delta: float):
    """Quantised draft logits of rows Y, and how far another implementation's quantised
    logits can be from them when its rows differ from Y by at most ``delta`` per element:
    for each row scale it could pick (the one of Y, and those of max|row| +- delta), its
    element y' / s' rounds to a grid value between round(y/s' - delta/s') and
    round(y/s' + delta/s') (rounding is monotone), so its dequantised element deviates from
    Y's by at most dev_k; the logit of head row v then by at most sum_k |H_vk| dev_k.
    Returns (logits, width)."""
    Y = np.atleast_2d(np.asarray(Y, dtype=np.float64))
    qy, sy = quantize_rows(Y)
    logits = (qy @ Hq.T) * sy[:, None] * Hs[None, :]
    dev = np.zeros_like(Y)
    for i, y in enumerate(Y):
        amax = np.max(np.abs(y))
        ref = qy[i] * sy[i]
        for sc in {sy[i], pow2_scale(amax + delta), pow2_scale(max(amax - delta, 0.0))}:
            lo = round_e4m3(np.clip((y - delta) / sc, -E4M3_MAX, E4M3_MAX)) * sc
            hi = round_e4m3(np.clip((y + delta) / sc, -E4M3_MAX, E4M3_MAX)) * sc
            dev[i] = np.maximum(dev[i], np.maximum(np.abs(hi - ref), np.abs(lo - ref)))
    width = dev @ (np.abs(Hq) * Hs[:, None]).T
    return logits, width
