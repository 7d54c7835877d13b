"""Independent re-derivations used to pin the oracle (test code only).

Nothing here calls the oracle or the CUDA library.  The E4M3 value table comes from PyTorch's
float8_e4m3fn dtype (a library decoder), and encoding is a nearest-value search over that
table, so a slip in the oracle's bit arithmetic (a wrong bias, a dropped sign, a tie rule)
shows up as a disagreement.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def torch_e4m3_values() -> np.ndarray:
    """Value of every code 0..255 via torch.float8_e4m3fn (NaN for 0x7F / 0xFF)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


_POS = None


def _positive_table():
    global _POS
    if _POS is None:
        v = torch_e4m3_values()[:0x7F]      # codes 0x00..0x7E, increasing, 0x7E = 448
        assert np.all(np.diff(v) > 0)
        _POS = v
    return _POS


def nearest_code(t: np.ndarray) -> np.ndarray:
    """Brute-force nearest E4M3 code by search; ties -> even code; |t| > 448 -> 448; sign kept."""
    t = np.asarray(t, dtype=np.float64)
    pos = _positive_table()
    a = np.abs(t)
    hi = np.clip(np.searchsorted(pos, a, side="left"), 0, len(pos) - 1)
    lo = np.clip(hi - 1, 0, len(pos) - 1)
    d_lo = np.abs(a - pos[lo])
    d_hi = np.abs(pos[hi] - a)
    pick = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    pick = np.where(tie, np.where(lo % 2 == 0, lo, hi), pick)
    pick = np.where(a >= pos[-1], len(pos) - 1, pick)
    sign = np.signbit(t).astype(np.uint8) << 7
    return (pick.astype(np.uint8) | sign).astype(np.uint8)


def block_scale_byte(amax: np.ndarray) -> np.ndarray:
    """E8M0 byte from block amax through numpy.frexp (mantissa in [0.5,1) -> floor(log2) = e-1)."""
    amax = np.asarray(amax, dtype=np.float64)
    _, e = np.frexp(amax)
    s = np.where(amax == 0, -127, np.clip(e.astype(np.int64) - 1 - 8, -127, 127))
    return (s + 127).astype(np.uint8)


def quantize_rows_bruteforce(v: np.ndarray):
    """Row-wise MXFP8 of a float64 [M, K] array by frexp + search (independent of the oracle)."""
    M, K = v.shape
    blocks = v.reshape(M, K // 32, 32)
    sf = block_scale_byte(np.abs(blocks).max(axis=2))
    t = np.ldexp(blocks, -(sf.astype(np.int64) - 127)[:, :, None])
    return nearest_code(t).reshape(M, K), sf


def decode(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """Dequantize row-wise codes [.., K] with bytes [.., K/32] through the torch table."""
    vals = torch_e4m3_values()[np.asarray(codes, dtype=np.int64)]
    return np.ldexp(vals, np.repeat(np.asarray(sf, dtype=np.int64) - 127, 32, axis=-1))


def silu(g: float) -> float:
    return g / (1.0 + math.exp(-g))


def bf16_round(v: np.ndarray) -> np.ndarray:
    """binary64 -> nearest bfloat16 value (ties to the even bit pattern), as binary64.

    torch converts float64 to bfloat16 through float32, which rounds twice; here torch's result
    only seeds a search: of its bit pattern and the two neighbouring patterns, the one nearest to
    v wins (the differences are exact in binary64: the candidates lie within a factor of two of
    |v|), and a tie goes to the even pattern."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    seed = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().astype(np.int64) & 0xFFFF
    cand = np.stack([np.maximum(seed - 1, 0), seed, seed + 1])
    vals = (cand.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    d = np.abs(vals - a[None])
    best = np.argmin(d, axis=0)
    dmin = np.take_along_axis(d, best[None], axis=0)[0]
    tie = (d == dmin[None]).sum(axis=0) > 1
    even = np.where(cand % 2 == 0, 0, 1)
    # among the tied candidates take the one with an even pattern
    tb = np.argmin(np.where(d == dmin[None], even, 2), axis=0)
    pick = np.where(tie, tb, best)
    out = np.take_along_axis(vals, pick[None], axis=0)[0]
    return np.where(np.signbit(v), -out, out)


E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)   # codes 0..7 (format definition)


def e2m1_nearest_code(t: np.ndarray) -> np.ndarray:
    """Brute-force nearest E2M1 code by search over the eight magnitudes; ties -> even code;
    |t| > 6 -> 6; sign (also of zero) in bit 3."""
    t = np.asarray(t, dtype=np.float64)
    a = np.abs(t)
    mags = np.array(E2M1_MAGNITUDES)
    d = np.abs(a[..., None] - mags)
    best = d.min(axis=-1, keepdims=True)
    cand = np.where(d == best, np.arange(8), 99)
    even = np.where(cand % 2 == 0, cand, 99).min(axis=-1)
    pick = np.where(even < 99, even, cand.min(axis=-1))
    pick = np.where(a >= 6.0, 7, pick)
    return (pick | (np.signbit(t).astype(np.int64) << 3)).astype(np.uint8)


def e2m1_value(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    mag = np.array(E2M1_MAGNITUDES)[c & 7]
    return np.where(c & 8, -mag, mag)
