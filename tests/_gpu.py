"""Helpers shared by the GPU parity tests (test code only)."""
from __future__ import annotations

import numpy as np


def to_dev_bf16(bits: np.ndarray, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def to_dev(a: np.ndarray, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def sf_mma_to_compact(buf: np.ndarray, rows: int, kb: int, kt: int | None = None) -> np.ndarray:
    """Tensor-core scale layout (512-byte atoms of 128 rows x 4 blocks, row-tile-major with kt
    atoms per 128-row tile; row 32j+i, block b of an atom at 16i + 4j + b) -> compact [rows, kb]."""
    kt = (kb + 3) // 4 if kt is None else kt
    r = np.arange(rows)[:, None]
    b = np.arange(kb)[None, :]
    off = ((r // 128) * kt + b // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (b % 4)
    return np.asarray(buf).reshape(-1)[off]


def e4m3_values() -> np.ndarray:
    import torch
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dequant(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    vals = e4m3_values()[np.asarray(codes, dtype=np.int64)]
    return np.ldexp(vals, np.repeat(np.asarray(sf, dtype=np.int64) - 127, 32, axis=-1))


def e4m3_ulp(mag: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """Spacing of the E4M3 grid at magnitude `mag` under block scale byte `sf` (per element)."""
    s = np.repeat(np.asarray(sf, dtype=np.int64) - 127, 32, axis=-1)
    t = np.ldexp(np.maximum(np.abs(mag), 1e-300), -s)
    _, ex = np.frexp(t)
    e = np.maximum(ex - 1, -6)
    return np.ldexp(1.0, e - 3 + s)


def compare_intermediate(hq_gpu, hs_gpu, hq_ref, hs_ref):
    """(fraction of elements whose dequantized values differ, worst difference in ulps at the
    coarser of the two blocks' grids)."""
    a = dequant(hq_gpu, hs_gpu)
    b = dequant(hq_ref, hs_ref)
    diff = np.abs(a - b)
    ulp = np.maximum(e4m3_ulp(np.maximum(np.abs(a), np.abs(b)), np.maximum(hs_gpu, hs_ref)),
                     e4m3_ulp(np.maximum(np.abs(a), np.abs(b)), hs_gpu))
    frac = float(np.mean(diff != 0))
    worst = float(np.max(diff / ulp)) if diff.size else 0.0
    return frac, worst


def y_errors(y: np.ndarray, y_ref: np.ndarray):
    rel = float(np.linalg.norm(y - y_ref) / max(np.linalg.norm(y_ref), 1e-300))
    mx = float(np.max(np.abs(y - y_ref)) / max(np.max(np.abs(y_ref)), 1e-300))
    return rel, mx


# tolerances stated for the forward: final output and requantized intermediate
Y_REL_TOL = 5e-3
Y_MAX_TOL = 1e-2
HQ_MISMATCH_FRAC = 1e-3
HQ_MAX_ULPS = 1.0


# ---- NVFP4 ----------------------------------------------------------------------------------
def nv_kt(K: int) -> int:
    """Atoms per 128-row tile of an NVFP4 tensor-core scale array (K padded to 256)."""
    return (K + 255) // 256 * 4


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """[.., K] codes one per byte -> [.., K/2] bytes, value 2i in the low nibble of byte i."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def nv_dequant(codes: np.ndarray, sf: np.ndarray, s_enc: float) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    v = np.where(c & 8, -_E2M1[c & 7], _E2M1[c & 7])
    S = e4m3_values()[np.asarray(sf, dtype=np.int64)]
    return v * np.repeat(S, 16, axis=-1) / np.float64(np.float32(s_enc))


def nv_compare_intermediate(hq_gpu, hs_gpu, hq_ref, hs_ref, s_enc):
    """(fraction of values whose dequantized values differ, worst difference in units of the E2M1
    step at the coarser of the two blocks' scales)."""
    a = nv_dequant(hq_gpu, hs_gpu, s_enc)
    b = nv_dequant(hq_ref, hs_ref, s_enc)
    diff = np.abs(a - b)
    S = np.repeat(np.maximum(e4m3_values()[np.asarray(hs_gpu, dtype=np.int64)],
                             e4m3_values()[np.asarray(hs_ref, dtype=np.int64)]), 16, axis=-1)
    unit = S / np.float64(np.float32(s_enc))
    mag = np.maximum(np.abs(a), np.abs(b)) / np.maximum(unit, 1e-300)
    step = np.where(mag < 2, 0.5, np.where(mag < 4, 1.0, 2.0)) * unit
    frac = float(np.mean(diff != 0))
    worst = float(np.max(np.where(diff > 0, diff / np.maximum(step, 1e-300), 0.0))) if diff.size else 0.0
    return frac, worst
