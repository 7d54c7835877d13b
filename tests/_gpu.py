"""Helpers shared by the GPU parity tests (test code only)."""
from __future__ import annotations

import numpy as np


def to_dev_bf16(bits: np.ndarray, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def to_dev(a: np.ndarray, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def sf_mma_to_compact(buf: np.ndarray, rows: int, kb: int) -> np.ndarray:
    """Tensor-core scale layout (512-byte atoms of 128 rows x 4 blocks, row-tile-major; row
    32j+i, block b of an atom at 16i + 4j + b) -> compact [rows, kb]."""
    kt = (kb + 3) // 4
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
