"""CPU oracle for the MXFP8 expert-MLP forward -- TEST INFRASTRUCTURE ONLY.

A ctypes front end over ``mxfp8_oracle.c`` (plain C, binary64 arithmetic).  It restates what
the page "Efficient MoE training for biology foundation models with Transformer Engine"
describes in sections 1-3 (GroupedLinear over split_sizes, MXFP8 blocks of 32, the fused
GroupedLinear -> ScaledSwiGLU -> GroupedLinear op), with the OCP-MX scale rule as the reading of
what the page leaves open.  Only ``tests/``, the package smoke check and the bench's CPU
baseline may import this module.  It shares no code with the CUDA library and never imports it.

Every function takes and returns numpy arrays; bf16 tensors travel as their uint16 bit
patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "mxfp8_oracle.c"), os.path.join(_HERE, "nvfp4_oracle.c")]
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
BAD_ARG = 1
SPLIT_MISMATCH = 6


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, so x86-64 and aarch64 agree)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or any(os.path.getmtime(_LIB_PATH) < os.path.getmtime(p)
                                                      for p in _SRCS):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", *_SRCS, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            L.ora_e4m3_decode.restype = ctypes.c_double
            L.ora_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.ora_e4m3_encode.restype = ctypes.c_uint8
            L.ora_e4m3_encode.argtypes = [ctypes.c_double]
            L.ora_block_exponent.restype = ctypes.c_int
            L.ora_block_exponent.argtypes = [ctypes.c_double]
            L.ora_quantize_block.restype = ctypes.c_uint8
            L.ora_quantize_block.argtypes = [P, ctypes.c_int, P]
            L.ora_e4m3_encode_array.restype = None
            L.ora_e4m3_encode_array.argtypes = [P, i64, P]
            L.ora_e4m3_decode_array.restype = None
            L.ora_e4m3_decode_array.argtypes = [P, i64, P]
            L.ora_quantize_rowwise.restype = ctypes.c_int
            L.ora_quantize_rowwise.argtypes = [P, i64, i64, P, P, ctypes.c_int]
            L.ora_quantize_colwise.restype = ctypes.c_int
            L.ora_quantize_colwise.argtypes = [P, i64, i64, P, P, ctypes.c_int]
            L.ora_grouped_mlp_rows.restype = ctypes.c_int
            L.ora_grouped_mlp_rows.argtypes = [P, i64, i64, i64, ctypes.c_int, P, P, P, P, P, P,
                                               P, i64, P, P, P, ctypes.c_int]
            L.ora_moe_permute.restype = ctypes.c_int
            L.ora_moe_permute.argtypes = [P, P, i64, ctypes.c_int, ctypes.c_int, P, P, P, P]
            L.ora_grouped_mlp_bwd_rows.restype = ctypes.c_int
            L.ora_grouped_mlp_bwd_rows.argtypes = [P, i64, i64, i64, ctypes.c_int, P, P, P, P, P, P, P, P, P,
                                                   P, i64, P, P, P, P, P, ctypes.c_int, ctypes.c_int]
            L.ora_grouped_mlp_bwd_dw.restype = ctypes.c_int
            L.ora_grouped_mlp_bwd_dw.argtypes = [P, i64, i64, i64, ctypes.c_int, P, P, P, P, P, P, P,
                                                 ctypes.c_int, P, i64, P, ctypes.c_int, ctypes.c_int]
            L.ora_round_bf16.restype = ctypes.c_double
            L.ora_round_bf16.argtypes = [ctypes.c_double]
            f32 = ctypes.c_float
            L.ora_e2m1_decode.restype = ctypes.c_double
            L.ora_e2m1_decode.argtypes = [ctypes.c_uint8]
            L.ora_e2m1_encode.restype = ctypes.c_uint8
            L.ora_e2m1_encode.argtypes = [ctypes.c_double]
            L.ora_e2m1_encode_array.restype = None
            L.ora_e2m1_encode_array.argtypes = [P, i64, P]
            L.ora_nvfp4_encode_scale.restype = f32
            L.ora_nvfp4_encode_scale.argtypes = [f32]
            L.ora_nvfp4_quantize_block.restype = ctypes.c_uint8
            L.ora_nvfp4_quantize_block.argtypes = [P, ctypes.c_int, f32, P]
            L.ora_nvfp4_dequant.restype = ctypes.c_double
            L.ora_nvfp4_dequant.argtypes = [ctypes.c_uint8, ctypes.c_uint8, f32]
            L.ora_bf16_amax.restype = f32
            L.ora_bf16_amax.argtypes = [P, i64]
            L.ora_nvfp4_quantize_rowwise.restype = ctypes.c_int
            L.ora_nvfp4_quantize_rowwise.argtypes = [P, i64, i64, P, P, P, ctypes.c_int]
            L.ora_nvfp4_quantize_f32.restype = ctypes.c_int
            L.ora_nvfp4_quantize_f32.argtypes = [P, i64, i64, f32, P, P]
            L.ora_nvfp4_grouped_mlp_rows.restype = ctypes.c_int
            L.ora_nvfp4_grouped_mlp_rows.argtypes = [P, i64, i64, i64, ctypes.c_int, P, P, P, P, f32, P, P, f32, f32,
                                                     P, i64, P, P, P, P, ctypes.c_int]
            L.ora_moe_combine.restype = ctypes.c_int
            L.ora_moe_combine.argtypes = [P, P, i64, ctypes.c_int, i64, P]
            _lib = L
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().ora_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(values: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code (ties to even, saturating) of exact binary64 values."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().ora_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def block_exponent(amax: float) -> int:
    return int(lib().ora_block_exponent(float(amax)))


def quantize_block(values) -> tuple[np.ndarray, int]:
    v = np.ascontiguousarray(values, dtype=np.float64)
    assert 0 < v.size <= 32
    codes = np.empty(v.size, dtype=np.uint8)
    sf = lib().ora_quantize_block(_ptr(v), v.size, _ptr(codes))
    return codes, int(sf)


def quantize_rowwise(x_bf16: np.ndarray, nthreads: int | None = None):
    """[M, K] bf16 bits -> (codes [M, K] uint8, E8M0 bytes [M, K/32] uint8)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    q = np.empty((M, K), dtype=np.uint8)
    sf = np.empty((M, K // 32), dtype=np.uint8)
    rc = lib().ora_quantize_rowwise(_ptr(x), M, K, _ptr(q), _ptr(sf), nthreads or default_threads())
    if rc != OK:
        raise ValueError(f"oracle quantize_rowwise rejected the arguments (status {rc})")
    return q, sf


def quantize_colwise(x_bf16: np.ndarray, nthreads: int | None = None):
    """[M, K] bf16 bits -> (codes [M, K] uint8, E8M0 bytes [ceil(M/32), K] uint8)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    q = np.empty((M, K), dtype=np.uint8)
    sf = np.empty(((M + 31) // 32, K), dtype=np.uint8)
    rc = lib().ora_quantize_colwise(_ptr(x), M, K, _ptr(q), _ptr(sf), nthreads or default_threads())
    if rc != OK:
        raise ValueError(f"oracle quantize_colwise rejected the arguments (status {rc})")
    return q, sf


def dequantize_rowwise(q: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """Value of row-wise codes under their E8M0 bytes, in binary64."""
    vals = e4m3_decode(q)
    return np.ldexp(vals, (np.repeat(sf.astype(np.int64), 32, axis=-1) - 127))


def grouped_mlp_rows(x_bf16, split_sizes, gates, w1q, w1sf, w2q, w2sf, rows, nthreads=None,
                     want_intermediate=True):
    """Rows of the grouped MLP forward in binary64.

    x_bf16 [R, H] bf16 bits; split_sizes [E]; gates [R] float32 or None (all ones);
    w1q [E*2F, H] codes + w1sf [E*2F, H/32]; w2q [E*H, F] codes + w2sf [E*H, F/32] (all from
    the oracle's own quantize_rowwise).  Returns (y [n, H] float64, hq [n, F], hsf [n, F/32]).
    """
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, H = x.shape
    split = np.ascontiguousarray(split_sizes, dtype=np.int32)
    E = split.size
    F = w2q.shape[1]
    g = None if gates is None else np.ascontiguousarray(gates, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    y = np.empty((n, H), dtype=np.float64)
    hq = np.empty((n, F), dtype=np.uint8) if want_intermediate else None
    hsf = np.empty((n, F // 32), dtype=np.uint8) if want_intermediate else None
    arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (w1q, w1sf, w2q, w2sf)]
    rc = lib().ora_grouped_mlp_rows(_ptr(x), R, H, F, E, _ptr(split), _ptr(g), *[_ptr(a) for a in arrs],
                                    _ptr(rows), n, _ptr(y), _ptr(hq), _ptr(hsf),
                                    nthreads or default_threads())
    if rc != OK:
        raise ValueError(f"oracle grouped_mlp_rows rejected the arguments (status {rc})")
    return y, hq, hsf


def moe_permute(experts: np.ndarray, gates: np.ndarray | None, E: int):
    """Stable sort of (token, slot) pairs by expert.  experts [T, k] int ->
    (split [E], row_of_slot [T, k], token_of_row [T*k], gates_sorted [T*k] or None)."""
    ex = np.ascontiguousarray(experts, dtype=np.int32)
    T, k = ex.shape
    g = None if gates is None else np.ascontiguousarray(gates, dtype=np.float32)
    split = np.empty(E, dtype=np.int32)
    row_of_slot = np.empty((T, k), dtype=np.int32)
    token_of_row = np.empty(T * k, dtype=np.int32)
    gs = None if g is None else np.empty(T * k, dtype=np.float32)
    rc = lib().ora_moe_permute(_ptr(ex), _ptr(g), T, k, E, _ptr(split), _ptr(row_of_slot), _ptr(token_of_row),
                               _ptr(gs))
    if rc != OK:
        raise ValueError(f"oracle moe_permute rejected the arguments (status {rc})")
    return split, row_of_slot, token_of_row, gs


def moe_combine(y: np.ndarray, row_of_slot: np.ndarray) -> np.ndarray:
    """out[t] = sum_j y[row_of_slot[t, j]] in binary64."""
    yy = np.ascontiguousarray(y, dtype=np.float64)
    rs = np.ascontiguousarray(row_of_slot, dtype=np.int32)
    T, k = rs.shape
    H = yy.shape[1]
    out = np.empty((T, H), dtype=np.float64)
    rc = lib().ora_moe_combine(_ptr(yy), _ptr(rs), T, k, H, _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle moe_combine rejected the arguments (status {rc})")
    return out


def round_bf16(v: float) -> float:
    return float(lib().ora_round_bf16(float(v)))


def quantize_transposed(w_bf16: np.ndarray, E: int, nthreads: int | None = None):
    """Per-expert transpose, then row-wise MXFP8: w [E*A, B] bf16 bits -> codes [E*B, A] and
    E8M0 bytes [E*B, A/32] (the weight quantized along its other axis, as the backward GEMMs
    contract over it)."""
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    EA, B = w.shape
    A = EA // E
    wt = np.ascontiguousarray(w.reshape(E, A, B).transpose(0, 2, 1).reshape(E * B, A))
    return quantize_rowwise(wt, nthreads)


def grouped_mlp_bwd_rows(x_bf16, split_sizes, gates, w1q, w1sf, w2tq, w2tsf, w1tq, w1tsf, dy_bf16, rows,
                         nthreads=None, quant=True, want_gu=False):
    """Backward rows in binary64: (dx [n, H], dgate [n], dGU bf16 bits [n, 2F], h bf16 bits [n, F]),
    and with want_gu also the forward's saved pre-activations [g | u] as bf16 bits [n, 2F].
    quant=False turns every quantization and bf16 rounding of x, dy and the intermediates into the
    identity (a test hook; the weights are always taken from their codes).

    w1q/w1sf: W1 row-wise (forward); w2tq/w2tsf: W2 quantized along H (quantize_transposed);
    w1tq/w1tsf: W1 quantized along 2F (quantize_transposed)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    dy = np.ascontiguousarray(dy_bf16, dtype=np.uint16)
    R, H = x.shape
    split = np.ascontiguousarray(split_sizes, dtype=np.int32)
    E = split.size
    F = w2tq.shape[0] // E
    g = None if gates is None else np.ascontiguousarray(gates, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    dx = np.empty((n, H), dtype=np.float64)
    dgate = np.empty(n, dtype=np.float64)
    dgu = np.empty((n, 2 * F), dtype=np.uint16)
    hb = np.empty((n, F), dtype=np.uint16)
    gu = np.empty((n, 2 * F), dtype=np.uint16) if want_gu else None
    arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (w1q, w1sf, w2tq, w2tsf, w1tq, w1tsf)]
    rc = lib().ora_grouped_mlp_bwd_rows(_ptr(x), R, H, F, E, _ptr(split), _ptr(g), *[_ptr(a) for a in arrs],
                                        _ptr(dy), _ptr(rows), n, _ptr(dx), _ptr(dgate), _ptr(dgu), _ptr(hb),
                                        _ptr(gu), 1 if quant else 0, nthreads or default_threads())
    if rc != OK:
        raise ValueError(f"oracle grouped_mlp_bwd_rows rejected the arguments (status {rc})")
    return (dx, dgate, dgu, hb, gu) if want_gu else (dx, dgate, dgu, hb)


def grouped_mlp_bwd_dw(x_bf16, split_sizes, gates, w1q, w1sf, w2tq, w2tsf, dy_bf16, which: int, entries,
                       nthreads=None, quant=True):
    """Weight-gradient entries in binary64.  which = 2: dW2 [E, H, F]; which = 1: dW1 [E, 2F, H];
    entries: int array [n, 3] of (expert, row, column)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    dy = np.ascontiguousarray(dy_bf16, dtype=np.uint16)
    R, H = x.shape
    split = np.ascontiguousarray(split_sizes, dtype=np.int32)
    E = split.size
    F = w2tq.shape[0] // E
    g = None if gates is None else np.ascontiguousarray(gates, dtype=np.float32)
    ent = np.ascontiguousarray(entries, dtype=np.int64).reshape(-1, 3)
    out = np.empty(ent.shape[0], dtype=np.float64)
    arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (w1q, w1sf, w2tq, w2tsf)]
    rc = lib().ora_grouped_mlp_bwd_dw(_ptr(x), R, H, F, E, _ptr(split), _ptr(g), *[_ptr(a) for a in arrs], _ptr(dy),
                                      which, _ptr(ent), ent.shape[0], _ptr(out), 1 if quant else 0,
                                      nthreads or default_threads())
    if rc != OK:
        raise ValueError(f"oracle grouped_mlp_bwd_dw rejected the arguments (status {rc})")
    return out


# ------------------------------------------------------------------------------------------------
# NVFP4 (nvfp4_oracle.c): E2M1 codes one per byte (sign in bit 3), E4M3 block-scale codes per 16
# values, per-tensor binary32 encode scale s_enc = 2688 / amax.
# ------------------------------------------------------------------------------------------------
def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    return np.vectorize(lambda v: lib().ora_e2m1_decode(int(v)), otypes=[np.float64])(c)


def e2m1_encode(values: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().ora_e2m1_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def nvfp4_encode_scale(amax: float) -> float:
    return float(lib().ora_nvfp4_encode_scale(float(amax)))


def nvfp4_quantize_block(values, s_enc: float) -> tuple[np.ndarray, int]:
    v = np.ascontiguousarray(values, dtype=np.float32)
    assert 0 < v.size <= 16
    codes = np.empty(v.size, dtype=np.uint8)
    sf = lib().ora_nvfp4_quantize_block(_ptr(v), v.size, float(s_enc), _ptr(codes))
    return codes, int(sf)


def nvfp4_quantize_rowwise(x_bf16: np.ndarray, nthreads: int | None = None):
    """[M, K] bf16 bits -> (E2M1 codes [M, K] one per byte, E4M3 scale codes [M, K/16], s_enc)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    q = np.empty((M, K), dtype=np.uint8)
    sf = np.empty((M, K // 16), dtype=np.uint8)
    s = ctypes.c_float(0.0)
    rc = lib().ora_nvfp4_quantize_rowwise(_ptr(x), M, K, _ptr(q), _ptr(sf), ctypes.byref(s),
                                          nthreads or default_threads())
    if rc != OK:
        raise ValueError(f"oracle nvfp4_quantize_rowwise rejected the arguments (status {rc})")
    return q, sf, float(s.value)


def nvfp4_quantize_f32(v: np.ndarray, s_enc: float):
    """Row-wise NVFP4 of binary32 values [M, K] under a given encode scale."""
    a = np.ascontiguousarray(v, dtype=np.float32)
    M, K = a.shape
    q = np.empty((M, K), dtype=np.uint8)
    sf = np.empty((M, K // 16), dtype=np.uint8)
    rc = lib().ora_nvfp4_quantize_f32(_ptr(a), M, K, float(s_enc), _ptr(q), _ptr(sf))
    if rc != OK:
        raise ValueError(f"oracle nvfp4_quantize_f32 rejected the arguments (status {rc})")
    return q, sf


def nvfp4_dequantize(q: np.ndarray, sf: np.ndarray, s_enc: float) -> np.ndarray:
    """Value of row-wise NVFP4 codes [.., K] with block-scale codes [.., K/16], in binary64."""
    vals = e2m1_decode(q)
    return vals * np.repeat(e4m3_decode(sf), 16, axis=-1) / np.float64(np.float32(s_enc))


def bf16_amax(x_bf16: np.ndarray) -> float:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    return float(lib().ora_bf16_amax(_ptr(x), x.size))


def nvfp4_grouped_mlp_rows(x_bf16, split_sizes, gates, w1, w2, h_amax: float, rows, nthreads=None,
                           want_intermediate=True):
    """Rows of the NVFP4 grouped MLP forward in binary64.  w1 = (codes, scale codes, s_enc) of
    W1 [E*2F, H] and w2 likewise of W2 [E*H, F], as nvfp4_quantize_rowwise returns them.
    Returns (y [n, H], hq [n, F] codes, hsf [n, F/16] scale codes, s_x)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, H = x.shape
    split = np.ascontiguousarray(split_sizes, dtype=np.int32)
    E = split.size
    F = w2[0].shape[1]
    g = None if gates is None else np.ascontiguousarray(gates, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    y = np.empty((n, H), dtype=np.float64)
    hq = np.empty((n, F), dtype=np.uint8) if want_intermediate else None
    hsf = np.empty((n, F // 16), dtype=np.uint8) if want_intermediate else None
    w1q, w1s = (np.ascontiguousarray(a, dtype=np.uint8) for a in w1[:2])
    w2q, w2s = (np.ascontiguousarray(a, dtype=np.uint8) for a in w2[:2])
    s_x = ctypes.c_float(0.0)
    rc = lib().ora_nvfp4_grouped_mlp_rows(_ptr(x), R, H, F, E, _ptr(split), _ptr(g), _ptr(w1q), _ptr(w1s),
                                          float(w1[2]), _ptr(w2q), _ptr(w2s), float(w2[2]), float(h_amax),
                                          _ptr(rows), n, _ptr(y), _ptr(hq), _ptr(hsf), ctypes.byref(s_x),
                                          nthreads or default_threads())
    if rc != OK:
        raise ValueError(f"oracle nvfp4_grouped_mlp_rows rejected the arguments (status {rc})")
    return y, hq, hsf, float(s_x.value)
