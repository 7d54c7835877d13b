"""mxfp8_block_scaled_03_gb300 -- MXFP8 expert-MLP forward for GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/mxfp8moe.h`` (library
``_build/libmxfp8moe.so``).  The functions keep the C names and only marshal arguments:
torch tensors supply device pointers and the current CUDA stream; every step of the computation
runs in the library's CUDA kernels.  There is no CPU fallback: if the library is missing, calls
raise ``RuntimeError``.

Operations (page "Efficient MoE training for biological foundation models", Key technical
approaches, items 1-3):
  mxfp8_quantize     bf16 -> E4M3 codes + E8M0 scale bytes, row-wise and/or column-wise blocks
                     of 32.
  grouped_mlp_fwd    GroupedLinear(split_sizes) -> ScaledSwiGLU -> MXFP8 requant ->
                     GroupedLinear, in one call.
  moe_permute / grouped_mlp_fwd_tokens / moe_combine
                     the MoE layer around it: device sort of the router's choices by expert,
                     the forward gathering token rows itself, and the per-token sum of outputs.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build_ext

__all__ = [
    "MXFP8Error", "ROWWISE", "COLWISE", "SF_COMPACT", "SF_MMA", "lib", "library_path",
    "mxfp8_sf_bytes", "mxfp8_quantize", "grouped_mlp_workspace_size", "grouped_mlp_workspace_layout",
    "grouped_mlp_fwd", "grouped_mlp_fwd_noalloc", "grouped_mlp_fwd_tokens", "moe_permute",
    "moe_permute_workspace_size", "moe_combine", "moe_gather_rows", "mxfp8_check_device_error", "mxfp8_quantize_colwise_t",
    "grouped_mlp_saved_bytes", "grouped_mlp_fwd_train", "grouped_mlp_bwd_workspace_size", "grouped_mlp_bwd",
    "grouped_mlp_fwd_tokens_train", "grouped_mlp_bwd_tokens", "mxfp8_status_string", "mxfp8_abi_version",
    "mxfp8_mma_peak", "grouped_mlp_bwd_workspace_layout", "nvfp4_sf_bytes", "nvfp4_quantize", "nvfp4_grouped_mlp_workspace_size",
    "nvfp4_grouped_mlp_workspace_layout", "nvfp4_grouped_mlp_fwd",
]

ROWWISE = 1
COLWISE = 2
SF_COMPACT = 0
SF_MMA = 1

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_SPLIT_MISMATCH = range(7)

_lock = threading.Lock()
_lib = None


class MXFP8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({mxfp8_status_string(status)})")


def library_path() -> str:
    return build_ext.LIB


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(build_ext.LIB):
                raise RuntimeError(f"MXFP8 CUDA library not built ({build_ext.LIB}); run "
                                   "mxfp8_block_scaled_03_gb300.build_ext.build() or __graft_entry__.build()")
            L = ctypes.CDLL(build_ext.LIB)
            P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            L.mxfp8_abi_version.restype = i32
            L.mxfp8_abi_version.argtypes = []
            L.mxfp8_status_string.restype = ctypes.c_char_p
            L.mxfp8_status_string.argtypes = [i32]
            L.mxfp8_sf_bytes.restype = sz
            L.mxfp8_sf_bytes.argtypes = [i64, i64, i32, i32]
            L.mxfp8_quantize.restype = i32
            L.mxfp8_quantize.argtypes = [P, i64, i64, i32, i32, P, P, P, P, P]
            L.grouped_mlp_workspace_size.restype = sz
            L.grouped_mlp_workspace_size.argtypes = [i64, i64, i64, i32]
            L.grouped_mlp_workspace_layout.restype = i32
            L.grouped_mlp_workspace_layout.argtypes = [i64, i64, i64, i32, P]
            L.grouped_mlp_fwd.restype = i32
            L.grouped_mlp_fwd.argtypes = [P, i64, i64, i64, i32, P, P, P, P, P, P, P, P, sz, P]
            L.grouped_mlp_fwd_timed.restype = i32
            L.grouped_mlp_fwd_timed.argtypes = [P, i64, i64, i64, i32, P, P, P, P, P, P, P, P, sz, P, P]
            L.grouped_mlp_saved_bytes.restype = sz
            L.grouped_mlp_saved_bytes.argtypes = [i64, i64, i64, i32]
            L.grouped_mlp_fwd_train.restype = i32
            L.grouped_mlp_fwd_train.argtypes = [P, i64, i64, i64, i32, P, P, P, P, P, P, P, P, sz, P, sz, P]
            L.grouped_mlp_bwd_workspace_size.restype = sz
            L.grouped_mlp_bwd_workspace_size.argtypes = [i64, i64, i64, i32]
            L.grouped_mlp_bwd_workspace_layout.restype = i32
            L.grouped_mlp_bwd_workspace_layout.argtypes = [i64, i64, i64, i32, P]
            L.grouped_mlp_bwd.restype = i32
            L.grouped_mlp_bwd.argtypes = [P, i64, i64, i64, i32, P, P, P, sz, P, P, P, P, P, P, P, P, P, P, sz, P]
            L.grouped_mlp_bwd_timed.restype = i32
            L.grouped_mlp_bwd_timed.argtypes = L.grouped_mlp_bwd.argtypes + [P]
            L.grouped_mlp_fwd_tokens_train.restype = i32
            L.grouped_mlp_fwd_tokens_train.argtypes = [P, i64, P, i64, i64, i64, i32, P, P, P, P, P, P, P, P, sz, P,
                                                       sz, P]
            L.grouped_mlp_bwd_tokens.restype = i32
            L.grouped_mlp_bwd_tokens.argtypes = [P, i64, P, i64, i64, i64, i32, P, P, P, sz, P, P, P, P, P, P, P, P,
                                                 P, P, sz, P]
            L.mxfp8_quantize_colwise_t.restype = i32
            L.mxfp8_quantize_colwise_t.argtypes = [P, i64, i64, i32, P, P, P]
            L.grouped_mlp_fwd_noalloc.restype = i32
            L.grouped_mlp_fwd_noalloc.argtypes = [P, i64, i64, i64, i32, P, P, P, P, P, P, P, P]
            L.grouped_mlp_fwd_tokens.restype = i32
            L.grouped_mlp_fwd_tokens.argtypes = [P, i64, P, i64, i64, i64, i32, P, P, P, P, P, P, P, P, sz, P]
            L.moe_permute_workspace_size.restype = sz
            L.moe_permute_workspace_size.argtypes = [i64, i32, i32]
            L.moe_permute.restype = i32
            L.moe_permute.argtypes = [P, P, i64, i32, i32, P, P, P, P, P, sz, P]
            L.moe_combine.restype = i32
            L.moe_combine.argtypes = [P, P, i64, i32, i64, P, P]
            L.moe_gather_rows.restype = i32
            L.moe_gather_rows.argtypes = [P, i64, i64, P, i64, P, P]
            L.mxfp8_check_device_error.restype = i32
            L.mxfp8_check_device_error.argtypes = [P, P, P]
            f32 = ctypes.c_float
            L.nvfp4_sf_bytes.restype = sz
            L.nvfp4_sf_bytes.argtypes = [i64, i64, i32]
            L.nvfp4_quantize.restype = i32
            L.nvfp4_quantize.argtypes = [P, i64, i64, i32, P, P, P, P]
            L.nvfp4_grouped_mlp_workspace_size.restype = sz
            L.nvfp4_grouped_mlp_workspace_size.argtypes = [i64, i64, i64, i32]
            L.nvfp4_grouped_mlp_workspace_layout.restype = i32
            L.nvfp4_grouped_mlp_workspace_layout.argtypes = [i64, i64, i64, i32, P]
            L.nvfp4_grouped_mlp_fwd.restype = i32
            L.nvfp4_grouped_mlp_fwd.argtypes = [P, i64, i64, i64, i32, P, P, P, P, P, P, P, P, f32, P, P, sz, P, P]
            L.mxfp8_mma_peak.restype = i32
            L.mxfp8_mma_peak.argtypes = [i64, i32, P, P, P]
            _lib = L
    return _lib


def _stream(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _check(status: int, where: str):
    if status != OK:
        raise MXFP8Error(status, where)


def mxfp8_abi_version() -> int:
    return int(lib().mxfp8_abi_version())


def mxfp8_status_string(status: int) -> str:
    return lib().mxfp8_status_string(int(status)).decode()


def mxfp8_sf_bytes(M: int, K: int, direction: int, sf_layout: int) -> int:
    return int(lib().mxfp8_sf_bytes(M, K, direction, sf_layout))


def mxfp8_quantize(x, rowwise: bool = True, colwise: bool = False, sf_layout: int = SF_COMPACT,
                   out=None, stream=None):
    """MXFP8 quantization of a contiguous bf16 CUDA tensor [M, K].

    Returns (q_row, sf_row, q_col, sf_col); entries of a direction not requested are None.  Codes
    are uint8 [M, K]; scale bytes are uint8 with mxfp8_sf_bytes(...) elements (compact layout:
    [M, K/32] row-wise, [ceil(M/32), K] column-wise).  `out` may pass preallocated outputs.
    """
    import torch
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous() and x.dim() == 2
    M, K = x.shape
    dirs = (ROWWISE if rowwise else 0) | (COLWISE if colwise else 0)
    if out is None:
        out = [None] * 4
        if rowwise:
            out[0] = torch.empty((M, K), dtype=torch.uint8, device=x.device)
            n = mxfp8_sf_bytes(M, K, ROWWISE, sf_layout)
            out[1] = torch.empty(n, dtype=torch.uint8, device=x.device)
            if sf_layout == SF_COMPACT:
                out[1] = out[1].view(M, K // 32)
        if colwise:
            out[2] = torch.empty((M, K), dtype=torch.uint8, device=x.device)
            n = mxfp8_sf_bytes(M, K, COLWISE, sf_layout)
            out[3] = torch.empty(n, dtype=torch.uint8, device=x.device)
            if sf_layout == SF_COMPACT:
                out[3] = out[3].view((M + 31) // 32, K)
    st = lib().mxfp8_quantize(_ptr(x), M, K, dirs, sf_layout, _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
                              _ptr(out[3]), _stream(stream))
    _check(st, "mxfp8_quantize")
    return tuple(out)


def mxfp8_quantize_colwise_t(x, sf_layout: int = SF_MMA, out=None, stream=None):
    """Column-wise MXFP8 of bf16 [M, K] with the codes transposed: returns (q_t uint8 [K, M],
    sf_t) where row k of q_t holds column k of x in blocks of 32 rows (the operand form of GEMMs
    that contract over x's rows; weights quantized for the backward)."""
    import torch
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous() and x.dim() == 2
    M, K = x.shape
    if out is None:
        q_t = torch.empty((K, M), dtype=torch.uint8, device=x.device)
        n = mxfp8_sf_bytes(K, M, ROWWISE, sf_layout)
        sf_t = torch.empty(n, dtype=torch.uint8, device=x.device)
        if sf_layout == SF_COMPACT:
            sf_t = sf_t.view(K, M // 32)
    else:
        q_t, sf_t = out
    _check(lib().mxfp8_quantize_colwise_t(_ptr(x), M, K, sf_layout, _ptr(q_t), _ptr(sf_t), _stream(stream)),
           "mxfp8_quantize_colwise_t")
    return q_t, sf_t


def grouped_mlp_workspace_size(R: int, H: int, F: int, E: int) -> int:
    return int(lib().grouped_mlp_workspace_size(R, H, F, E))


def grouped_mlp_workspace_layout(R: int, H: int, F: int, E: int) -> dict:
    arr = (ctypes.c_uint64 * 7)()
    _check(lib().grouped_mlp_workspace_layout(R, H, F, E, arr), "grouped_mlp_workspace_layout")
    keys = ["error", "schedule", "xq", "xsf", "hq", "hsf", "r_pad"]
    return {k: int(v) for k, v in zip(keys, arr)}


def grouped_mlp_fwd(x_sorted, split_sizes, gates, w1_q, w1_sf, w2_q, w2_sf, y=None, workspace=None,
                    stream=None, stage_events=None):
    """Fused MXFP8 grouped expert MLP forward.

    x_sorted bf16 [R, H]; split_sizes int32 [E] (device); gates float32 [R] or None; w1_q uint8
    [E*2F, H] with w1_sf in the tensor-core scale layout; w2_q uint8 [E*H, F] with w2_sf.
    Returns y bf16 [R, H].  `workspace` (uint8 CUDA tensor) is allocated here when not given.
    """
    import torch
    R, H = x_sorted.shape
    E = int(split_sizes.numel())
    F = int(w2_q.shape[1])
    assert x_sorted.dtype == torch.bfloat16 and split_sizes.dtype == torch.int32
    assert gates is None or gates.dtype == torch.float32
    for t in (x_sorted, split_sizes, gates, w1_q, w1_sf, w2_q, w2_sf):
        assert t is None or (t.is_cuda and t.is_contiguous())
    if y is None:
        y = torch.empty((R, H), dtype=torch.bfloat16, device=x_sorted.device)
    need = grouped_mlp_workspace_size(R, H, F, E)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x_sorted.device)
    args = (_ptr(x_sorted), R, H, F, E, _ptr(split_sizes), _ptr(gates), _ptr(w1_q), _ptr(w1_sf), _ptr(w2_q),
            _ptr(w2_sf), _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream))
    if stage_events is None:
        _check(lib().grouped_mlp_fwd(*args), "grouped_mlp_fwd")
    else:
        # 5 torch.cuda.Event(enable_timing=True), already recorded once (torch creates the CUDA
        # event lazily): re-recorded before each of the 4 kernels and after the last
        handles = [int(ev.cuda_event) for ev in stage_events]
        if len(handles) != 5 or not all(handles):
            raise ValueError("stage_events: 5 CUDA events that have been recorded at least once")
        arr = (ctypes.c_void_p * 5)(*handles)
        _check(lib().grouped_mlp_fwd_timed(*args, arr), "grouped_mlp_fwd_timed")
    return y


def grouped_mlp_saved_bytes(R: int, H: int, F: int, E: int) -> int:
    return int(lib().grouped_mlp_saved_bytes(R, H, F, E))


def grouped_mlp_bwd_workspace_size(R: int, H: int, F: int, E: int) -> int:
    return int(lib().grouped_mlp_bwd_workspace_size(R, H, F, E))


def grouped_mlp_fwd_train(x_sorted, split_sizes, gates, w1_q, w1_sf, w2_q, w2_sf, y=None, saved=None,
                          workspace=None, stream=None):
    """grouped_mlp_fwd that also keeps the bf16 pre-activations [G | U] the backward needs.
    Returns (y, saved); `saved` is a uint8 CUDA tensor of grouped_mlp_saved_bytes(...) bytes."""
    import torch
    R, H = x_sorted.shape
    E = int(split_sizes.numel())
    F = int(w2_q.shape[1])
    dev = x_sorted.device
    if y is None:
        y = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    if saved is None:
        saved = torch.empty(grouped_mlp_saved_bytes(R, H, F, E), dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = torch.empty(grouped_mlp_workspace_size(R, H, F, E), dtype=torch.uint8, device=dev)
    st = lib().grouped_mlp_fwd_train(_ptr(x_sorted), R, H, F, E, _ptr(split_sizes), _ptr(gates), _ptr(w1_q),
                                     _ptr(w1_sf), _ptr(w2_q), _ptr(w2_sf), _ptr(y), _ptr(saved), saved.numel(),
                                     _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "grouped_mlp_fwd_train")
    return y, saved


def grouped_mlp_bwd(x_sorted, split_sizes, gates, saved, w1t_q, w1t_sf, w2t_q, w2t_sf, dy, dx=None, dgates=True,
                    dw1=None, dw2=None, workspace=None, stream=None, stage_events=None):
    """Backward of the grouped MLP.  w1t_*/w2t_* are W1 [E*2F, H] and W2 [E*H, F] quantized
    along their other axis (mxfp8_quantize_colwise_t, tensor-core layout).  Returns
    (dx bf16 [R, H], dgates float32 [R] or None, dW1 float32 [E, 2F, H], dW2 float32 [E, H, F],
    workspace)."""
    import torch
    R, H = x_sorted.shape
    E = int(split_sizes.numel())
    F = int(w2t_q.shape[0])
    dev = x_sorted.device
    if dx is None:
        dx = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    if dgates is True:
        dgates = torch.empty(R, dtype=torch.float32, device=dev)
    elif dgates is False:
        dgates = None
    if dw1 is None:
        dw1 = torch.empty((E, 2 * F, H), dtype=torch.float32, device=dev)
    if dw2 is None:
        dw2 = torch.empty((E, H, F), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(grouped_mlp_bwd_workspace_size(R, H, F, E), dtype=torch.uint8, device=dev)
    args = (_ptr(x_sorted), R, H, F, E, _ptr(split_sizes), _ptr(gates), _ptr(saved), saved.numel(), _ptr(w1t_q),
            _ptr(w1t_sf), _ptr(w2t_q), _ptr(w2t_sf), _ptr(dy), _ptr(dx), _ptr(dgates), _ptr(dw1), _ptr(dw2),
            _ptr(workspace), workspace.numel(), _stream(stream))
    if stage_events is None:
        _check(lib().grouped_mlp_bwd(*args), "grouped_mlp_bwd")
    else:
        handles = [int(ev.cuda_event) for ev in stage_events]
        if len(handles) != 7 or not all(handles):
            raise ValueError("stage_events: 7 CUDA events that have been recorded at least once")
        _check(lib().grouped_mlp_bwd_timed(*args, (ctypes.c_void_p * 7)(*handles)), "grouped_mlp_bwd_timed")
    return dx, dgates, dw1, dw2, workspace


def grouped_mlp_fwd_tokens_train(x_tokens, token_of_row, split_sizes, gates_sorted, w1_q, w1_sf, w2_q, w2_sf,
                                 y=None, saved=None, workspace=None, stream=None):
    """grouped_mlp_fwd_tokens that also saves the pre-activations.  Returns (y_rows, saved)."""
    import torch
    T, H = x_tokens.shape
    R = int(token_of_row.numel())
    E = int(split_sizes.numel())
    F = int(w2_q.shape[1])
    dev = x_tokens.device
    if y is None:
        y = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    if saved is None:
        saved = torch.empty(grouped_mlp_saved_bytes(R, H, F, E), dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = torch.empty(grouped_mlp_workspace_size(R, H, F, E), dtype=torch.uint8, device=dev)
    st = lib().grouped_mlp_fwd_tokens_train(_ptr(x_tokens), T, _ptr(token_of_row), R, H, F, E, _ptr(split_sizes),
                                            _ptr(gates_sorted), _ptr(w1_q), _ptr(w1_sf), _ptr(w2_q), _ptr(w2_sf),
                                            _ptr(y), _ptr(saved), saved.numel(), _ptr(workspace), workspace.numel(),
                                            _stream(stream))
    _check(st, "grouped_mlp_fwd_tokens_train")
    return y, saved


def grouped_mlp_bwd_tokens(x_tokens, token_of_row, split_sizes, gates_sorted, saved, w1t_q, w1t_sf, w2t_q, w2t_sf,
                           d_out_tokens, workspace=None, stream=None):
    """grouped_mlp_bwd reading x and the output gradient as token rows through token_of_row.
    Returns (dx_rows bf16 [R, H], dgates_sorted float32 [R] or None, dW1, dW2, workspace)."""
    import torch
    T, H = x_tokens.shape
    R = int(token_of_row.numel())
    E = int(split_sizes.numel())
    F = int(w2t_q.shape[0])
    dev = x_tokens.device
    dx = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    dg = torch.empty(R, dtype=torch.float32, device=dev) if gates_sorted is not None else None
    dw1 = torch.empty((E, 2 * F, H), dtype=torch.float32, device=dev)
    dw2 = torch.empty((E, H, F), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(grouped_mlp_bwd_workspace_size(R, H, F, E), dtype=torch.uint8, device=dev)
    st = lib().grouped_mlp_bwd_tokens(_ptr(x_tokens), T, _ptr(token_of_row), R, H, F, E, _ptr(split_sizes),
                                      _ptr(gates_sorted), _ptr(saved), saved.numel(), _ptr(w1t_q), _ptr(w1t_sf),
                                      _ptr(w2t_q), _ptr(w2t_sf), _ptr(d_out_tokens), _ptr(dx), _ptr(dg), _ptr(dw1),
                                      _ptr(dw2), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "grouped_mlp_bwd_tokens")
    return dx, dg, dw1, dw2, workspace


def grouped_mlp_fwd_noalloc(x_sorted, split_sizes, gates, w1_q, w1_sf, w2_q, w2_sf, y, stream=None):
    """grouped_mlp_fwd without a workspace, for callers that cannot allocate device memory at the
    call site: scratch comes from the library's fixed 64 MiB device array (shared by all calls on
    a device; overlapping calls race).  `y` (bf16 [R, H]) must be passed in; nothing is
    allocated.  Sizes whose workspace exceeds 64 MiB raise MXFP8Error (status ERR_WORKSPACE)."""
    R, H = x_sorted.shape
    E = int(split_sizes.numel())
    F = int(w2_q.shape[1])
    st = lib().grouped_mlp_fwd_noalloc(_ptr(x_sorted), R, H, F, E, _ptr(split_sizes), _ptr(gates), _ptr(w1_q),
                                       _ptr(w1_sf), _ptr(w2_q), _ptr(w2_sf), _ptr(y), _stream(stream))
    _check(st, "grouped_mlp_fwd_noalloc")
    return y


def moe_permute_workspace_size(T: int, k: int, E: int) -> int:
    return int(lib().moe_permute_workspace_size(T, k, E))


def moe_permute(experts, gates, E: int, workspace=None, out=None, stream=None):
    """Stable device sort of the router's (token, slot) choices by expert.

    experts int32 [T, k] (CUDA), gates float32 [T, k] or None.  Returns (split_sizes [E],
    row_of_slot [T, k], token_of_row [T*k], gates_sorted [T*k] or None, workspace); `out`
    may pass the first four to be reused."""
    import torch
    T, k = experts.shape
    dev = experts.device
    if out is not None:
        split, row_of_slot, token_of_row, gates_sorted = out
    else:
        split = torch.empty(E, dtype=torch.int32, device=dev)
        row_of_slot = torch.empty((T, k), dtype=torch.int32, device=dev)
        token_of_row = torch.empty(T * k, dtype=torch.int32, device=dev)
        gates_sorted = None if gates is None else torch.empty(T * k, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(256, moe_permute_workspace_size(T, k, E)), dtype=torch.uint8, device=dev)
    st = lib().moe_permute(_ptr(experts), _ptr(gates), T, k, E, _ptr(split), _ptr(row_of_slot), _ptr(token_of_row),
                           _ptr(gates_sorted), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "moe_permute")
    return split, row_of_slot, token_of_row, gates_sorted, workspace


def grouped_mlp_fwd_tokens(x_tokens, token_of_row, split_sizes, gates_sorted, w1_q, w1_sf, w2_q, w2_sf, y=None,
                           workspace=None, stream=None):
    """grouped_mlp_fwd that gathers its rows from x_tokens [T, H] through token_of_row [R] inside
    the activation quantize.  Returns y [R, H] bf16 in sorted-row order."""
    import torch
    T, H = x_tokens.shape
    R = int(token_of_row.numel())
    E = int(split_sizes.numel())
    F = int(w2_q.shape[1])
    if y is None:
        y = torch.empty((R, H), dtype=torch.bfloat16, device=x_tokens.device)
    if workspace is None:
        workspace = torch.empty(grouped_mlp_workspace_size(R, H, F, E), dtype=torch.uint8, device=x_tokens.device)
    st = lib().grouped_mlp_fwd_tokens(_ptr(x_tokens), T, _ptr(token_of_row), R, H, F, E, _ptr(split_sizes),
                                      _ptr(gates_sorted), _ptr(w1_q), _ptr(w1_sf), _ptr(w2_q), _ptr(w2_sf), _ptr(y),
                                      _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "grouped_mlp_fwd_tokens")
    return y


def moe_combine(y_rows, row_of_slot, out=None, stream=None):
    """out[t] = sum_j y_rows[row_of_slot[t, j]] (bf16 out, fp32 sum)."""
    import torch
    T, k = row_of_slot.shape
    H = y_rows.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=y_rows.device)
    _check(lib().moe_combine(_ptr(y_rows), _ptr(row_of_slot), T, k, H, _ptr(out), _stream(stream)), "moe_combine")
    return out


def moe_gather_rows(src, index, out=None, stream=None):
    """out[i] = src[index[i]] (rows copied bit for bit; rows of an index outside [0, len(src)) are
    zeros).  src [N, ...] (rows of a multiple of 4 bytes), index int32 [n]."""
    import torch
    n = int(index.numel())
    row_shape = tuple(src.shape[1:])
    if out is None:
        out = torch.empty((n,) + row_shape, dtype=src.dtype, device=src.device)
    row_bytes = src.element_size() * (int(np.prod(row_shape)) if row_shape else 1)
    _check(lib().moe_gather_rows(_ptr(src), int(src.shape[0]), row_bytes, _ptr(index), n, _ptr(out), _stream(stream)),
           "moe_gather_rows")
    return out


def grouped_mlp_bwd_workspace_layout(R: int, H: int, F: int, E: int) -> list[int]:
    """Byte offsets in a backward workspace: [error word, dGU row-wise codes [R_pad, 2F], their
    scale bytes, dGU column-wise codes transposed [2F, R_pad], their scale bytes, h column-wise
    codes transposed [F, R_pad], their scale bytes, R_pad]; scale bytes in the tensor-core
    layout."""
    out = (ctypes.c_uint64 * 8)()
    _check(lib().grouped_mlp_bwd_workspace_layout(R, H, F, E, out), "grouped_mlp_bwd_workspace_layout")
    return list(out)


def nvfp4_sf_bytes(M: int, K: int, sf_layout: int = SF_COMPACT) -> int:
    return int(lib().nvfp4_sf_bytes(M, K, sf_layout))


def nvfp4_quantize(x, sf_layout: int = SF_COMPACT, out=None, stream=None):
    """NVFP4 of a bf16 [M, K] CUDA tensor.  Returns (codes uint8 [M, K/2], scale codes uint8,
    amax float32 [1]: max |x|, which defines the per-tensor encode scale).  `out` may pass the
    three to be reused."""
    import torch
    M, K = x.shape
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous()
    if out is None:
        out = (torch.empty((M, K // 2), dtype=torch.uint8, device=x.device),
               torch.empty(max(1, nvfp4_sf_bytes(M, K, sf_layout)), dtype=torch.uint8, device=x.device),
               torch.empty(1, dtype=torch.float32, device=x.device))
    q, sf, amax = out
    _check(lib().nvfp4_quantize(_ptr(x), M, K, sf_layout, _ptr(q), _ptr(sf), _ptr(amax), _stream(stream)),
           "nvfp4_quantize")
    return q, sf, amax


def nvfp4_grouped_mlp_workspace_size(R: int, H: int, F: int, E: int) -> int:
    return int(lib().nvfp4_grouped_mlp_workspace_size(R, H, F, E))


def nvfp4_grouped_mlp_workspace_layout(R: int, H: int, F: int, E: int) -> list[int]:
    out = (ctypes.c_uint64 * 7)()
    _check(lib().nvfp4_grouped_mlp_workspace_layout(R, H, F, E, out), "nvfp4_grouped_mlp_workspace_layout")
    return list(out)


def nvfp4_grouped_mlp_fwd(x_sorted, split_sizes, gates, w1, w2, h_amax: float, y=None, workspace=None, stream=None,
                          stage_events=None):
    """NVFP4 grouped expert MLP forward.  w1 = (codes, scale codes in SF_MMA layout, amax) from
    nvfp4_quantize of W1 [E*2F, H]; w2 likewise of W2 [E*H, F]; h_amax: the magnitude the
    intermediate's encode scale is derived from.  Returns y bf16 [R, H]."""
    import torch
    R, H = x_sorted.shape
    E = int(split_sizes.numel())
    F = int(w2[0].shape[1]) * 2
    assert x_sorted.dtype == torch.bfloat16 and split_sizes.dtype == torch.int32
    assert gates is None or gates.dtype == torch.float32
    for t in (x_sorted, split_sizes, gates, *w1, *w2):
        assert t is None or (t.is_cuda and t.is_contiguous())
    if y is None:
        y = torch.empty((R, H), dtype=torch.bfloat16, device=x_sorted.device)
    if workspace is None:
        workspace = torch.empty(nvfp4_grouped_mlp_workspace_size(R, H, F, E), dtype=torch.uint8,
                                device=x_sorted.device)
    ev = None
    if stage_events is not None:   # 5 torch.cuda.Event(enable_timing=True), already recorded once
        handles = [int(e.cuda_event) for e in stage_events]
        if len(handles) != 5 or not all(handles):
            raise ValueError("stage_events: 5 CUDA events that have been recorded at least once")
        ev = (ctypes.c_void_p * 5)(*handles)
    _check(lib().nvfp4_grouped_mlp_fwd(_ptr(x_sorted), R, H, F, E, _ptr(split_sizes), _ptr(gates), _ptr(w1[0]),
                                       _ptr(w1[1]), _ptr(w1[2]), _ptr(w2[0]), _ptr(w2[1]), _ptr(w2[2]),
                                       float(h_amax), _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream),
                                       ev), "nvfp4_grouped_mlp_fwd")
    return y


def mxfp8_mma_peak(iters: int, workspace, fmt: int = 0, stream=None) -> int:
    """Enqueue the block-scaled MMA rate measurement (see include/mxfp8moe.h; fmt 0 MXFP8, 1
    NVFP4); returns the number of CTA-pair clusters launched.  `workspace`: a CUDA tensor of at
    least 4 bytes."""
    n = ctypes.c_int(0)
    _check(lib().mxfp8_mma_peak(int(iters), int(fmt), _ptr(workspace), ctypes.byref(n), _stream(stream)),
           "mxfp8_mma_peak")
    return int(n.value)


def mxfp8_check_device_error(workspace, stream=None) -> tuple[int, int]:
    """(status, raw error bits) of the last grouped_mlp_fwd on this workspace (synchronizes)."""
    flags = ctypes.c_uint32(0)
    st = lib().mxfp8_check_device_error(_ptr(workspace), _stream(stream), ctypes.byref(flags))
    return int(st), int(flags.value)
