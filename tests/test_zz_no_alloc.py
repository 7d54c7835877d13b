"""grouped_mlp_fwd_noalloc: the forward for callers that cannot allocate device memory where
they run it (allocator hooks, out-of-memory handlers, hosts that own the memory pool).  Its
scratch is the library's fixed file-scope device array instead of a caller workspace.  It runs
the same kernels on the same inputs as grouped_mlp_fwd, so its output must equal that entry
point's bit for bit, on consecutive calls (the second call reuses the array the first one left
behind) and on a second, differently shaped problem that finds the first one's contents there.
After the set-up call on the device, repeat calls must not change the device's free memory.
This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

from mxfp8_block_scaled_03_gb300 import workloads as W
from tests import _gpu as G

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mxfp8_block_scaled_03_gb300 import build_ext
    build_ext.build()
    import mxfp8_block_scaled_03_gb300 as mx
    L = mx.lib()

    cases = [W.custom_moe([0, 77, 300, 129], H=256, F=384, seed=41),
             W.custom_moe([500, 12], H=512, F=256, seed=42, with_gates=False)]
    for w in cases:
        x = G.to_dev_bf16(w.x_sorted)
        w1q, w1s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w1), sf_layout=mx.SF_MMA)
        w2q, w2s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w2), sf_layout=mx.SF_MMA)
        split = G.to_dev(w.split_sizes)
        gates = G.to_dev(w.gates) if w.gates is not None else None
        y_ref = mx.grouped_mlp_fwd(x, split, gates, w1q, w1s, w2q, w2s).cpu()
        stream = torch.cuda.current_stream().cuda_stream
        ys = [torch.full((w.R, w.H), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
        torch.cuda.synchronize()

        def call(y):
            return L.grouped_mlp_fwd_noalloc(
                ctypes.c_void_p(x.data_ptr()), w.R, w.H, w.F, w.E, ctypes.c_void_p(split.data_ptr()),
                None if gates is None else ctypes.c_void_p(gates.data_ptr()),
                ctypes.c_void_p(w1q.data_ptr()), ctypes.c_void_p(w1s.data_ptr()),
                ctypes.c_void_p(w2q.data_ptr()), ctypes.c_void_p(w2s.data_ptr()),
                ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(stream))

        st = call(ys[0])                      # on the first case: the device's set-up call
        assert st == 0, mx.mxfp8_status_string(st)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        for y in ys[1:]:
            st = call(y)
            assert st == 0, mx.mxfp8_status_string(st)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before, "a repeat call changed the device's free memory"
        for y in ys:
            assert torch.equal(y.cpu().view(torch.int16), y_ref.view(torch.int16)), \
                "noalloc output differs from grouped_mlp_fwd"
        yn = y_ref.float().numpy()
        assert np.isfinite(yn).all()

    # a problem whose workspace exceeds the fixed array is refused before anything runs
    big = mx.grouped_mlp_workspace_size(65536, 4096, 14336, 8)
    assert big > (64 << 20)
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = L.grouped_mlp_fwd_noalloc(p, 65536, 4096, 14336, 8, p, None, p, p, p, p, p, None)
    assert st == mx.ERR_WORKSPACE
