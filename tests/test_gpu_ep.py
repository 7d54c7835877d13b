"""Expert-parallel MoE layer on the GPU with one NCCL rank (every call in this test suite has one
GPU): the exchanges are copies, so the layer must equal the single-GPU MoE layer (moe_permute ->
grouped_mlp_fwd_tokens -> moe_combine) bit for bit.

Page "Efficient MoE training for biological foundation models", How to run the recipe (experts
spread over the GPUs) and Key technical approaches item 1.  The exchange logic over several ranks
is covered on CPU by tests/test_ep_gloo.py.
"""
import datetime
import os
import socket

import numpy as np
import pytest

from mxfp8_block_scaled_03_gb300 import workloads as W
from tests import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mxfp8_block_scaled_03_gb300 import build_ext
    build_ext.build()
    import mxfp8_block_scaled_03_gb300 as m
    m.lib()
    return m


@pytest.fixture(scope="module")
def nccl_group():
    import torch
    import torch.distributed as dist
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            timeout=datetime.timedelta(seconds=120))
    yield None
    dist.destroy_process_group()


def _weights(mx, w):
    w1q, w1s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w1), sf_layout=mx.SF_MMA)
    w2q, w2s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w2), sf_layout=mx.SF_MMA)
    return w1q, w1s, w2q, w2s


@pytest.mark.parametrize("name,with_gates", [("tiny", True), ("tiny", False), ("mixtral", True)])
def test_one_rank_equals_the_moe_layer(mx, nccl_group, name, with_gates):
    import torch
    from mxfp8_block_scaled_03_gb300 import ep
    w = W.moe_workload(name)
    x = G.to_dev_bf16(w.x_tokens)
    ex = G.to_dev(w.topk_experts.astype(np.int32))
    g = G.to_dev(w.topk_gates) if with_gates else None
    wts = _weights(mx, w)
    split, ros, tor, gs, pws = mx.moe_permute(ex, g, w.E)
    y_rows = mx.grouped_mlp_fwd_tokens(x, tor, split, gs, *wts)
    ref = mx.moe_combine(y_rows, ros)
    got = ep.ep_moe_forward(x, ex, g, wts, w.E)
    torch.cuda.synchronize()
    assert got.shape == ref.shape and got.dtype == torch.bfloat16
    a = got.view(torch.int16).cpu().numpy()
    b = ref.view(torch.int16).cpu().numpy()
    assert np.array_equal(a, b), f"{int((a != b).sum())} elements differ"
    assert np.abs(b.view(np.uint16).astype(np.int64)).max() > 0
