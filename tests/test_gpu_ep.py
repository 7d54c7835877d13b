"""Expert-parallel MoE layer on the GPU with one NCCL rank (every call in this test suite has one
GPU): the exchanges are copies, so the layer must equal the single-GPU MoE layer (moe_permute ->
grouped_mlp_fwd_tokens -> moe_combine, and its backward) bit for bit.  Also the row gather the
layer moves rows with (moe_gather_rows), bit-exact against numpy indexing.

The expert-parallel layer's forward output, input gradient and routing-weight gradients are
also put beside the oracle's combined layer directly (element by element at the forward's y
tolerances), on every token of the tiny workload and on sampled tokens of the Mixtral-shaped one.

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


@pytest.mark.parametrize("dtype,width", [("bf16", 4096), ("f32", 1), ("f32", 3), ("i32", 8)])
def test_gather_rows_bit_exact(mx, dtype, width):
    import torch
    rng = np.random.default_rng(width)
    n_src, n = 1000, 2500
    if dtype == "bf16":
        src_np = rng.integers(0, 1 << 16, size=(n_src, width), dtype=np.uint16)
        src = torch.from_numpy(src_np.view(np.int16)).cuda().view(torch.bfloat16)
    elif dtype == "f32":
        src_np = rng.integers(0, 1 << 32, size=(n_src, width), dtype=np.uint32)   # any bit pattern, NaNs included
        src = torch.from_numpy(src_np.view(np.int32)).cuda().view(torch.float32)
    else:
        src_np = rng.integers(0, 1 << 32, size=(n_src, width), dtype=np.uint32)
        src = torch.from_numpy(src_np.view(np.int32)).cuda()
    if width == 1:
        src = src.view(-1)
    idx = rng.integers(-3, n_src + 3, size=n).astype(np.int32)   # a few out of range: zero rows
    got = mx.moe_gather_rows(src, torch.from_numpy(idx).cuda())
    bits = got.view(torch.int16 if dtype == "bf16" else torch.int32).cpu().numpy().reshape(n, -1)
    ref = np.zeros((n, width), dtype=src_np.dtype)
    ok = (idx >= 0) & (idx < n_src)
    ref[ok] = src_np[idx[ok]]
    assert np.array_equal(bits.view(src_np.dtype), ref)


@pytest.mark.parametrize("with_gates", [True, False])
def test_one_rank_training_equals_the_moe_layer(mx, nccl_group, with_gates):
    import torch
    from mxfp8_block_scaled_03_gb300 import ep
    w = W.moe_workload("tiny")
    x = G.to_dev_bf16(w.x_tokens)
    ex = G.to_dev(w.topk_experts.astype(np.int32))
    g = G.to_dev(w.topk_gates) if with_gates else None
    wts = _weights(mx, w)
    w1t = mx.mxfp8_quantize_colwise_t(G.to_dev_bf16(w.w1))
    w2t = mx.mxfp8_quantize_colwise_t(G.to_dev_bf16(w.w2))
    wts_t = (w1t[0], w1t[1], w2t[0], w2t[1])
    d_out = G.to_dev_bf16(W.bf16_bits(np.random.default_rng(4).standard_normal(w.x_tokens.shape).astype(np.float32)))
    # the single-GPU layer and its backward
    split, ros, tor, gs, _ = mx.moe_permute(ex, g, w.E)
    y_rows, saved = mx.grouped_mlp_fwd_tokens_train(x, tor, split, gs, *wts)
    ref = mx.moe_combine(y_rows, ros)
    dx_rows, dg_rows, dw1, dw2, _ = mx.grouped_mlp_bwd_tokens(x, tor, split, gs, saved, *wts_t, d_out)
    dx_ref = mx.moe_combine(dx_rows, ros)
    # through the expert-parallel path
    out, ctx = ep.ep_moe_forward_train(x, ex, g, wts, w.E)
    dx, dg, edw1, edw2 = ep.ep_moe_backward(d_out, ctx, wts_t)
    torch.cuda.synchronize()

    def bits(t):
        return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()

    assert np.array_equal(bits(out), bits(ref))
    assert np.array_equal(bits(dx), bits(dx_ref))
    assert np.array_equal(bits(edw1), bits(dw1)) and np.array_equal(bits(edw2), bits(dw2))
    if with_gates:
        assert np.array_equal(bits(dg), bits(dg_rows[ros.long()]))
    else:
        assert dg is None


def _tokens(w, name):
    if name == "tiny":
        return np.arange(w.T)
    rng = np.random.default_rng(5)
    return np.unique(np.concatenate([[0, 1, w.T - 1], rng.choice(w.T, 21, replace=False)]))


@pytest.mark.parametrize("name", ["tiny", "mixtral"])
def test_ep_layer_forward_and_backward_match_oracle(mx, nccl_group, oracle, name):
    """ep_moe_forward_train -> ep_moe_backward on one NCCL rank against the oracle: the oracle's
    own permutation of the router choices, its binary64 forward and backward of the sorted rows
    (the output gradient of row r is d_out[token_of_row[r]]), and its combine."""
    import torch
    from mxfp8_block_scaled_03_gb300 import ep
    w = W.moe_workload(name)
    x = G.to_dev_bf16(w.x_tokens)
    ex = G.to_dev(w.topk_experts.astype(np.int32))
    g = G.to_dev(w.topk_gates)
    w1, w2 = G.to_dev_bf16(w.w1), G.to_dev_bf16(w.w2)
    wts = _weights(mx, w)
    w1t = mx.mxfp8_quantize_colwise_t(w1)
    w2t = mx.mxfp8_quantize_colwise_t(w2)
    d_out = W.bf16_bits(np.random.default_rng(8).standard_normal((w.T, w.H)).astype(np.float32))
    out, ctx = ep.ep_moe_forward_train(x, ex, g, wts, w.E)
    out_inf = ep.ep_moe_forward(x, ex, g, wts, w.E)
    dx, dg, _, _ = ep.ep_moe_backward(G.to_dev_bf16(d_out), ctx, (w1t[0], w1t[1], w2t[0], w2t[1]))
    torch.cuda.synchronize()
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    out, out_inf, dx, dg = f64(out), f64(out_inf), f64(dx), dg.cpu().numpy().astype(np.float64)

    split, ros, tor, gs = oracle.moe_permute(w.topk_experts, w.topk_gates, w.E)
    x_sorted = w.x_tokens[tor]
    toks = _tokens(w, name)
    rows = ros[toks].reshape(-1)
    o1q, o1s = oracle.quantize_rowwise(w.w1)
    o2q, o2s = oracle.quantize_rowwise(w.w2)
    o2tq, o2ts = oracle.quantize_transposed(w.w2, w.E)
    o1tq, o1ts = oracle.quantize_transposed(w.w1, w.E)
    y_ref, _, _ = oracle.grouped_mlp_rows(x_sorted, split, gs, o1q, o1s, o2q, o2s, rows, want_intermediate=False)
    out_ref = y_ref.reshape(len(toks), w.topk, w.H).sum(axis=1)
    rdx, rdg, _, _ = oracle.grouped_mlp_bwd_rows(x_sorted, split, gs, o1q, o1s, o2tq, o2ts, o1tq, o1ts,
                                                 d_out[tor], rows)
    dx_ref = rdx.reshape(len(toks), w.topk, w.H).sum(axis=1)
    dg_ref = rdg.reshape(len(toks), w.topk)
    for what, got, ref in (("forward (training)", out[toks], out_ref), ("forward", out_inf[toks], out_ref),
                           ("dx", dx[toks], dx_ref), ("d gates", dg[toks], dg_ref)):
        rel, mxe = G.y_errors(got, ref)
        assert rel <= G.Y_REL_TOL and mxe <= G.Y_MAX_TOL, f"{what}: rel {rel:.3e} max {mxe:.3e}"


def test_ep_layer_without_tokens(mx, nccl_group):
    """A rank with no tokens (T = 0, so it also owns no routed rows): the expert-parallel layer's
    forward, training forward and backward run through the empty exchanges and return empty
    outputs; the weight gradients are None (no row reached the rank's experts) or zero."""
    import torch
    from mxfp8_block_scaled_03_gb300 import ep
    w = W.moe_workload("tiny")
    x = torch.zeros((0, w.H), dtype=torch.bfloat16, device="cuda")
    ex = torch.zeros((0, w.topk), dtype=torch.int32, device="cuda")
    g = torch.zeros((0, w.topk), dtype=torch.float32, device="cuda")
    wts = _weights(mx, w)
    w1t = mx.mxfp8_quantize_colwise_t(G.to_dev_bf16(w.w1))
    w2t = mx.mxfp8_quantize_colwise_t(G.to_dev_bf16(w.w2))
    out = ep.ep_moe_forward(x, ex, g, wts, w.E)
    out_t, ctx = ep.ep_moe_forward_train(x, ex, g, wts, w.E)
    dx, dg, dw1, dw2 = ep.ep_moe_backward(torch.zeros((0, w.H), dtype=torch.bfloat16, device="cuda"), ctx,
                                          (w1t[0], w1t[1], w2t[0], w2t[1]))
    torch.cuda.synchronize()
    assert tuple(out.shape) == (0, w.H) and tuple(out_t.shape) == (0, w.H) and tuple(dx.shape) == (0, w.H)
    assert dg.numel() == 0
    for dw in (dw1, dw2):
        assert dw is None or not bool(dw.any())
