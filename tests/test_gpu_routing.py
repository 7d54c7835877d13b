"""GPU parity of the MoE layer around the grouped MLP: dispatch (moe_permute), the forward that
gathers token rows itself (grouped_mlp_fwd_tokens) and combine (moe_combine).

Page "Efficient MoE training for biological foundation models": Key technical approaches item 1
(tokens gathered per expert, counted by split_sizes) and section "Dense vs. MoE scaling" (each
token uses top-k experts).

Bars: the permutation is integer work, so it is bit-exact against the oracle.  The forward that
gathers rows is the same arithmetic as grouped_mlp_fwd on pre-sorted rows, so its output is
bit-identical to that call and within the forward's tolerances of the oracle.  Combine sums k
bf16 values in fp32 and rounds once to bf16: every element is within half a bf16 step of the
exact sum plus k * 2^-24 of the summed magnitudes.
"""
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


def _np(t):
    return t.cpu().numpy()


def _permute_parity(mx, oracle, ex, g, E):
    import torch
    dg = None if g is None else G.to_dev(g)
    split, ros, tor, gs, ws = mx.moe_permute(G.to_dev(ex), dg, E)
    st, bits = mx.mxfp8_check_device_error(ws)
    assert st == 0, f"device error word {bits:#x}"
    o_split, o_ros, o_tor, o_gs = oracle.moe_permute(ex, g, E)
    assert np.array_equal(_np(split), o_split)
    assert np.array_equal(_np(ros), o_ros)
    assert np.array_equal(_np(tor), o_tor)
    if g is not None:
        assert np.array_equal(_np(gs).view(np.uint32), o_gs.view(np.uint32))
    torch.cuda.synchronize()


@pytest.mark.parametrize("T,k,E,seed", [(1, 1, 1, 0), (5000, 3, 13, 1), (1024, 2, 8, 2), (1025, 1, 1024, 3),
                                        (40000, 8, 64, 4), (3, 4, 1024, 5)])
def test_permute_random_bit_exact(mx, oracle, T, k, E, seed):
    rng = np.random.default_rng(seed)
    ex = rng.integers(0, E, size=(T, k)).astype(np.int32)
    _permute_parity(mx, oracle, ex, rng.random((T, k)).astype(np.float32), E)


def test_permute_skewed_and_without_gates(mx, oracle):
    rng = np.random.default_rng(11)
    ex = np.where(rng.random((9000, 2)) < 0.9, 3, rng.integers(0, 16, size=(9000, 2))).astype(np.int32)
    _permute_parity(mx, oracle, ex, None, 16)


@pytest.mark.parametrize("name", ["tiny", "mixtral", "fine"])
def test_permute_of_workload_routing(mx, oracle, name):
    w = W.moe_workload(name)
    _permute_parity(mx, oracle, w.topk_experts, w.topk_gates, w.E)


def test_permute_empty_tokens(mx):
    import torch
    ex = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    split, _, _, _, ws = mx.moe_permute(ex, None, 5)
    assert _np(split).tolist() == [0] * 5
    assert mx.mxfp8_check_device_error(ws) == (0, 0)


def test_permute_reports_bad_expert(mx):
    ex = np.array([[0, 1], [2, 7], [-1, 0]], dtype=np.int32)
    _, _, _, _, ws = mx.moe_permute(G.to_dev(ex), None, 4)
    st, bits = mx.mxfp8_check_device_error(ws)
    assert st == mx.ERR_INVALID_ARG and bits & 4


def _weights(mx, w):
    w1q, w1s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w1), sf_layout=mx.SF_MMA)
    w2q, w2s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w2), sf_layout=mx.SF_MMA)
    return w1q, w1s, w2q, w2s


def _layer(mx, w):
    """permute -> grouped_mlp_fwd_tokens -> combine on the device; returns host arrays."""
    import torch
    x = G.to_dev_bf16(w.x_tokens)
    split, ros, tor, gs, pws = mx.moe_permute(G.to_dev(w.topk_experts), G.to_dev(w.topk_gates), w.E)
    ws = torch.empty(mx.grouped_mlp_workspace_size(w.R, w.H, w.F, w.E), dtype=torch.uint8, device="cuda")
    y_rows = mx.grouped_mlp_fwd_tokens(x, tor, split, gs, *_weights(mx, w), workspace=ws)
    out = mx.moe_combine(y_rows, ros)
    assert mx.mxfp8_check_device_error(pws)[0] == 0
    st, bits = mx.mxfp8_check_device_error(ws)
    assert st == 0, f"device error word {bits:#x}"
    return _np(y_rows.view(torch.int16)).view(np.uint16), _np(out.view(torch.int16)).view(np.uint16), _np(ros)


def _presorted_y(mx, w):
    import torch
    ws = torch.empty(mx.grouped_mlp_workspace_size(w.R, w.H, w.F, w.E), dtype=torch.uint8, device="cuda")
    y = mx.grouped_mlp_fwd(G.to_dev_bf16(w.x_sorted), G.to_dev(w.split_sizes), G.to_dev(w.gates), *_weights(mx, w),
                           workspace=ws)
    return _np(y.view(torch.int16)).view(np.uint16)


def _combine_bound(y_rows_f64, ros, out_f64):
    terms = np.abs(y_rows_f64[ros]).sum(axis=1)
    exact = y_rows_f64[ros].sum(axis=1)
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(exact), 1e-300))[1] - 8)   # bf16 step at |exact|
    bound = 0.5 * ulp + ros.shape[1] * 2.0 ** -24 * terms
    return np.abs(out_f64 - exact) <= bound * (1 + 1e-12)


def test_tiny_layer_matches_presorted_and_oracle(mx, oracle):
    w = W.moe_workload("tiny")
    y_rows, out, ros = _layer(mx, w)
    assert np.array_equal(y_rows, _presorted_y(mx, w))
    o1q, o1s = oracle.quantize_rowwise(w.w1)
    o2q, o2s = oracle.quantize_rowwise(w.w2)
    y_ref, _, _ = oracle.grouped_mlp_rows(w.x_sorted, w.split_sizes, w.gates, o1q, o1s, o2q, o2s, np.arange(w.R))
    out_ref = oracle.moe_combine(y_ref, ros)
    rel, mxe = G.y_errors(W.bf16_to_f32(out).astype(np.float64), out_ref)
    assert rel <= G.Y_REL_TOL and mxe <= G.Y_MAX_TOL, f"layer out rel {rel:.3e} max {mxe:.3e}"
    yr = W.bf16_to_f32(y_rows).astype(np.float64)
    assert np.all(_combine_bound(yr, ros, W.bf16_to_f32(out).astype(np.float64)))


def test_mixtral_layer_sampled(mx, oracle):
    """Full Mixtral-shaped layer (16384 tokens, top-2 of 8): the gathered forward equals the
    pre-sorted one bit for bit, sampled tokens of the combined output against the oracle."""
    w = W.moe_workload("mixtral")
    y_rows, out, ros = _layer(mx, w)
    assert np.array_equal(y_rows, _presorted_y(mx, w))
    rng = np.random.default_rng(0)
    toks = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, 24, replace=False)]))
    rows = ros[toks].reshape(-1)
    o1q, o1s = oracle.quantize_rowwise(w.w1)
    o2q, o2s = oracle.quantize_rowwise(w.w2)
    y_ref, _, _ = oracle.grouped_mlp_rows(w.x_sorted, w.split_sizes, w.gates, o1q, o1s, o2q, o2s, rows)
    out_ref = y_ref.reshape(len(toks), w.topk, w.H).sum(axis=1)
    rel, mxe = G.y_errors(W.bf16_to_f32(out[toks]).astype(np.float64), out_ref)
    assert rel <= G.Y_REL_TOL and mxe <= G.Y_MAX_TOL, f"layer out rel {rel:.3e} max {mxe:.3e}"
    yr = W.bf16_to_f32(y_rows).astype(np.float64)
    assert np.all(_combine_bound(yr, ros, W.bf16_to_f32(out).astype(np.float64)))


def test_combine_random_rows(mx, oracle):
    import torch
    rng = np.random.default_rng(12)
    T, k, H = 333, 3, 264
    y = W.bf16_bits(rng.standard_normal((T * k + 5, H)).astype(np.float32) * 4)
    ros = rng.permutation(T * k).reshape(T, k).astype(np.int32)
    out = mx.moe_combine(G.to_dev_bf16(y), G.to_dev(ros))
    outf = W.bf16_to_f32(_np(out.view(torch.int16)).view(np.uint16)).astype(np.float64)
    yf = W.bf16_to_f32(y).astype(np.float64)
    assert np.all(_combine_bound(yf, ros, outf))
    ref = oracle.moe_combine(yf, ros)
    assert np.max(np.abs(outf - ref)) <= np.max(np.abs(ref)) * 2.0 ** -7


def test_gather_reports_bad_token(mx):
    import torch
    w = W.custom_moe([40, 24], H=128, F=128, seed=13)
    x = G.to_dev_bf16(w.x_sorted)
    tor = np.arange(64, dtype=np.int32)
    tor[17] = 64
    ws = torch.empty(mx.grouped_mlp_workspace_size(64, 128, 128, 2), dtype=torch.uint8, device="cuda")
    mx.grouped_mlp_fwd_tokens(x, G.to_dev(tor), G.to_dev(w.split_sizes), None, *_weights(mx, w), workspace=ws)
    st, bits = mx.mxfp8_check_device_error(ws)
    assert st == mx.ERR_INVALID_ARG and bits & 8
    mx.grouped_mlp_fwd_tokens(x, G.to_dev(np.arange(64, dtype=np.int32)), G.to_dev(w.split_sizes), None,
                              *_weights(mx, w), workspace=ws)
    assert mx.mxfp8_check_device_error(ws) == (0, 0)


def test_tiny_layer_backward_through_tokens(mx, oracle):
    """The MoE layer in training on the device: permute -> token forward (pre-activations saved)
    -> combine; backward from a token-space output gradient: the token backward (the combine's
    gradient gathers d_out rows by token) -> moe_combine of dx rows (the gather's gradient).
    Checked against the oracle's backward on the sorted rows, combined by the oracle."""
    import torch
    w = W.moe_workload("tiny")
    x = G.to_dev_bf16(w.x_tokens)
    split, ros, tor, gs, _ = mx.moe_permute(G.to_dev(w.topk_experts), G.to_dev(w.topk_gates), w.E)
    w1, w2 = G.to_dev_bf16(w.w1), G.to_dev_bf16(w.w2)
    w1q, w1s, _, _ = mx.mxfp8_quantize(w1, sf_layout=mx.SF_MMA)
    w2q, w2s, _, _ = mx.mxfp8_quantize(w2, sf_layout=mx.SF_MMA)
    w1tq, w1ts = mx.mxfp8_quantize_colwise_t(w1)
    w2tq, w2ts = mx.mxfp8_quantize_colwise_t(w2)
    y_rows, saved = mx.grouped_mlp_fwd_tokens_train(x, tor, split, gs, w1q, w1s, w2q, w2s)
    rng = np.random.default_rng(31)
    d_out = W.bf16_bits(rng.standard_normal((w.T, w.H)).astype(np.float32))
    dx_rows, dg, dw1, dw2, ws = mx.grouped_mlp_bwd_tokens(x, tor, split, gs, saved, w1tq, w1ts, w2tq, w2ts,
                                                          G.to_dev_bf16(d_out))
    assert mx.mxfp8_check_device_error(ws) == (0, 0)
    dx_tok = mx.moe_combine(dx_rows, ros)
    ros_h = _np(ros)
    # oracle: the same rows through the pre-sorted backward, the output gradient gathered by token
    dy_rows = d_out[w.token_of_row]
    o1q, o1s = oracle.quantize_rowwise(w.w1)
    o2tq, o2ts = oracle.quantize_transposed(w.w2, w.E)
    o1tq, o1ts = oracle.quantize_transposed(w.w1, w.E)
    rdx, rdg, _, _ = oracle.grouped_mlp_bwd_rows(w.x_sorted, w.split_sizes, w.gates, o1q, o1s, o2tq, o2ts, o1tq,
                                                 o1ts, dy_rows, np.arange(w.R))
    rdx_tok = oracle.moe_combine(rdx, ros_h)
    got = W.bf16_to_f32(_np(dx_tok.view(torch.int16)).view(np.uint16)).astype(np.float64)
    rel, mxe = G.y_errors(got, rdx_tok)
    assert rel <= G.Y_REL_TOL and mxe <= G.Y_MAX_TOL, f"dx tokens rel {rel:.3e} max {mxe:.3e}"
    rel, mxe = G.y_errors(_np(dg).astype(np.float64)[ros_h], rdg[ros_h])
    assert rel <= G.Y_REL_TOL and mxe <= G.Y_MAX_TOL, f"d gates rel {rel:.3e} max {mxe:.3e}"
    ent = np.array([[0, 0, 0], [1, 100, 300], [2, 255, 511], [3, 17, 5]])
    ref = oracle.grouped_mlp_bwd_dw(w.x_sorted, w.split_sizes, w.gates, o1q, o1s, o2tq, o2ts, dy_rows, 2, ent)
    got = _np(dw2)[ent[:, 0], ent[:, 1], ent[:, 2]]
    assert np.allclose(got, ref, rtol=1e-2, atol=1e-3 * np.abs(ref).max())
