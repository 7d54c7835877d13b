"""GPU parity of the grouped-MLP backward (grouped_mlp_fwd_train + grouped_mlp_bwd) and of the
transposed column-wise quantize against the oracle.

Page "Efficient MoE training for biological foundation models", Key technical approaches item 3
(the fused op's corresponding backward).  The oracle computes the same reading in binary64; the
GPU accumulates in fp32, so every tensor both sides quantize agrees except for rare codes whose
input lies within fp32 rounding of a rounding boundary.  Bars (same as the forward's y):
||out - ref|| / ||ref|| <= 5e-3 and max|out - ref| <= 1e-2 * max|ref| for dx, dgates and the
weight-gradient entries; weight gradients of experts without rows are exactly zero; the
transposed quantize is bit-exact.
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
    return t.float().cpu().numpy().astype(np.float64)


def _gpu_bwd(mx, w, dy_bits):
    import torch
    x = G.to_dev_bf16(w.x_sorted)
    split = G.to_dev(w.split_sizes)
    g = G.to_dev(w.gates) if w.gates is not None else None
    w1 = G.to_dev_bf16(w.w1)
    w2 = G.to_dev_bf16(w.w2)
    w1q, w1s, _, _ = mx.mxfp8_quantize(w1, sf_layout=mx.SF_MMA)
    w2q, w2s, _, _ = mx.mxfp8_quantize(w2, sf_layout=mx.SF_MMA)
    w1tq, w1ts = mx.mxfp8_quantize_colwise_t(w1)
    w2tq, w2ts = mx.mxfp8_quantize_colwise_t(w2)
    fws = torch.empty(mx.grouped_mlp_workspace_size(w.R, w.H, w.F, w.E), dtype=torch.uint8, device="cuda")
    y, saved = mx.grouped_mlp_fwd_train(x, split, g, w1q, w1s, w2q, w2s, workspace=fws)
    assert mx.mxfp8_check_device_error(fws) == (0, 0)
    dx, dg, dw1, dw2, ws = mx.grouped_mlp_bwd(x, split, g, saved, w1tq, w1ts, w2tq, w2ts, G.to_dev_bf16(dy_bits))
    st, bits = mx.mxfp8_check_device_error(ws)
    assert st == 0, f"device error word {bits:#x}"
    return _np(dx), _np(dg), _np(dw1), _np(dw2), y, ws


def _oracle_weights(oracle, w):
    o1q, o1s = oracle.quantize_rowwise(w.w1)
    o2tq, o2ts = oracle.quantize_transposed(w.w2, w.E)
    o1tq, o1ts = oracle.quantize_transposed(w.w1, w.E)
    return o1q, o1s, o2tq, o2ts, o1tq, o1ts


def _check(name, got, ref):
    rel, mxe = G.y_errors(np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64))
    assert rel <= G.Y_REL_TOL and mxe <= G.Y_MAX_TOL, f"{name}: rel {rel:.3e} max {mxe:.3e}"
    return rel, mxe


def _dy(w, seed):
    rng = np.random.default_rng(seed)
    return W.bf16_bits(rng.standard_normal((w.R, w.H)).astype(np.float32))


def _entries(rng, w, which, n, nonempty):
    e = rng.choice(nonempty, n)
    A, B = (w.H, w.F) if which == 2 else (2 * w.F, w.H)
    return np.stack([e, rng.integers(0, A, n), rng.integers(0, B, n)], axis=1)


def _padded_rows(w, rows):
    off = np.concatenate([[0], np.cumsum(w.split_sizes)])
    pad = np.concatenate([[0], np.cumsum(256 * ((w.split_sizes + 255) // 256))])
    e = np.searchsorted(off, rows, side="right") - 1
    return pad[e] + (rows - off[e])


def _check_bf16_rows(name, got_bits, ref_bits):
    """bf16 tensors handed between the backward GEMMs: the GPU's fp32 sums and its saved bf16
    pre-activations can round the other way from the oracle's binary64 near a rounding
    boundary, so >= 99.5% of the elements must be bit-equal and the whole must meet the y bars."""
    frac = float(np.mean(got_bits != ref_bits))
    assert frac <= 5e-3, f"{name}: {frac:.2e} of the elements differ"
    _check(name, W.bf16_to_f32(got_bits), W.bf16_to_f32(ref_bits))


def _assert_bwd_parity(mx, oracle, w, rows, n_entries, seed=0):
    dyb = _dy(w, seed)
    dx, dg, dw1, dw2, _, ws = _gpu_bwd(mx, w, dyb)
    ow = _oracle_weights(oracle, w)
    rdx, rdg, rdgu, rh = oracle.grouped_mlp_bwd_rows(w.x_sorted, w.split_sizes, w.gates, *ow, dyb, rows)
    _check("dx", dx[rows], rdx)
    if w.gates is not None:
        _check("dgates", dg[rows], rdg)
    # the bf16 [dG | dU] and h the dh GEMM's epilogue wrote, element by element
    lay = mx.grouped_mlp_bwd_workspace_layout(w.R, w.H, w.F, w.E)
    r_pad, F = lay[3], w.F
    prow = _padded_rows(w, rows)
    wsn = ws.cpu().numpy()
    dgu = wsn[lay[1]:lay[1] + r_pad * 2 * F * 2].view(np.uint16).reshape(r_pad, 2 * F)[prow]
    hb = wsn[lay[2]:lay[2] + r_pad * F * 2].view(np.uint16).reshape(r_pad, F)[prow]
    _check_bf16_rows("dGU", dgu, rdgu)
    _check_bf16_rows("h", hb, rh)
    rng = np.random.default_rng(seed + 1)
    nonempty = np.nonzero(w.split_sizes)[0]
    for which, dw in ((2, dw2), (1, dw1)):
        ent = _entries(rng, w, which, n_entries, nonempty)
        ref = oracle.grouped_mlp_bwd_dw(w.x_sorted, w.split_sizes, w.gates, *ow[:4], dyb, which, ent)
        _check(f"dW{which}", dw[ent[:, 0], ent[:, 1], ent[:, 2]], ref)
    for e in np.nonzero(w.split_sizes == 0)[0]:
        assert not np.any(dw1[e]) and not np.any(dw2[e])
    return dx, dg, dw1, dw2


def test_colwise_transposed_quantize_bit_exact(mx, oracle):
    rng = np.random.default_rng(4)
    x = W.bf16_bits((rng.standard_normal((384, 640)) * np.exp(rng.standard_normal((384, 640)))).astype(np.float32))
    q_ref, sf_ref = oracle.quantize_colwise(x)
    q_t, sf_t = mx.mxfp8_quantize_colwise_t(G.to_dev_bf16(x), sf_layout=mx.SF_COMPACT)
    assert np.array_equal(q_t.cpu().numpy(), q_ref.T) and np.array_equal(sf_t.cpu().numpy(), sf_ref.T)
    q_t, sf_t = mx.mxfp8_quantize_colwise_t(G.to_dev_bf16(x), sf_layout=mx.SF_MMA)
    assert np.array_equal(q_t.cpu().numpy(), q_ref.T)
    assert np.array_equal(G.sf_mma_to_compact(sf_t.cpu().numpy(), 640, 384 // 32), sf_ref.T)


def test_tiny_backward_all_rows(mx, oracle):
    w = W.moe_workload("tiny")
    _assert_bwd_parity(mx, oracle, w, np.arange(w.R), 1500)


def test_ragged_backward_with_empty_experts(mx, oracle):
    w = W.custom_moe([0, 300, 0, 45, 211, 1], H=256, F=256, seed=21)
    _assert_bwd_parity(mx, oracle, w, np.arange(w.R), 800, seed=3)


def test_backward_half_last_column_tile(mx, oracle):
    """F % 256 == 128: the last 256-wide column tile of dh and dW2 is half past the end."""
    w = W.custom_moe([100, 0, 200, 3], H=256, F=384, seed=25)
    _assert_bwd_parity(mx, oracle, w, np.arange(w.R), 800, seed=9)


def test_backward_without_gates(mx, oracle):
    w = W.custom_moe([130, 126], H=512, F=256, seed=22, with_gates=False)
    _assert_bwd_parity(mx, oracle, w, np.arange(w.R), 600, seed=5)


def test_backward_deterministic(mx):
    w = W.custom_moe([70, 190], H=256, F=256, seed=23)
    dyb = _dy(w, 7)
    a = _gpu_bwd(mx, w, dyb)
    b = _gpu_bwd(mx, w, dyb)
    for u, v in zip(a[:4], b[:4]):
        assert np.array_equal(u, v)


def test_fine_grained_backward_sampled(mx, oracle):
    """Full fine-grained workload (64 experts, 3 of them empty, top-8, F = 1408 = 5.5 x 256):
    sampled rows (per expert the first and last 8, 8 random, and both sides of every 128-row tile
    boundary) and weight-gradient entries against the oracle, zero gradients of the empty
    experts."""
    w = W.moe_workload("fine")
    rows = W.sample_rows(w.split_sizes, seed=1, first=8, last=8, rand=8, tile=128)
    _assert_bwd_parity(mx, oracle, w, rows, 160, seed=11)


def test_backward_rejects_unsupported_shapes(mx):
    import torch
    w = W.custom_moe([64], H=384, F=256, seed=24)
    x = G.to_dev_bf16(w.x_sorted)
    z = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.MXFP8Error) as ei:
        mx.grouped_mlp_bwd(x, G.to_dev(w.split_sizes), None, z, z, z, z.view(256, -1), z, x,
                           workspace=torch.zeros(1 << 10, dtype=torch.uint8, device="cuda"))
    assert ei.value.status == mx.ERR_UNSUPPORTED


def test_mixtral_backward_sampled(mx, oracle):
    """Full Mixtral-shaped layer (R=32768, H=4096, F=14336, E=8) in the launch configuration the
    bench times; the oracle checks sampled rows (per expert the first and last 8, 8 random, and
    both sides of every 128-row tile boundary) of dx, dgates, dGU and h, and sampled
    weight-gradient entries."""
    w = W.moe_workload("mixtral")
    rows = W.sample_rows(w.split_sizes, seed=0, first=8, last=8, rand=8, tile=128)
    _assert_bwd_parity(mx, oracle, w, rows, 160)
