"""Pins of the oracle's backward of the grouped MLP.

Page "Efficient MoE training for biological foundation models", Key technical approaches item 3:
the fused GroupedLinear -> ScaledSwiGLU -> GroupedLinear op has a corresponding fused backward.
The pages do not spell the backward out; the oracle takes the usual MXFP8-training reading
(straight-through gradients, each backward GEMM's operands quantized along its contraction
axis, bf16 hand-off tensors, pre-activations saved by the forward as bf16).  The pins below
check
  - the calculus alone (quantization switched off) against torch.autograd in float64 on a
    ragged problem with an empty expert;
  - the quantization axes, with inputs built so that quantizing along the wrong axis changes
    the result (a large element crushes its block neighbours to zero along one axis only);
  - power-of-two scaling of dy, which MXFP8 and bf16 rounding commute with exactly;
  - the whole quantized backward (every bf16 rounding and every MXFP8 step in its place)
    against an independent torch-float64 restatement with the search quantizer, on a ragged
    problem with an empty expert and partial 32-row blocks.
"""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_03_gb300 import workloads as W
from tests import _independent as ind


def _lossless(rng, shape):
    """Values k * 2^-4 with |k| <= 7: exactly representable under MXFP8 with any blocking."""
    k = rng.integers(-7, 8, size=shape).astype(np.float32)
    return W.bf16_bits(k * np.float32(1.0 / 16))


def _weights(oracle, w1, w2, E):
    w1q, w1s = oracle.quantize_rowwise(w1)
    w2tq, w2ts = oracle.quantize_transposed(w2, E)
    w1tq, w1ts = oracle.quantize_transposed(w1, E)
    return w1q, w1s, w2tq, w2ts, w1tq, w1ts


def _all_entries(E, A, B):
    e, i, j = np.meshgrid(np.arange(E), np.arange(A), np.arange(B), indexing="ij")
    return np.stack([e.ravel(), i.ravel(), j.ravel()], axis=1)


def test_calculus_matches_autograd_without_quantization(oracle):
    rng = np.random.default_rng(0)
    split = np.array([5, 0, 40], dtype=np.int32)
    E, R, H, F = 3, 45, 64, 96
    x = _lossless(rng, (R, H))
    w1 = _lossless(rng, (E * 2 * F, H))
    w2 = _lossless(rng, (E * H, F))
    dy = _lossless(rng, (R, H))
    gates = rng.uniform(0.1, 1.0, R).astype(np.float32)
    wq = _weights(oracle, w1, w2, E)
    dx, dgate, _, _ = oracle.grouped_mlp_bwd_rows(x, split, gates, *wq, dy, np.arange(R), quant=False)
    dw2 = oracle.grouped_mlp_bwd_dw(x, split, gates, *wq[:4], dy, 2, _all_entries(E, H, F), quant=False)
    dw1 = oracle.grouped_mlp_bwd_dw(x, split, gates, *wq[:4], dy, 1, _all_entries(E, 2 * F, H), quant=False)

    t = lambda b: torch.from_numpy(W.bf16_to_f32(b).astype(np.float64))
    X = t(x).requires_grad_()
    W1 = t(w1).reshape(E, 2 * F, H).requires_grad_()
    W2 = t(w2).reshape(E, H, F).requires_grad_()
    Gt = torch.from_numpy(gates.astype(np.float64)).requires_grad_()
    off = np.concatenate([[0], np.cumsum(split)])
    ys = []
    for e in range(E):
        xe = X[off[e]:off[e + 1]]
        g = xe @ W1[e, :F].T
        u = xe @ W1[e, F:].T
        h = Gt[off[e]:off[e + 1], None] * torch.nn.functional.silu(g) * u
        ys.append(h @ W2[e].T)
    (torch.cat(ys) * t(dy)).sum().backward()
    np.testing.assert_allclose(dx, X.grad.numpy(), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dgate, Gt.grad.numpy(), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dw2, W2.grad.numpy().ravel(), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dw1, W1.grad.numpy().ravel(), rtol=1e-11, atol=1e-11)
    assert np.all(dw1.reshape(E, 2 * F, H)[1] == 0) and np.all(dw2.reshape(E, H, F)[1] == 0)


def _colq(values):
    """Column-wise MXFP8 (32-row blocks, zero-padded last block) through the independent
    quantizer: quantize the transposed, zero-padded columns row-wise."""
    n, m = values.shape
    pad = (-n) % 32
    v = np.concatenate([values, np.zeros((pad, m))]) if pad else values
    q, s = ind.quantize_rows_bruteforce(np.ascontiguousarray(v.T))
    return ind.decode(q, s).T[:n]


def test_quantization_axes(oracle):
    rng = np.random.default_rng(1)
    E, R, H, F = 1, 64, 64, 64
    split = np.array([R], dtype=np.int32)
    w1 = _lossless(rng, (2 * F, H))
    w2 = _lossless(rng, (H, F))
    xf = (rng.standard_normal((R, H)) * 0.5).astype(np.float32)
    xf[0, 0], xf[1, 0], xf[0, 1] = 2.0 ** 14, 2.0 ** -6, 2.0 ** -6   # x column 0: row 1 crushed only column-wise
    x = W.bf16_bits(xf)
    dyf = np.zeros((R, H), dtype=np.float32)
    dyf[0, 0], dyf[0, 1], dyf[1, 0] = 2.0 ** 20, 1.0, 1.0            # (0,1) crushed row-wise, (1,0) column-wise
    dy = W.bf16_bits(dyf)
    wq = _weights(oracle, w1, w2, E)
    rows = np.arange(R)
    dx, dgate, dgu, hb = oracle.grouped_mlp_bwd_rows(x, split, None, *wq, dy, rows)

    # dgrad operands are quantized along H: row 1 of dy holds a lone 1 in its row block, so row 1's
    # gradients equal those of a dy that has nothing else
    dy_lone = np.zeros((R, H), dtype=np.float32)
    dy_lone[1, 0] = 1.0
    dx2, dgate2, _, _ = oracle.grouped_mlp_bwd_rows(x, split, None, *wq, W.bf16_bits(dy_lone), rows)
    assert np.array_equal(dx[1], dx2[1]) and dgate[1] == dgate2[1] and dgate[1] != 0

    # weight-gradient operands are quantized along the rows
    hq = _colq(W.bf16_to_f32(hb).astype(np.float64))
    f = np.arange(F)
    dw2_c0 = oracle.grouped_mlp_bwd_dw(x, split, None, *wq[:4], dy, 2, np.stack([0 * f, 0 * f, f], 1))
    dw2_c1 = oracle.grouped_mlp_bwd_dw(x, split, None, *wq[:4], dy, 2, np.stack([0 * f, 0 * f + 1, f], 1))
    assert np.array_equal(dw2_c0, 2.0 ** 20 * hq[0])      # dy[1, 0] is crushed in its column block
    assert np.array_equal(dw2_c1, hq[0])                  # dy[0, 1] survives in its column block
    gq = _colq(W.bf16_to_f32(dgu).astype(np.float64))
    j = np.arange(2 * F)
    dw1_k0 = oracle.grouped_mlp_bwd_dw(x, split, None, *wq[:4], dy, 1, np.stack([0 * j, j, 0 * j], 1))
    assert np.array_equal(dw1_k0, 2.0 ** 14 * gq[0])      # x[1, 0] is crushed in its column block


def test_power_of_two_scaling_of_dy(oracle):
    w = W.moe_workload("tiny")
    rng = np.random.default_rng(2)
    dyf = rng.standard_normal((w.R, w.H)).astype(np.float32)
    wq = _weights(oracle, w.w1, w.w2, w.E)
    rows = np.arange(0, w.R, 7)
    ent2 = np.array([[0, 0, 0], [1, 100, 300], [3, 255, 511], [2, 17, 5]])
    ent1 = np.array([[0, 0, 0], [1, 700, 100], [3, 1023, 255], [2, 511, 3]])
    base = oracle.grouped_mlp_bwd_rows(w.x_sorted, w.split_sizes, w.gates, *wq, W.bf16_bits(dyf), rows)
    scaled = oracle.grouped_mlp_bwd_rows(w.x_sorted, w.split_sizes, w.gates, *wq, W.bf16_bits(dyf * 8), rows)
    assert np.array_equal(scaled[0], 8 * base[0]) and np.array_equal(scaled[1], 8 * base[1])
    for which, ent in ((2, ent2), (1, ent1)):
        a = oracle.grouped_mlp_bwd_dw(w.x_sorted, w.split_sizes, w.gates, *wq[:4], W.bf16_bits(dyf), which, ent)
        b = oracle.grouped_mlp_bwd_dw(w.x_sorted, w.split_sizes, w.gates, *wq[:4], W.bf16_bits(dyf * 8), which, ent)
        assert np.array_equal(b, 8 * a)


def test_bf16_rounding_helper(oracle):
    vals = [1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -3.0e-39, 2.0 ** -133 * 1.5, 123456.789]
    for v in vals:
        ref = float(torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).to(torch.float64))
        assert oracle.round_bf16(v) == ref


def test_rejects_bad_entries(oracle):
    w = W.custom_moe([32], H=64, F=64, seed=3)
    wq = _weights(oracle, w.w1, w.w2, 1)
    dy = np.zeros((32, 64), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.grouped_mlp_bwd_dw(w.x_sorted, w.split_sizes, None, *wq[:4], dy, 2, np.array([[0, 64, 0]]))
    with pytest.raises(ValueError):
        oracle.grouped_mlp_bwd_dw(w.x_sorted, w.split_sizes, None, *wq[:4], dy, 3, np.array([[0, 0, 0]]))


def _rowq(v):
    """Row-wise MXFP8 (blocks of 32 along the last axis) through the independent quantizer."""
    q, s = ind.quantize_rows_bruteforce(np.ascontiguousarray(v, dtype=np.float64))
    return ind.decode(q, s)


def test_quantized_backward_matches_independent_restatement(oracle):
    """The whole quantized backward restated step by step in torch float64 with the independent
    search quantizer and a direct bf16 rounding, on a ragged problem with an empty expert and
    partial 32-row blocks.  Steps, in the reading the oracle documents:
      a = dq(Q_row(x));  g, u = bf16(a W1g^T), bf16(a W1u^T)  (the forward's saved pre-activations)
      dh = dq(Q_row(dy)) W2q   (W2 quantized along H)
      dG = dh gate u silu'(g),  dU = dh gate silu(g),  dgate = sum dh silu(g) u
      dGU = bf16([dG | dU]);  dx = dq(Q_row(dGU)) W1q  (both quantized along 2F)
      h = bf16(gate silu(g) u)
      dW2[e] = dq(Q_col(dy_e))^T dq(Q_col(h_e)),  dW1[e] = dq(Q_col(dGU_e))^T dq(Q_col(x_e))
    Dropping the row-wise quantization of dGU, or moving any bf16 rounding, changes dx, dGU or the
    weight gradients far beyond the 1e-12 bar."""
    rng = np.random.default_rng(7)
    split = np.array([5, 0, 40, 19], dtype=np.int32)
    E, H, F = 4, 64, 64
    R = int(split.sum())
    x = W.bf16_bits(rng.standard_normal((R, H)).astype(np.float32))
    dy = W.bf16_bits(rng.standard_normal((R, H)).astype(np.float32))
    w1 = W.bf16_bits((rng.standard_normal((E * 2 * F, H)) * 0.15).astype(np.float32))
    w2 = W.bf16_bits((rng.standard_normal((E * H, F)) * 0.15).astype(np.float32))
    gates = rng.uniform(0.1, 1.0, R).astype(np.float32)
    wq = _weights(oracle, w1, w2, E)
    rows = np.arange(R)
    dx_o, dgate_o, dgu_o, h_o, gu_o = oracle.grouped_mlp_bwd_rows(x, split, gates, *wq, dy, rows, want_gu=True)
    dw2_o = oracle.grouped_mlp_bwd_dw(x, split, gates, *wq[:4], dy, 2, _all_entries(E, H, F))
    dw1_o = oracle.grouped_mlp_bwd_dw(x, split, gates, *wq[:4], dy, 1, _all_entries(E, 2 * F, H))

    f64 = lambda b: W.bf16_to_f32(b).astype(np.float64)
    xf, dyf = f64(x), f64(dy)
    w1f = f64(w1).reshape(E, 2 * F, H)
    w2f = f64(w2).reshape(E, H, F)
    off = np.concatenate([[0], np.cumsum(split)])
    dx = np.zeros((R, H))
    dgate = np.zeros(R)
    dgu = np.zeros((R, 2 * F))
    hb = np.zeros((R, F))
    gub = np.zeros((R, 2 * F))
    dw2 = np.zeros((E, H, F))
    dw1 = np.zeros((E, 2 * F, H))
    T = torch.from_numpy
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        W1q = _rowq(w1f[e])                   # [2F, H], blocks along H (forward operand)
        W2q_t = _rowq(w2f[e].T)               # [F, H]: W2 quantized along H
        W1q_t = _rowq(w1f[e].T)               # [H, 2F]: W1 quantized along 2F
        a = _rowq(xf[r0:r1])
        g = ind.bf16_round((T(a) @ T(W1q[:F]).T).numpy())
        u = ind.bf16_round((T(a) @ T(W1q[F:]).T).numpy())
        gub[r0:r1] = np.concatenate([g, u], axis=1)
        gt = gates[r0:r1].astype(np.float64)[:, None]
        sig = 1.0 / (1.0 + np.exp(-g))
        s = g * sig
        ds = sig * (1.0 + g * (1.0 - sig))
        dh = (T(_rowq(dyf[r0:r1])) @ T(W2q_t).T).numpy()
        dGU = ind.bf16_round(np.concatenate([dh * gt * u * ds, dh * gt * s], axis=1))
        dgu[r0:r1] = dGU
        dgate[r0:r1] = (dh * s * u).sum(axis=1)
        dx[r0:r1] = (T(_rowq(dGU)) @ T(W1q_t).T).numpy()
        h = ind.bf16_round(gt * s * u)
        hb[r0:r1] = h
        dw2[e] = (T(_colq(dyf[r0:r1])).T @ T(_colq(h))).numpy()
        dw1[e] = (T(_colq(dGU)).T @ T(_colq(xf[r0:r1]))).numpy()

    assert np.array_equal(f64(dgu_o), dgu)
    assert np.array_equal(f64(h_o), hb)
    assert np.array_equal(f64(gu_o), gub)   # the forward's saved pre-activations
    np.testing.assert_allclose(dx_o, dx, rtol=1e-12, atol=1e-12 * np.abs(dx).max())
    np.testing.assert_allclose(dgate_o, dgate, rtol=1e-12, atol=1e-12 * np.abs(dgate).max())
    np.testing.assert_allclose(dw2_o, dw2.ravel(), rtol=1e-12, atol=1e-12 * np.abs(dw2).max())
    np.testing.assert_allclose(dw1_o, dw1.ravel(), rtol=1e-12, atol=1e-12 * np.abs(dw1).max())
    assert np.all(dw1[1] == 0) and np.all(dw2[1] == 0)
