"""Pins of the oracle's grouped expert-MLP forward.

Page "Efficient MoE training for biological foundation models", Key technical approaches:
item 1 (GroupedLinear over per-expert token counts split_sizes), item 2 (MXFP8 blocks of 32),
item 3 (GroupedLinear -> ScaledSwiGLU -> GroupedLinear fused into one op that applies the
routing weight with the SwiGLU activation and keeps the intermediate in 8 bits).
"""
import math

import numpy as np
import pytest
import torch

from mxfp8_block_scaled_03_gb300 import workloads as W
from tests import _independent as ind


def _oracle_weights(oracle, w):
    q1, s1 = oracle.quantize_rowwise(w.w1)
    q2, s2 = oracle.quantize_rowwise(w.w2)
    return q1, s1, q2, s2


def _run(oracle, w, rows=None, gates="same"):
    q1, s1, q2, s2 = _oracle_weights(oracle, w)
    rows = np.arange(w.R) if rows is None else rows
    g = w.gates if isinstance(gates, str) else gates
    return oracle.grouped_mlp_rows(w.x_sorted, w.split_sizes, g, q1, s1, q2, s2, rows)


def test_single_expert_equals_dense_swiglu_mlp(oracle):
    """E=1 with gate 1 is the dense MLP y = W2 (silu(W1g x) * (W1u x)), computed here with
    torch float64 matmuls on operands quantized by the independent search-based quantizer."""
    w = W.custom_moe([70], H=128, F=96, seed=21, with_gates=False)
    y, hq, hsf = _run(oracle, w)
    xf = W.bf16_to_f32(w.x_sorted).astype(np.float64)
    xq, xs = ind.quantize_rows_bruteforce(xf)
    w1q, w1s = ind.quantize_rows_bruteforce(W.bf16_to_f32(w.w1).astype(np.float64))
    w2q, w2s = ind.quantize_rows_bruteforce(W.bf16_to_f32(w.w2).astype(np.float64))
    a = torch.from_numpy(ind.decode(xq, xs))
    w1 = torch.from_numpy(ind.decode(w1q, w1s))
    w2 = torch.from_numpy(ind.decode(w2q, w2s))
    F = w.F
    G = a @ w1[:F].T
    U = a @ w1[F:].T
    h = (G / (1.0 + torch.exp(-G))) * U
    hq_ref, hs_ref = ind.quantize_rows_bruteforce(h.numpy())
    y_ref = torch.from_numpy(ind.decode(hq_ref, hs_ref)) @ w2.T
    assert np.array_equal(hsf, hs_ref)
    assert np.array_equal(hq, hq_ref)
    rel = np.linalg.norm(y - y_ref.numpy()) / np.linalg.norm(y_ref.numpy())
    assert rel < 1e-12


def test_bruteforce_exact_sums_tiny(oracle):
    """Per-element evaluation with correctly rounded sums (math.fsum) on a tiny ragged MoE,
    including an empty expert and routing weights."""
    w = W.custom_moe([13, 0, 27], H=64, F=64, seed=22)
    y, hq, hsf = _run(oracle, w)
    F, H = w.F, w.H
    xq, xs = ind.quantize_rows_bruteforce(W.bf16_to_f32(w.x_sorted).astype(np.float64))
    a = ind.decode(xq, xs)
    w1q, w1s = ind.quantize_rows_bruteforce(W.bf16_to_f32(w.w1).astype(np.float64))
    w2q, w2s = ind.quantize_rows_bruteforce(W.bf16_to_f32(w.w2).astype(np.float64))
    w1 = ind.decode(w1q, w1s)
    w2 = ind.decode(w2q, w2s)
    off = np.concatenate([[0], np.cumsum(w.split_sizes)])
    for r in range(w.R):
        e = int(np.searchsorted(off, r, side="right") - 1)
        h = np.empty(F)
        for j in range(F):
            g = math.fsum(a[r, k] * w1[e * 2 * F + j, k] for k in range(H))
            u = math.fsum(a[r, k] * w1[e * 2 * F + F + j, k] for k in range(H))
            h[j] = float(w.gates[r]) * ind.silu(g) * u
        hq_r, hs_r = ind.quantize_rows_bruteforce(h[None, :])
        assert np.array_equal(hq[r], hq_r[0]) and np.array_equal(hsf[r], hs_r[0])
        hd = ind.decode(hq_r, hs_r)[0]
        y_r = np.array([math.fsum(hd[j] * w2[e * H + i, j] for j in range(F)) for i in range(H)])
        assert np.max(np.abs(y[r] - y_r)) <= 1e-12 * max(1e-300, np.max(np.abs(y_r)))


def test_one_hot_weights_closed_form(oracle):
    """Gate row j picks x_j, up row j picks 0.5*x_(j+1), W2 row i picks 2*h_(pi_e(i)):
    h_j = gate * silu(x_j) * 0.5 * x_(j+1) and y_i = 2 * hq_(pi_e(i)) exactly.  A swapped gate/up
    half, a transposed operand or a wrong expert index all change the result."""
    H = F = 64
    E = 2
    split = np.array([9, 6], dtype=np.int32)
    R = int(split.sum())
    rng = np.random.default_rng(23)
    x = W.bf16_bits(rng.standard_normal((R, H)).astype(np.float32))
    w1 = np.zeros((E * 2 * F, H), dtype=np.float32)
    w2 = np.zeros((E * H, F), dtype=np.float32)
    perms = [rng.permutation(F) for _ in range(E)]
    for e in range(E):
        for j in range(F):
            w1[e * 2 * F + j, j] = 1.0
            w1[e * 2 * F + F + j, (j + 1) % H] = 0.5
        for i in range(H):
            w2[e * H + i, perms[e][i]] = 2.0
    gates = rng.uniform(0.1, 1.0, R).astype(np.float32)
    inp = W.MoEInputs("onehot", R, 1, E, H, F, x, split, gates, W.bf16_bits(w1), W.bf16_bits(w2),
                      np.arange(R))
    y, hq, hsf = _run(oracle, inp)
    xq, xs = ind.quantize_rows_bruteforce(W.bf16_to_f32(x).astype(np.float64))
    a = ind.decode(xq, xs)
    for r in range(R):
        e = 0 if r < split[0] else 1
        h = np.array([float(gates[r]) * ind.silu(a[r, j]) * (0.5 * a[r, (j + 1) % H]) for j in range(F)])
        hq_r, hs_r = ind.quantize_rows_bruteforce(h[None, :])
        assert np.array_equal(hq[r], hq_r[0])
        hd = ind.decode(hq_r, hs_r)[0]
        assert np.array_equal(y[r], 2.0 * hd[perms[e]])


def test_routing_weight_scales_intermediate_before_requant(oracle):
    """A power-of-two routing weight 2^k shifts the intermediate's E8M0 bytes by k, keeps its
    codes, and scales y by exactly 2^k: the weight multiplies h before requantization."""
    w = W.custom_moe([20, 11], H=64, F=128, seed=24, with_gates=False)
    rng = np.random.default_rng(25)
    k = rng.integers(-3, 4, w.R)
    g = np.ldexp(np.ones(w.R), k).astype(np.float32)
    y1, hq1, hs1 = _run(oracle, w, gates=None)
    y2, hq2, hs2 = _run(oracle, w, gates=g)
    assert np.array_equal(hq1, hq2)
    assert np.array_equal(hs2.astype(int), hs1.astype(int) + k[:, None])
    assert np.array_equal(y2, y1 * np.ldexp(1.0, k)[:, None])


def test_row_order_within_experts_is_irrelevant(oracle):
    w = W.custom_moe([17, 30, 5], H=64, F=64, seed=26)
    y, hq, _ = _run(oracle, w)
    off = np.concatenate([[0], np.cumsum(w.split_sizes)])
    rng = np.random.default_rng(27)
    perm = np.concatenate([off[e] + rng.permutation(int(w.split_sizes[e])) for e in range(3)])
    w2 = W.MoEInputs("perm", w.T, 1, w.E, w.H, w.F, np.ascontiguousarray(w.x_sorted[perm]), w.split_sizes,
                     w.gates[perm], w.w1, w.w2, perm)
    yp, hqp, _ = _run(oracle, w2)
    assert np.array_equal(yp, y[perm])
    assert np.array_equal(hqp, hq[perm])


def test_empty_expert_changes_nothing(oracle):
    w = W.custom_moe([8, 12, 9], H=64, F=64, seed=28)
    y, hq, _ = _run(oracle, w)
    E, F, H = w.E, w.F, w.H
    rng = np.random.default_rng(29)
    junk1 = W.bf16_bits(rng.standard_normal((2 * F, H)).astype(np.float32))
    junk2 = W.bf16_bits(rng.standard_normal((H, F)).astype(np.float32))
    w1 = np.concatenate([w.w1[:2 * F], junk1, w.w1[2 * F:]])
    w2 = np.concatenate([w.w2[:H], junk2, w.w2[H:]])
    wz = W.MoEInputs("zero", w.T, 1, E + 1, H, F, w.x_sorted, np.array([8, 0, 12, 9], dtype=np.int32),
                     w.gates, w1, w2, w.token_of_row)
    yz, hqz, _ = _run(oracle, wz)
    assert np.array_equal(yz, y) and np.array_equal(hqz, hq)


def test_split_sizes_must_cover_rows(oracle):
    w = W.custom_moe([4, 4], H=64, F=64, seed=30)
    q1, s1, q2, s2 = _oracle_weights(oracle, w)
    with pytest.raises(ValueError, match="status 6"):
        oracle.grouped_mlp_rows(w.x_sorted, np.array([4, 3], dtype=np.int32), None, q1, s1, q2, s2, [0])
    with pytest.raises(ValueError, match="status 1"):
        oracle.grouped_mlp_rows(w.x_sorted, np.array([9, -1], dtype=np.int32), None, q1, s1, q2, s2, [0])
