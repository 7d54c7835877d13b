"""Pins of the oracle's NVFP4 variant (oracle/nvfp4_oracle.c).

Reading (the Llama 3 recipe page names NVFP4 as a quantized-training recipe, feature table and
section "Quantized Training (FP8 / MXFP8 / NVFP4)", without defining it): NVIDIA's published
NVFP4 -- E2M1 elements, one E4M3 scale per 16 values, a per-tensor binary32 encode scale
s_enc = 448 * 6 / amax.  What pins each part:
  - the E2M1 codec: the 16 codes against the format's value table; the encoder against an
    independent nearest-value search on every binary32 value with up to 12 significant bits in
    the range, all midpoints and their binary32 neighbours, and random values;
  - the block rule: hand-worked blocks (tests/golden/nvfp4_blocks.txt, derivations in the file);
  - invariants: power-of-two scaling of a tensor leaves codes and block scales unchanged (only
    s_enc moves), sign symmetry, exact round trips for values on the scaled E2M1 grid;
  - the MLP: with E = 1 it equals a textbook dense SwiGLU MLP in torch float64 on the same
    dequantized operands; a ragged three-expert case with an empty expert against correctly
    rounded sums (math.fsum); doubling the routing weights doubles y exactly (the gate is
    applied before the intermediate is quantized); rows reordered within an expert reorder y.
"""
import math
import os

import numpy as np
import pytest
import torch

from mxfp8_block_scaled_03_gb300 import workloads as W
from tests import _independent as ind

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_blocks.txt")


def test_e2m1_code_table(oracle):
    vals = [oracle.lib().ora_e2m1_decode(c) for c in range(16)]
    assert vals[:8] == list(ind.E2M1_MAGNITUDES)
    assert vals[8:] == [-v for v in ind.E2M1_MAGNITUDES]
    assert math.copysign(1.0, vals[8]) == -1.0
    for c in range(16):
        assert oracle.lib().ora_e2m1_encode(vals[c]) == c


def test_e2m1_encoder_matches_search(oracle):
    # every binary32 value in [2^-4, 8) with at most 12 significant bits, both signs
    m = np.arange(2048, 4096, dtype=np.float64)
    grid = np.concatenate([m * 2.0 ** (e - 11) for e in range(-4, 3)])
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0])
    f32 = lambda v: np.asarray(v, dtype=np.float32)
    near = np.concatenate([np.nextafter(f32(mids), f32(0)), f32(mids), np.nextafter(f32(mids), f32(9))]).astype(np.float64)
    rng = np.random.default_rng(3)
    rnd = rng.uniform(0, 10, 200000).astype(np.float32).astype(np.float64)
    vals = np.concatenate([grid, near, rnd, [0.0, 6.0, 100.0, 1e30]])
    vals = np.concatenate([vals, -vals])
    assert np.array_equal(oracle.e2m1_encode(vals), ind.e2m1_nearest_code(vals))
    assert oracle.e2m1_encode(np.array([-0.0]))[0] == 0x8


def _golden_cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {"name": rest, "values": np.zeros(16, dtype=np.float32), "codes": np.zeros(16, dtype=np.uint8)}
            cases.append(cur)
        elif key == "senc":
            cur["senc"] = rest
        elif key == "values":
            for tok in rest.split():
                i, v = tok.split(":")
                cur["values"][int(i)] = np.float32(float(v))
        elif key == "sf":
            cur["sf"] = int(rest, 16)
        elif key == "codes":
            for tok in rest.split():
                i, v = tok.split(":")
                cur["codes"][int(i)] = int(v, 16)
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_blocks(oracle, case):
    if case["senc"] == "tensor":
        bits = W.bf16_bits(case["values"])
        assert np.array_equal(W.bf16_to_f32(bits), case["values"])      # the values are exact in bf16
        q, sf, s_enc = oracle.nvfp4_quantize_rowwise(bits[None, :])
        codes, sfc = q[0], int(sf[0, 0])
    else:
        codes, sfc = oracle.nvfp4_quantize_block(case["values"], float(case["senc"]))
    assert sfc == case["sf"], hex(sfc)
    assert np.array_equal(codes, case["codes"]), codes


def test_encode_scale(oracle):
    assert oracle.nvfp4_encode_scale(6.0) == 448.0
    assert oracle.nvfp4_encode_scale(0.0) == 1.0
    assert oracle.nvfp4_encode_scale(2.0 ** -130) == float(np.finfo(np.float32).max)
    assert oracle.nvfp4_encode_scale(2688.0) == 1.0


def _tensor(rng, M, K, scale=1.0):
    return W.bf16_bits((rng.standard_normal((M, K)) * scale).astype(np.float32))


def test_power_of_two_scaling_moves_only_the_tensor_scale(oracle):
    rng = np.random.default_rng(4)
    x = _tensor(rng, 8, 64)
    xf = W.bf16_to_f32(x)
    q0, s0, e0 = oracle.nvfp4_quantize_rowwise(x)
    for k in (-20, -3, 1, 7, 30):
        q, s, e = oracle.nvfp4_quantize_rowwise(W.bf16_bits(xf * np.float32(2.0 ** k)))
        assert np.array_equal(q, q0) and np.array_equal(s, s0)
        assert e == e0 * 2.0 ** -k


def test_sign_symmetry(oracle):
    rng = np.random.default_rng(5)
    x = _tensor(rng, 4, 128)
    q0, s0, e0 = oracle.nvfp4_quantize_rowwise(x)
    q1, s1, e1 = oracle.nvfp4_quantize_rowwise(x ^ np.uint16(0x8000))
    assert np.array_equal(q1, q0 ^ 0x8) and np.array_equal(s1, s0) and e1 == e0


def test_values_on_the_scaled_grid_round_trip(oracle):
    # every block holds 6 * 2^m (the tensor amax), so s_enc = 448 * 2^-m, every block scale is
    # 448 and r = 2^-m: values q * 2^m with q on the E2M1 grid come back exactly
    rng = np.random.default_rng(6)
    for m in (-3, 0, 5):
        g = ind.e2m1_value(rng.integers(0, 16, size=(6, 64)))
        g[:, ::16] = 6.0
        xf = (g * 2.0 ** m).astype(np.float32)
        q, sf, s_enc = oracle.nvfp4_quantize_rowwise(W.bf16_bits(xf))
        assert s_enc == 448.0 * 2.0 ** -m and np.all(sf == 0x7E)
        assert np.array_equal(oracle.nvfp4_dequantize(q, sf, s_enc), xf.astype(np.float64))


def _weights(oracle, w):
    return oracle.nvfp4_quantize_rowwise(w.w1), oracle.nvfp4_quantize_rowwise(w.w2)


def _deq(q, sf, s):
    """Dequantization through the independent tables (E2M1 by the format, E4M3 by torch)."""
    S = ind.torch_e4m3_values()[np.asarray(sf, dtype=np.int64)]
    return ind.e2m1_value(q) * np.repeat(S, 16, axis=-1) / np.float64(np.float32(s))


def test_dense_single_expert_equals_textbook_mlp(oracle):
    w = W.custom_moe([40], H=64, F=96, seed=21, with_gates=False)
    (w1q, w1s, s1), (w2q, w2s, s2) = _weights(oracle, w)
    h_amax = 3.0
    y, hq, hsf, s_x = oracle.nvfp4_grouped_mlp_rows(w.x_sorted, w.split_sizes, None, (w1q, w1s, s1),
                                                    (w2q, w2s, s2), h_amax, np.arange(w.R))
    xq, xs, s_x2 = oracle.nvfp4_quantize_rowwise(w.x_sorted)
    assert s_x == s_x2
    T = torch.from_numpy
    a = T(_deq(xq, xs, s_x))
    W1 = T(_deq(w1q, w1s, s1))
    W2 = T(_deq(w2q, w2s, s2))
    F = w.F
    g, u = a @ W1[:F].T, a @ W1[F:].T
    h = (torch.nn.functional.silu(g) * u).numpy().astype(np.float32)
    s_h = oracle.nvfp4_encode_scale(h_amax)
    hq2, hsf2 = oracle.nvfp4_quantize_f32(h, s_h)
    assert np.array_equal(hq, hq2) and np.array_equal(hsf, hsf2)
    y2 = (T(_deq(hq2, hsf2, s_h)) @ W2.T).numpy()
    np.testing.assert_allclose(y, y2, rtol=1e-12, atol=1e-12 * np.abs(y2).max())


def test_ragged_bruteforce_exact_sums(oracle):
    w = W.custom_moe([7, 0, 33], H=32, F=48, seed=22)
    (w1q, w1s, s1), (w2q, w2s, s2) = _weights(oracle, w)
    h_amax = 0.5
    rows = np.arange(w.R)
    y, hq, hsf, s_x = oracle.nvfp4_grouped_mlp_rows(w.x_sorted, w.split_sizes, w.gates, (w1q, w1s, s1),
                                                    (w2q, w2s, s2), h_amax, rows)
    xq, xs, _ = oracle.nvfp4_quantize_rowwise(w.x_sorted)
    a = _deq(xq, xs, s_x)
    W1 = _deq(w1q, w1s, s1)
    W2 = _deq(w2q, w2s, s2)
    s_h = oracle.nvfp4_encode_scale(h_amax)
    off = np.concatenate([[0], np.cumsum(w.split_sizes)])
    F, H = w.F, w.H
    for r in rows:
        e = int(np.searchsorted(off, r, side="right") - 1)
        g = [math.fsum(a[r] * W1[e * 2 * F + j]) for j in range(F)]
        u = [math.fsum(a[r] * W1[e * 2 * F + F + j]) for j in range(F)]
        h = np.array([float(w.gates[r]) * ind.silu(gj) * uj for gj, uj in zip(g, u)], dtype=np.float32)
        q, s = oracle.nvfp4_quantize_f32(h[None, :], s_h)
        assert np.array_equal(q[0], hq[r]) and np.array_equal(s[0], hsf[r])
        hd = _deq(q, s, s_h)[0]
        yr = np.array([math.fsum(hd * W2[e * H + i]) for i in range(H)])
        np.testing.assert_allclose(y[r], yr, rtol=1e-13, atol=1e-13 * np.abs(yr).max())


def test_doubled_gates_double_the_output(oracle):
    w = W.custom_moe([30, 20], H=64, F=64, seed=23)
    w.gates[:] = np.maximum(w.gates, 0.5)
    wq = _weights(oracle, w)
    rows = np.arange(w.R)
    # an encode scale for h that keeps every block scale, doubled or not, in E4M3's normal range
    # (there, doubling commutes with rounding): h_amax = 4 x the largest |h|
    _, hq0, hsf0, _ = oracle.nvfp4_grouped_mlp_rows(w.x_sorted, w.split_sizes, w.gates, *wq, 1.0, rows)
    h_amax = 4 * float(np.abs(oracle.nvfp4_dequantize(hq0, hsf0, oracle.nvfp4_encode_scale(1.0))).max())
    y1, hq1, hsf1, _ = oracle.nvfp4_grouped_mlp_rows(w.x_sorted, w.split_sizes, w.gates, *wq, h_amax, rows)
    y2, hq2, hsf2, _ = oracle.nvfp4_grouped_mlp_rows(w.x_sorted, w.split_sizes, w.gates * 2, *wq, h_amax, rows)
    assert np.all((hsf1 & 0x78) != 0) and np.all(hsf2 <= 0x7E)
    assert np.array_equal(hq1, hq2)                        # same codes, block scales one binade up
    assert np.array_equal(ind.torch_e4m3_values()[hsf2], 2 * ind.torch_e4m3_values()[hsf1])
    assert np.array_equal(y2, 2 * y1)


def test_row_order_and_empty_experts(oracle):
    w = W.custom_moe([9, 0, 14], H=32, F=32, seed=24)
    wq = _weights(oracle, w)
    rows = np.arange(w.R)
    y, _, _, _ = oracle.nvfp4_grouped_mlp_rows(w.x_sorted, w.split_sizes, w.gates, *wq, 1.0, rows)
    perm = np.concatenate([np.arange(9)[::-1], 9 + np.random.default_rng(1).permutation(14)])
    yp, _, _, _ = oracle.nvfp4_grouped_mlp_rows(w.x_sorted[perm], w.split_sizes, w.gates[perm], *wq, 1.0, rows)
    assert np.array_equal(yp, y[perm])
    with pytest.raises(ValueError):
        oracle.nvfp4_grouped_mlp_rows(w.x_sorted, np.array([9, 1, 14], dtype=np.int32), w.gates, *wq, 1.0, rows)
