"""Pins of the oracle's dispatch (stable sort of (token, slot) pairs by expert) and combine.

Page "Efficient MoE training for biological foundation models": section "Dense vs. MoE scaling"
(each token uses a few experts) and Key technical approaches item 1 (GroupedLinear on tokens
gathered per expert, with per-expert counts split_sizes)."""
import numpy as np
import pytest

from mxfp8_block_scaled_03_gb300 import workloads as W


def test_permute_equals_numpy_stable_argsort(oracle):
    rng = np.random.default_rng(1)
    T, k, E = 777, 3, 13
    ex = rng.integers(0, E, size=(T, k)).astype(np.int32)
    g = rng.random((T, k)).astype(np.float32)
    split, ros, tor, gs = oracle.moe_permute(ex, g, E)
    order = np.argsort(ex.reshape(-1), kind="stable")      # library sort, independent of the oracle
    assert np.array_equal(split, np.bincount(ex.reshape(-1), minlength=E))
    assert np.array_equal(tor, order // k)
    assert np.array_equal(gs, g.reshape(-1)[order])
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    assert np.array_equal(ros.reshape(-1), inv)


def test_permute_invariants_with_empty_experts(oracle):
    rng = np.random.default_rng(2)
    T, k, E = 300, 8, 64
    keys = rng.random((T, E)) + (np.arange(E) >= 61) * -10.0     # experts 61..63 never chosen
    ex = np.argsort(-keys, axis=1)[:, :k].astype(np.int32)
    split, ros, tor, _ = oracle.moe_permute(ex, None, E)
    assert split[61:].sum() == 0 and split.sum() == T * k
    assert sorted(ros.reshape(-1).tolist()) == list(range(T * k))            # a bijection
    assert np.array_equal(tor[ros], np.repeat(np.arange(T), k).reshape(T, k))
    off = np.concatenate([[0], np.cumsum(split)])
    for e in range(E):                                                        # (token, slot) order kept
        seg = [(t, j) for t in range(T) for j in range(k) if ex[t, j] == e]
        assert [ros[t, j] for t, j in seg] == list(range(off[e], off[e + 1]))


def test_permute_matches_workload_routing(oracle):
    w = W.moe_workload("tiny")
    split, _, tor, gs = oracle.moe_permute(w.topk_experts, w.topk_gates, w.E)
    assert np.array_equal(split, w.split_sizes) and np.array_equal(tor, w.token_of_row)
    assert np.array_equal(gs, w.gates)


def test_permute_rejects_bad_expert(oracle):
    with pytest.raises(ValueError):
        oracle.moe_permute(np.array([[0, 5]], dtype=np.int32), None, 4)


def test_combine_sums_the_token_rows(oracle):
    rng = np.random.default_rng(3)
    T, k, H = 50, 2, 16
    y = rng.standard_normal((T * k, H))
    ros = rng.permutation(T * k).reshape(T, k).astype(np.int32)
    out = oracle.moe_combine(y, ros)
    for t in range(T):
        assert np.array_equal(out[t], y[ros[t, 0]] + y[ros[t, 1]])
    assert np.array_equal(oracle.moe_combine(y, np.arange(T * k, dtype=np.int32).reshape(T * k, 1)), y)
