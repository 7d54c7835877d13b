"""GPU parity of grouped_mlp_fwd against the oracle.

Page "Efficient MoE training for biological foundation models", Key technical approaches,
items 1-3: GroupedLinear over split_sizes -> ScaledSwiGLU (routing weight applied with the
activation) -> MXFP8 requantized intermediate -> GroupedLinear.

Tolerances (the GPU accumulates in fp32 and rounds y to bf16, the oracle works in binary64):
  y:   ||y - y_ref|| / ||y_ref|| <= 5e-3 and max|y - y_ref| <= 1e-2 * max|y_ref|
  h_q: dequantized intermediate equal on >= 99.9% of elements, every difference within one
       E4M3 step at the coarser of the two blocks' scales.
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


def _gpu_forward(mx, w, gates=True):
    import torch
    x = G.to_dev_bf16(w.x_sorted)
    w1q, w1s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w1), sf_layout=mx.SF_MMA)
    w2q, w2s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w2), sf_layout=mx.SF_MMA)
    split = G.to_dev(w.split_sizes)
    g = G.to_dev(w.gates) if (gates and w.gates is not None) else None
    ws = torch.empty(mx.grouped_mlp_workspace_size(w.R, w.H, w.F, w.E), dtype=torch.uint8, device="cuda")
    y = mx.grouped_mlp_fwd(x, split, g, w1q, w1s, w2q, w2s, workspace=ws)
    st, bits = mx.mxfp8_check_device_error(ws)
    assert st == 0, f"device error word {bits:#x}"
    return y.float().cpu().numpy().astype(np.float64), ws.cpu().numpy()


def _gpu_intermediate(mx, w, ws, rows):
    """h_q codes and scale bytes of the given sorted rows, read from the workspace."""
    L = mx.grouped_mlp_workspace_layout(w.R, w.H, w.F, w.E)
    split = w.split_sizes.astype(np.int64)
    off = np.concatenate([[0], np.cumsum(split)])
    pad = np.concatenate([[0], np.cumsum((split + 255) // 256 * 256)])   # experts padded to 256 rows
    e = np.searchsorted(off, rows, side="right") - 1
    prow = pad[e] + (rows - off[e])
    hq_all = ws[L["hq"]:L["hq"] + L["r_pad"] * w.F].reshape(L["r_pad"], w.F)
    hs_all = G.sf_mma_to_compact(ws[L["hsf"]:L["hsf"] + L["r_pad"] * w.F // 32], L["r_pad"], w.F // 32)
    return hq_all[prow], hs_all[prow], prow, pad


def _oracle_rows(oracle, w, rows, gates=True):
    o1q, o1s = oracle.quantize_rowwise(w.w1)
    o2q, o2s = oracle.quantize_rowwise(w.w2)
    g = w.gates if gates else None
    return oracle.grouped_mlp_rows(w.x_sorted, w.split_sizes, g, o1q, o1s, o2q, o2s, rows)


def _assert_parity(mx, oracle, w, rows=None, gates=True):
    rows = np.arange(w.R) if rows is None else np.asarray(rows)
    y, ws = _gpu_forward(mx, w, gates)
    y_ref, hq_ref, hs_ref = _oracle_rows(oracle, w, rows, gates)
    hq, hs, prow, pad = _gpu_intermediate(mx, w, ws, rows)
    frac, worst = G.compare_intermediate(hq, hs, hq_ref, hs_ref)
    assert frac <= G.HQ_MISMATCH_FRAC, f"intermediate mismatch fraction {frac:.2e}"
    assert worst <= G.HQ_MAX_ULPS + 1e-9, f"intermediate differs by {worst:.3f} E4M3 steps"
    rel, mxe = G.y_errors(y[rows], y_ref)
    assert rel <= G.Y_REL_TOL and mxe <= G.Y_MAX_TOL, f"y rel {rel:.3e} max {mxe:.3e}"
    # padding rows of the intermediate are zero codes with zero scale bytes
    L = mx.grouped_mlp_workspace_layout(w.R, w.H, w.F, w.E)
    split = w.split_sizes.astype(np.int64)
    pad_rows = [pad[e] + r for e in range(w.E) for r in range(int(split[e]), int(pad[e + 1] - pad[e]))]
    if pad_rows:
        hq_all = ws[L["hq"]:L["hq"] + L["r_pad"] * w.F].reshape(L["r_pad"], w.F)
        assert not np.any(hq_all[pad_rows] & 0x7F)
    return rel, mxe, frac


def test_tiny_moe_config_all_rows(mx, oracle):
    _assert_parity(mx, oracle, W.moe_workload("tiny"))


@pytest.mark.parametrize("split,H,F", [
    ([0, 1, 31, 32, 127, 128, 129, 255, 0], 256, 384),
    ([300], 512, 256),
    ([5, 0, 0, 260], 384, 128),          # H % 256 != 0: 128-column output tiles
    ([130, 70], 128, 640),
])
def test_ragged_splits(mx, oracle, split, H, F):
    w = W.custom_moe(split, H=H, F=F, seed=sum(split) + H + F)
    _assert_parity(mx, oracle, w)


def test_single_expert_without_gates(mx, oracle):
    w = W.custom_moe([384], H=256, F=256, seed=5, with_gates=False)
    _assert_parity(mx, oracle, w, gates=False)


def test_all_experts_empty_but_one(mx, oracle):
    w = W.custom_moe([0] * 7 + [45] + [0] * 8, H=128, F=128, seed=6)
    _assert_parity(mx, oracle, w)


def test_large_activations_and_small_weights(mx, oracle):
    w = W.custom_moe([200, 56], H=256, F=256, seed=7, x_std=30.0, w_std=0.001)
    _assert_parity(mx, oracle, w)


def test_repeat_calls_are_deterministic(mx):
    w = W.custom_moe([70, 190], H=256, F=256, seed=8)
    y1, _ = _gpu_forward(mx, w)
    y2, _ = _gpu_forward(mx, w)
    assert np.array_equal(y1, y2)


def test_split_mismatch_reported_on_device(mx):
    import torch
    w = W.custom_moe([64, 64], H=128, F=128, seed=9)
    x = G.to_dev_bf16(w.x_sorted)
    w1q, w1s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w1), sf_layout=mx.SF_MMA)
    w2q, w2s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w2), sf_layout=mx.SF_MMA)
    ws = torch.empty(mx.grouped_mlp_workspace_size(w.R, w.H, w.F, w.E), dtype=torch.uint8, device="cuda")
    for bad, bit in (([64, 63], 1), ([130, -2], 2)):
        mx.grouped_mlp_fwd(x, G.to_dev(np.array(bad, dtype=np.int32)), None, w1q, w1s, w2q, w2s, workspace=ws)
        st, bits = mx.mxfp8_check_device_error(ws)
        assert st == mx.ERR_SPLIT_MISMATCH and (bits & bit)
    mx.grouped_mlp_fwd(x, G.to_dev(w.split_sizes), None, w1q, w1s, w2q, w2s, workspace=ws)
    assert mx.mxfp8_check_device_error(ws) == (0, 0)


def _big_sample(split, seed=0):
    return W.sample_rows(split, seed=seed, first=4, last=4, rand=8, tile=1 << 30)


@pytest.mark.parametrize("name", ["llama", "mixtral", "fine"])
def test_full_size_configs_sampled_rows(mx, oracle, name):
    """Full-size workloads in the same launch configuration the bench times; the oracle checks a
    deterministic row sample (first/last rows and random rows of every expert)."""
    w = W.moe_workload(name)
    rows = _big_sample(w.split_sizes)
    off = np.concatenate([[0], np.cumsum(w.split_sizes)])
    # add the rows on both sides of the first and last 128-row tile boundary of each expert
    extra = []
    for e in range(w.E):
        n = int(w.split_sizes[e])
        for b in {128, (n // 128) * 128}:
            if 0 < b < n:
                extra += [off[e] + b - 1, off[e] + b]
    rows = np.unique(np.concatenate([rows, np.array(extra, dtype=np.int64)]))
    _assert_parity(mx, oracle, w, rows=rows, gates=w.gates is not None)
