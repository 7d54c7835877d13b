"""GPU parity of the NVFP4 variant (nvfp4_quantize, nvfp4_grouped_mlp_fwd) against the oracle.

Reading: the Llama 3 recipe page names NVFP4 as a quantized-training recipe (feature table;
section "Quantized Training (FP8 / MXFP8 / NVFP4)"); the format is NVIDIA's published NVFP4
(E2M1 elements, E4M3 scale per 16 values, per-tensor binary32 encode scale 448*6/amax), with
every rounding decision in binary32 on both sides.

Bars: the quantization is bit-exact (codes, scale codes, tensor amax), on the quantize sweep's
4096 x 4096 matrix, ragged and padded shapes and edge values.  The forward's y meets the same
bars as the MXFP8 forward (||y - y_ref|| / ||y_ref|| <= 5e-3, max|dy| <= 1e-2 max|y_ref|); the
GPU's fp32 accumulation differs from the oracle's binary64 sums, so an intermediate value near a
rounding boundary may round the other way: >= 99.9% of the requantized intermediate's values
equal the oracle's, every other within one E2M1 step of the coarser block grid.  The first case
is a single 256 x 256 tile per GEMM, which checks the MMA's instruction descriptor and operand
layouts in isolation.
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


def _quant_parity(mx, oracle, bits, layout):
    M, K = bits.shape
    q, sf, amax = mx.nvfp4_quantize(G.to_dev_bf16(bits), sf_layout=layout)
    oq, osf, _ = oracle.nvfp4_quantize_rowwise(bits)
    assert float(amax.cpu().item()) == oracle.bf16_amax(bits)
    assert np.array_equal(q.cpu().numpy(), G.pack_e2m1(oq))
    sfn = sf.cpu().numpy()
    if layout == mx.SF_COMPACT:
        assert np.array_equal(sfn.reshape(M, K // 16), osf)
    else:
        kt = G.nv_kt(K)
        assert sfn.size == (M // 128) * kt * 512
        assert np.array_equal(G.sf_mma_to_compact(sfn, M, K // 16, kt), osf)
        padded = G.sf_mma_to_compact(sfn, M, kt * 4, kt)   # blocks past K up to the next 256 values
        assert not padded[:, K // 16:].any()


@pytest.mark.parametrize("layout", [0, 1], ids=["compact", "mma"])
def test_quantize_sweep_matrix_bit_exact(mx, oracle, layout):
    _quant_parity(mx, oracle, W.quant_matrix(4096, 4096, seed=0), layout)


def test_quantize_edge_values(mx, oracle):
    rng = np.random.default_rng(9)
    v = rng.standard_normal((96, 160)).astype(np.float32)
    v[0] = 0.0
    v[1] = -0.0
    v[2, :16] = np.float32(2.0 ** -133)                  # bf16 subnormals
    v[3, :16] = np.float32(3.0e38)
    v[4] = np.repeat([6.0, 5.0, 0.75, 0.25, -1.75, 2.5, 3.5, -4.9, 0.2, 1.25], 16)[:160]
    v[5, 16:32] = 1e-6                                    # a block whose scale rounds to zero
    _quant_parity(mx, oracle, W.bf16_bits(v), 0)


def test_quantize_all_zero_and_padded_k(mx, oracle):
    _quant_parity(mx, oracle, np.zeros((128, 256), dtype=np.uint16), 1)
    rng = np.random.default_rng(10)
    _quant_parity(mx, oracle, W.bf16_bits(rng.standard_normal((256, 384)).astype(np.float32) * 3), 1)


def _h_amax(w, rows):
    """1.5 x the largest |h| over the sampled rows, from the unquantized bf16 operands (a
    calibration of the intermediate's encode scale; any positive value is a valid input)."""
    x = W.bf16_to_f32(w.x_sorted[rows])
    off = np.concatenate([[0], np.cumsum(w.split_sizes)])
    e = np.searchsorted(off, rows, side="right") - 1
    h = 0.0
    for ex in np.unique(e):
        xe = x[e == ex]
        w1e = W.bf16_to_f32(w.w1[ex * 2 * w.F:(ex + 1) * 2 * w.F])
        g, u = (xe @ w1e[:w.F].T).astype(np.float64), (xe @ w1e[w.F:].T).astype(np.float64)
        gt = np.ones(len(xe)) if w.gates is None else w.gates[rows[e == ex]].astype(np.float64)
        h = max(h, float(np.abs(gt[:, None] * g / (1 + np.exp(-g)) * u).max()))
    return 1.5 * h


def _forward_parity(mx, oracle, w, rows):
    import torch
    x = G.to_dev_bf16(w.x_sorted)
    split = G.to_dev(w.split_sizes)
    gates = G.to_dev(w.gates) if w.gates is not None else None
    w1 = mx.nvfp4_quantize(G.to_dev_bf16(w.w1), sf_layout=mx.SF_MMA)
    w2 = mx.nvfp4_quantize(G.to_dev_bf16(w.w2), sf_layout=mx.SF_MMA)
    h_amax = _h_amax(w, rows)
    ws = torch.empty(mx.nvfp4_grouped_mlp_workspace_size(w.R, w.H, w.F, w.E), dtype=torch.uint8, device="cuda")
    y = mx.nvfp4_grouped_mlp_fwd(x, split, gates, w1, w2, h_amax, workspace=ws)
    st, bits = mx.mxfp8_check_device_error(ws)
    assert st == 0, f"device error word {bits:#x}"
    y = y.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(y).all()

    ow1 = oracle.nvfp4_quantize_rowwise(w.w1)
    ow2 = oracle.nvfp4_quantize_rowwise(w.w2)
    assert float(w1[2].cpu().item()) == oracle.bf16_amax(w.w1)
    y_ref, hq_ref, hsf_ref, _ = oracle.nvfp4_grouped_mlp_rows(w.x_sorted, w.split_sizes, w.gates, ow1, ow2, h_amax,
                                                              rows)
    rel, mxe = G.y_errors(y[rows], y_ref)
    assert rel <= G.Y_REL_TOL and mxe <= G.Y_MAX_TOL, f"y rel {rel:.3e} max {mxe:.3e}"

    # the requantized intermediate, read from the workspace at each sampled row's padded row
    lay = mx.nvfp4_grouped_mlp_workspace_layout(w.R, w.H, w.F, w.E)
    wsn = ws.cpu().numpy()
    r_pad, F = lay[6], w.F
    off = np.concatenate([[0], np.cumsum(w.split_sizes)])
    pad = np.concatenate([[0], np.cumsum(256 * ((w.split_sizes + 255) // 256))])
    e = np.searchsorted(off, rows, side="right") - 1
    prow = pad[e] + (rows - off[e])
    hq = G.unpack_e2m1(wsn[lay[4]:lay[4] + r_pad * F // 2].reshape(r_pad, F // 2)[prow])
    kt = G.nv_kt(F)
    hsf_all = G.sf_mma_to_compact(wsn[lay[5]:lay[5] + (r_pad // 128) * kt * 512], r_pad, F // 16, kt)
    frac, worst = G.nv_compare_intermediate(hq, hsf_all[prow], hq_ref, hsf_ref, oracle.nvfp4_encode_scale(h_amax))
    assert frac <= G.HQ_MISMATCH_FRAC and worst <= 1.0, (frac, worst)
    seen = np.frombuffer(wsn[lay[1]:lay[1] + 8].tobytes(), dtype=np.float32)
    assert seen[0] == oracle.bf16_amax(w.x_sorted) and 0 < seen[1] <= 1.0e30
    return y


def test_single_tile(mx, oracle):
    w = W.custom_moe([256], H=256, F=128, seed=51)
    _forward_parity(mx, oracle, w, np.arange(w.R))


def test_tiny_all_rows(mx, oracle):
    w = W.moe_workload("tiny")
    _forward_parity(mx, oracle, w, np.arange(w.R))


def test_ragged_half_k_step_and_empty_experts(mx, oracle):
    # F = 384: GroupedLinear 2's last K step is half past the end (zero codes, zero scales)
    w = W.custom_moe([0, 1, 31, 32, 127, 128, 129, 255, 0], H=512, F=384, seed=52)
    _forward_parity(mx, oracle, w, np.arange(w.R))


def test_no_gates(mx, oracle):
    w = W.custom_moe([300, 212], H=256, F=256, seed=53, with_gates=False)
    _forward_parity(mx, oracle, w, np.arange(w.R))


def test_fine_grained_sampled(mx, oracle):
    w = W.moe_workload("fine")
    _forward_parity(mx, oracle, w, W.sample_rows(w.split_sizes, first=2, last=2, rand=2))


def test_mixtral_sampled(mx, oracle):
    w = W.moe_workload("mixtral")
    _forward_parity(mx, oracle, w, W.sample_rows(w.split_sizes, first=4, last=4, rand=6))


def test_rejects_unsupported_shapes(mx):
    import torch
    t = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    f = torch.empty(4, dtype=torch.float32, device="cuda")
    L = mx.lib()
    P = lambda a: a.data_ptr()
    st = L.nvfp4_grouped_mlp_fwd(P(t), 128, 384, 128, 1, P(t), None, P(t), P(t), P(f), P(t), P(t), P(f), 1.0,
                                 P(t), P(t), t.numel(), None, None)
    assert st == mx.ERR_UNSUPPORTED            # H % 256 != 0
    st = L.nvfp4_grouped_mlp_fwd(P(t), 128, 256, 128, 1, P(t), None, P(t), P(t), P(f), P(t), P(t), P(f), 0.0,
                                 P(t), P(t), t.numel(), None, None)
    assert st == mx.ERR_INVALID_ARG            # h_amax must be positive
