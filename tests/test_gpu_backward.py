"""GPU parity of the grouped-MLP backward (grouped_mlp_fwd_train + grouped_mlp_bwd) and of the
transposed column-wise quantize against the oracle.

Page "Efficient MoE training for biological foundation models", Key technical approaches item 3
(the fused op's corresponding backward).  The oracle computes the same reading in binary64; the
GPU accumulates in fp32, so every tensor both sides quantize agrees except for rare codes whose
input lies within fp32 rounding of a rounding boundary.  Bars (same as the forward's y):
||out - ref|| / ||ref|| <= 5e-3 and max|out - ref| <= 1e-2 * max|ref| for dx, dgates and the
weight-gradient entries; weight gradients of experts without rows are exactly zero; the
transposed quantize is bit-exact.  The quantized [dG | dU] (row-wise and column-wise) and h
(column-wise) that the dh GEMM's epilogue writes meet the forward intermediate's bar against the
oracle's quantizations of its bf16 dGU and h: at most 0.1% of the codes differ, each by at most one
E4M3 step (two subnormal steps near zero: see _check_codes).
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
    return _np(dx), _np(dg), _np(dw1), _np(dw2), y, ws, saved


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


def _check_saved_gu(w, saved, rows, rgu):
    """The training forward's saved pre-activations [G | U] (bf16, blocks of 32 padded rows x 8
    columns, row-major inside) against the oracle's: the GPU rounds its fp32 sums to bf16 and the
    oracle its binary64 ones, so at most 0.5% of the elements may differ (one bf16 step, or a few
    next to zero, where the fp32 sum's absolute error exceeds the bf16 spacing), within the y bars.
    Returns the [n, F] mask of (row, f) whose g or u differ: there dG = dh gate u silu'(g) can move
    by far more than one E4M3 step (silu'(g) crosses zero at g = -1.278; a one-step change of g
    next to it changes silu'(g) by a large fraction), so those elements are held to the norm bars
    only."""
    import torch
    F = w.F
    prow = _padded_rows(w, rows)
    sv = saved.view(torch.int16)[: (int(prow.max()) // 32 + 1) * 32 * 2 * F]
    blocks = sv.view(-1, 2 * F // 8, 32, 8)
    pr = torch.as_tensor(prow, device=saved.device)
    got = blocks[pr // 32, :, pr % 32, :].reshape(len(prow), 2 * F).cpu().numpy().view(np.uint16)
    differs = got != rgu
    frac = float(np.mean(differs))
    assert frac <= 5e-3, f"saved [G | U]: {frac:.2e} of the elements differ"
    _check("saved [G | U]", W.bf16_to_f32(got), W.bf16_to_f32(rgu))
    return differs[:, :F] | differs[:, F:]


def _check_codes(name, q, sf, q_ref, sf_ref, exempt=None):
    """MXFP8 tensors handed between the backward GEMMs (blocks of 32 along the last axis): the
    GPU's fp32 sums and its saved bf16 pre-activations can round the other way from the oracle's
    binary64 near a rounding boundary, so the bar is the forward intermediate's: a small fraction
    of elements may differ, each by at most one E4M3 step of the coarser grid.  One allowance:
    an element within a few subnormal E4M3 steps of zero on its block's grid may differ by up to
    two such steps (2^(s-9) each, s the block's scale exponent).  dh is an fp32 sum over H
    products whose absolute rounding error, about 2^-24 sqrt(H) of the block's largest term, is
    of the order of that step, and a dh near zero from cancellation keeps it whole."""
    a = G.dequant(q, sf)
    b = G.dequant(q_ref, sf_ref)
    diff = np.abs(a - b)
    big = np.maximum(np.abs(a), np.abs(b))
    s = np.maximum(np.asarray(sf, dtype=np.int64), np.asarray(sf_ref, dtype=np.int64))
    ulp = np.maximum(G.e4m3_ulp(big, s), G.e4m3_ulp(big, sf))
    tiny = np.ldexp(1.0, np.repeat(s - 127 - 9, 32, axis=-1))
    frac = float(np.mean(diff != 0))
    bad = diff > np.maximum(G.HQ_MAX_ULPS * ulp, 2.0 * tiny) * (1 + 1e-12)
    if exempt is not None:   # elements whose saved inputs rounded differently (see _check_saved_gu)
        bad &= ~exempt
        rel, _ = G.y_errors(a, b)
        assert rel <= G.Y_REL_TOL, f"{name}: rel {rel:.3e}"
    assert frac <= G.HQ_MISMATCH_FRAC, f"{name}: mismatch fraction {frac:.2e}"
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        blk = i[:-1] + (i[-1] // 32,)
        raise AssertionError(f"{name}: element {i} gpu {a[i]!r} (code {q[i]}, scale {sf[blk]}) oracle "
                             f"{b[i]!r} (code {q_ref[i]}, scale {sf_ref[blk]}); {int(bad.sum())} elements "
                             f"beyond the bar")


def _block_rows(w, ends_only):
    """Sorted rows and padded-row starts of complete 32-row column blocks: every block of every
    expert, or (ends_only) each non-empty expert's first and last block (the last one ends in
    padding rows when the expert's count is not a multiple of 32)."""
    off = np.concatenate([[0], np.cumsum(w.split_sizes)])
    pad = np.concatenate([[0], np.cumsum(256 * ((w.split_sizes + 255) // 256))])
    rows, starts = [], []
    for e in np.nonzero(w.split_sizes)[0]:
        n = int(w.split_sizes[e])
        nb = (n + 31) // 32
        for j in (sorted({0, nb - 1}) if ends_only else range(nb)):
            rows.extend(range(off[e] + 32 * j, off[e] + min(32 * j + 32, n)))
            starts.append(pad[e] + 32 * j)
    return np.array(rows, dtype=np.int64), np.array(starts, dtype=np.int64)


def _check_dgu_h(mx, oracle, w, ws, rows, rdgu, rh, col_starts, gu_differs):
    """The quantized [dG | dU] (row-wise, for dx; column-wise, for dW1) and h (column-wise, for
    dW2) that the dh GEMM's epilogue wrote, against the oracle's quantizations of its own bf16 dGU
    and h: rows `rows` row-wise; the 32-row blocks starting at padded rows col_starts column-wise
    (their real rows are among `rows`; padding rows are zeros).  gu_differs [n, F]: the (row, f)
    whose saved g or u rounded differently on the two sides (exempt from the per-element bar)."""
    import torch
    lay = mx.grouped_mlp_bwd_workspace_layout(w.R, w.H, w.F, w.E)
    r_pad, F = lay[7], w.F
    prow = _padded_rows(w, rows)
    dev = ws.device
    dguq = ws[lay[1]:lay[1] + r_pad * 2 * F].view(r_pad, 2 * F)[torch.as_tensor(prow, device=dev)].cpu().numpy()
    dgusf = G.sf_mma_to_compact(ws[lay[2]:lay[2] + r_pad * 2 * F // 32].cpu().numpy(), r_pad, 2 * F // 32)[prow]
    q_ref, sf_ref = oracle.quantize_rowwise(rdgu)
    ex2 = np.concatenate([gu_differs, gu_differs], axis=1)
    _check_codes("dGU row-wise", dguq, dgusf, q_ref, sf_ref, ex2)
    # column blocks: the oracle's rows of each block, zeros on its padding rows
    pos = {int(p): i for i, p in enumerate(prow)}
    blk_rows = (col_starts[:, None] + np.arange(32)[None, :]).reshape(-1)
    sel = np.array([pos.get(int(p), -1) for p in blk_rows])
    cols = torch.as_tensor(blk_rows, device=dev)
    for name, ref_bits, qo, so, K, ex in (("dGU column-wise", rdgu, lay[3], lay[4], 2 * F, ex2),
                                          ("h column-wise", rh, lay[5], lay[6], F, gu_differs)):
        xb = np.where(sel[:, None] >= 0, ref_bits[np.maximum(sel, 0)], 0).astype(np.uint16)
        exb = np.where(sel[:, None] >= 0, ex[np.maximum(sel, 0)], False)
        cq_ref, csf_ref = oracle.quantize_colwise(xb)          # [32 nb, K], [nb, K]
        cq = ws[qo:qo + K * r_pad].view(K, r_pad)[:, cols].cpu().numpy()
        csf = G.sf_mma_to_compact(ws[so:so + K * r_pad // 32].cpu().numpy(), K, r_pad // 32)[:, col_starts // 32]
        _check_codes(name, cq, csf, cq_ref.T, csf_ref.T, exb.T)
    # padding rows of the row-wise codes are zeros
    pad_rows = blk_rows[sel < 0]
    if pad_rows.size:
        zq = ws[lay[1]:lay[1] + r_pad * 2 * F].view(r_pad, 2 * F)[torch.as_tensor(pad_rows, device=dev)]
        assert not bool(zq.any()), "padding rows of the row-wise dGU codes are not zero"


def _assert_bwd_parity(mx, oracle, w, rows, n_entries, seed=0, all_blocks=True):
    dyb = _dy(w, seed)
    dx, dg, dw1, dw2, _, ws, saved = _gpu_bwd(mx, w, dyb)
    ow = _oracle_weights(oracle, w)
    brows, col_starts = _block_rows(w, ends_only=not all_blocks)
    rows = np.union1d(rows, brows)
    rdx, rdg, rdgu, rh, rgu = oracle.grouped_mlp_bwd_rows(w.x_sorted, w.split_sizes, w.gates, *ow, dyb, rows,
                                                          want_gu=True)
    _check("dx", dx[rows], rdx)
    if w.gates is not None:
        _check("dgates", dg[rows], rdg)
    gu_differs = _check_saved_gu(w, saved, rows, rgu)
    _check_dgu_h(mx, oracle, w, ws, rows, rdgu, rh, col_starts, gu_differs)
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
    sampled rows (per expert the first and last 8, 8 random, both sides of every 128-row tile
    boundary, and its first and last 32-row block) of dx, dgates and the quantized dGU and h,
    sampled weight-gradient entries against the oracle, zero gradients of the empty experts."""
    w = W.moe_workload("fine")
    rows = W.sample_rows(w.split_sizes, seed=1, first=8, last=8, rand=8, tile=128)
    _assert_bwd_parity(mx, oracle, w, rows, 160, seed=11, all_blocks=False)


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
    both sides of every 128-row tile boundary, plus each expert's first and last 32-row block) of
    dx, dgates and the quantized dGU and h, and sampled weight-gradient entries."""
    w = W.moe_workload("mixtral")
    rows = W.sample_rows(w.split_sizes, seed=0, first=8, last=8, rand=8, tile=128)
    _assert_bwd_parity(mx, oracle, w, rows, 160, all_blocks=False)


def test_no_routed_rows_forward_and_backward(mx):
    """R = 0 (every expert empty, as on an expert-parallel rank that received no tokens): the
    forward, the training forward and the backward accept empty row buffers, report no device
    error, and the weight gradients are exactly zero."""
    import torch
    w = W.custom_moe([0, 0, 0], H=256, F=256, seed=31)
    x = G.to_dev_bf16(w.x_sorted)
    split = G.to_dev(w.split_sizes)
    g = G.to_dev(w.gates)
    w1 = G.to_dev_bf16(w.w1)
    w2 = G.to_dev_bf16(w.w2)
    w1q, w1s, _, _ = mx.mxfp8_quantize(w1, sf_layout=mx.SF_MMA)
    w2q, w2s, _, _ = mx.mxfp8_quantize(w2, sf_layout=mx.SF_MMA)
    ws = torch.zeros(mx.grouped_mlp_workspace_size(0, w.H, w.F, w.E), dtype=torch.uint8, device="cuda")
    y = mx.grouped_mlp_fwd(x, split, g, w1q, w1s, w2q, w2s, workspace=ws)
    assert tuple(y.shape) == (0, w.H) and mx.mxfp8_check_device_error(ws) == (0, 0)
    y, saved = mx.grouped_mlp_fwd_train(x, split, g, w1q, w1s, w2q, w2s, workspace=ws)
    assert mx.mxfp8_check_device_error(ws) == (0, 0)
    w1tq, w1ts = mx.mxfp8_quantize_colwise_t(w1)
    w2tq, w2ts = mx.mxfp8_quantize_colwise_t(w2)
    dx, dg, dw1, dw2, bws = mx.grouped_mlp_bwd(x, split, g, saved, w1tq, w1ts, w2tq, w2ts,
                                               G.to_dev_bf16(_dy(w, 1)))
    assert mx.mxfp8_check_device_error(bws) == (0, 0)
    assert tuple(dx.shape) == (0, w.H)
    assert not bool(dw1.any()) and not bool(dw2.any())
