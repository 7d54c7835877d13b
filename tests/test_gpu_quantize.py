"""GPU parity of mxfp8_quantize against the oracle: codes and scale bytes must be bit-exact.

Page "Efficient MoE training for biological foundation models", Key technical approaches,
item 2 (MXFP8: one scale per 32 consecutive values); scale rule OCP MX v1.0.
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


def _check(mx, oracle, x_bits, rowwise=True, colwise=True, layout=0):
    import torch
    x = G.to_dev_bf16(x_bits)
    q_r, s_r, q_c, s_c = mx.mxfp8_quantize(x, rowwise=rowwise, colwise=colwise, sf_layout=layout)
    torch.cuda.synchronize()
    M, K = x_bits.shape
    if rowwise:
        oq, osf = oracle.quantize_rowwise(x_bits)
        gq = q_r.cpu().numpy()
        gs = s_r.cpu().numpy()
        if layout == mx.SF_MMA:
            gs = G.sf_mma_to_compact(gs, M, K // 32)
        assert np.array_equal(gs, osf), f"row-wise scale bytes differ at {np.argwhere(gs != osf)[:5]}"
        assert np.array_equal(gq, oq), f"row-wise codes differ at {np.argwhere(gq != oq)[:5]}"
    if colwise:
        oq, osf = oracle.quantize_colwise(x_bits)
        gq = q_c.cpu().numpy()
        gs = s_c.cpu().numpy()
        if layout == mx.SF_MMA:
            gs = G.sf_mma_to_compact(gs, K, (M + 31) // 32).T
        assert np.array_equal(gs, osf), f"column-wise scale bytes differ at {np.argwhere(gs != osf)[:5]}"
        assert np.array_equal(gq, oq), f"column-wise codes differ at {np.argwhere(gq != oq)[:5]}"


@pytest.mark.parametrize("M,K", [(32, 32), (1, 64), (77, 96), (128, 256), (300, 1056), (513, 4128)])
def test_quantize_small_shapes_compact(mx, oracle, M, K):
    _check(mx, oracle, W.quant_matrix(M, K, seed=M + K))


@pytest.mark.parametrize("M,K", [(128, 128), (256, 384), (640, 1280)])
def test_quantize_mma_layout(mx, oracle, M, K):
    _check(mx, oracle, W.quant_matrix(M, K, seed=3 * M + K), layout=mx.SF_MMA)


@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_quantize_single_direction(mx, oracle, rowwise, colwise):
    _check(mx, oracle, W.quant_matrix(200, 512, seed=9), rowwise=rowwise, colwise=colwise)


def test_quantize_every_finite_bf16_pattern(mx, oracle):
    """All finite bf16 bit patterns, 32 per row in order (so block maxima sweep every binade,
    subnormals included), plus a second copy where every block also holds a large value so the
    small patterns land in the E4M3 subnormal range and round to zero at the ties."""
    pats = np.arange(65536, dtype=np.uint32)
    finite = ((pats >> 7) & 0xFF) != 0xFF
    vals = pats[finite].astype(np.uint16)
    vals = np.concatenate([vals, np.zeros((-vals.size) % 32, dtype=np.uint16)])
    a = vals.reshape(-1, 32)
    b = a.copy()
    b[:, 0] = np.uint16(0x4300)   # 128.0
    x = np.concatenate([a, b]).reshape(-1, 256)
    _check(mx, oracle, np.ascontiguousarray(x))


def test_quantize_hand_worked_values_in_a_matrix(mx, oracle):
    rows = []
    for amax in (1.0, 1.9375, 448.0, 2.0 ** -130, 0.0, 3.3895313892515355e38):
        v = np.zeros(64, dtype=np.float32)
        v[0] = amax
        v[1:8] = [amax / 3, -amax, amax * 2 ** -17, amax * 2 ** -18, amax * 3 * 2 ** -18, -0.0, amax / 7]
        rows.append(v)
    x = W.bf16_bits(np.array(rows))
    _check(mx, oracle, x)


@pytest.mark.parametrize("M,K", W.QUANT_SWEEP)
def test_quantize_sweep_full_size(mx, oracle, M, K):
    """The quantize sweep at full size, both directions, every element compared."""
    _check(mx, oracle, W.quant_matrix(M, K, seed=0))


def test_quantize_sweep_full_size_mma_layout(mx, oracle):
    _check(mx, oracle, W.quant_matrix(4096, 4096, seed=0), layout=mx.SF_MMA)


def test_quantize_empty_is_noop(mx):
    import torch
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    q, s, _, _ = mx.mxfp8_quantize(x)
    assert q.shape == (0, 64)
