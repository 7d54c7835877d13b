"""Pins of the oracle's row-wise and column-wise MXFP8 quantization of whole matrices.

Page "Efficient MoE training for biological foundation models", Key technical approaches,
item 2 (blocks of 32 consecutive values).  Row-wise blocks run along K; column-wise blocks run
down 32 consecutive rows of a column (the layout a transposed operand needs).
"""
import numpy as np

from mxfp8_block_scaled_03_gb300 import workloads as W
from tests import _independent as ind


def test_rowwise_matches_bruteforce_pipeline(oracle):
    x = W.quant_matrix(96, 512, seed=1)
    q, sf = oracle.quantize_rowwise(x)
    q_ref, sf_ref = ind.quantize_rows_bruteforce(W.bf16_to_f32(x).astype(np.float64))
    assert np.array_equal(sf, sf_ref)
    assert np.array_equal(q, q_ref)


def test_rowwise_zero_block_and_outliers(oracle):
    x = W.quant_matrix(64, 1024, seed=2)
    q, sf = oracle.quantize_rowwise(x)
    xf = W.bf16_to_f32(x).reshape(64, 32, 32)
    zero_blocks = np.all(xf == 0, axis=2)
    assert zero_blocks.sum(axis=1).min() >= 1            # the recipe zeroes one block per row
    assert np.all(sf[zero_blocks] == 0)
    assert np.all(q.reshape(64, 32, 32)[zero_blocks] & 0x7F == 0)


def test_colwise_equals_transposed_rowwise(oracle):
    x = W.quant_matrix(128, 96, seed=3)
    qc, sfc = oracle.quantize_colwise(x)
    qr, sfr = oracle.quantize_rowwise(np.ascontiguousarray(x.T))
    assert np.array_equal(qc, qr.T)
    assert np.array_equal(sfc, sfr.T)


def test_colwise_partial_last_block_equals_zero_padding(oracle):
    """A last block of fewer than 32 rows takes the amax of the rows present; padding the matrix
    with zero rows leaves every amax, and so every code, unchanged."""
    M = 77
    x = W.quant_matrix(M, 64, seed=4)
    qc, sfc = oracle.quantize_colwise(x)
    xp = np.zeros((96, 64), dtype=np.uint16)
    xp[:M] = x
    qr, sfr = oracle.quantize_rowwise(np.ascontiguousarray(xp.T))
    assert np.array_equal(qc, qr.T[:M])
    assert np.array_equal(sfc, sfr.T)


def test_rowwise_thread_count_does_not_matter(oracle):
    x = W.quant_matrix(300, 256, seed=5)
    a = oracle.quantize_rowwise(x, nthreads=1)
    b = oracle.quantize_rowwise(x, nthreads=7)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))


def test_bad_arguments_rejected(oracle):
    import pytest
    with pytest.raises(ValueError):
        oracle.quantize_rowwise(np.zeros((4, 48), dtype=np.uint16))
