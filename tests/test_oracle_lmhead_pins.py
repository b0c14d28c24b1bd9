"""Pins for the oracle's int8 head (i8_gemm) and greedy choice (argmax),
checked against numpy's integer and float matrix products on inputs where
every sum is exact, closed forms (unit vectors pick a column, ones give the
row sums), negation, and numpy's argmax (first occurrence) for the tie rule.
"""
import numpy as np
import pytest

import oracle
from packed_bit_gemv_tern_b300 import synth


def _int_x(rng, m, k, lo=-8, hi=9):
    """bf16 bits of small integers: every product and sum is exact in double."""
    return synth.f32_to_bf16_bits(rng.integers(lo, hi, (m, k)).astype(np.float32))


def _w(rng, rows, k):
    return rng.integers(-128, 128, (rows, k), dtype=np.int16).astype(np.int8)


@pytest.mark.parametrize("rows,k,m", [(7, 64, 1), (33, 256, 3), (5, 4096, 8)])
def test_matches_integer_matmul(rows, k, m):
    rng = np.random.default_rng(rows * k + m)
    w = _w(rng, rows, k)
    scale = np.ones(rows, dtype=np.float32)
    x = _int_x(rng, m, k)
    xi = synth.bf16_bits_to_f32(x).astype(np.int64)
    y, a = oracle.i8_gemm(w, scale, x, with_abs=True)
    assert np.array_equal(y, (xi @ w.astype(np.int64).T).astype(np.float64))
    assert np.array_equal(a, (np.abs(xi) @ np.abs(w.astype(np.int64)).T).astype(np.float64))
    # the fp32 row scale multiplies once, in double
    s = synth.scales(rng, rows)
    assert np.array_equal(oracle.i8_gemm(w, s, x), y * s.astype(np.float64)[None, :])


def test_unit_vectors_pick_columns_and_ones_sum_rows():
    rng = np.random.default_rng(3)
    rows, k = 19, 128
    w = _w(rng, rows, k)
    scale = synth.scales(rng, rows)
    for j in (0, 1, 63, 64, 127):
        e = np.zeros((1, k), dtype=np.float32)
        e[0, j] = 1.0
        y = oracle.i8_gemm(w, scale, synth.f32_to_bf16_bits(e))
        assert np.array_equal(y[0], scale.astype(np.float64) * w[:, j])
    ones = synth.f32_to_bf16_bits(np.ones((1, k), dtype=np.float32))
    y = oracle.i8_gemm(w, scale, ones)
    assert np.array_equal(y[0], scale.astype(np.float64) * w.astype(np.int64).sum(axis=1))


def test_negating_weights_negates_logits():
    rng = np.random.default_rng(4)
    w = _w(rng, 12, 256)
    w[w == -128] = -127  # keep the negation inside int8
    scale = synth.scales(rng, 12)
    x = synth.f32_to_bf16_bits(rng.standard_normal((2, 256), dtype=np.float32))
    assert np.array_equal(oracle.i8_gemm(-w, scale, x), -oracle.i8_gemm(w, scale, x))


def test_argmax_lowest_index_on_ties():
    y = np.array([[1.0, 3.0, 3.0, -2.0],
                  [5.0, 5.0, 5.0, 5.0],
                  [-3.0, -1.0, -2.0, -1.0],
                  [0.0, 0.0, 0.0, 7.0]])
    assert list(oracle.argmax(y)) == [1, 0, 1, 3]
    rng = np.random.default_rng(5)
    z = rng.integers(-3, 4, (50, 300)).astype(np.float64)  # many ties
    assert np.array_equal(oracle.argmax(z), np.argmax(z, axis=1))


def test_argmax_of_head_logits():
    rng = np.random.default_rng(6)
    w = _w(rng, 500, 256)
    scale = synth.scales(rng, 500)
    x = synth.f32_to_bf16_bits(rng.standard_normal((3, 256), dtype=np.float32))
    y = oracle.i8_gemm(w, scale, x, threads=4)
    assert np.array_equal(oracle.argmax(y), np.argmax(y, axis=1))
