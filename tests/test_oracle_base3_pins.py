"""Pins for the oracle's base-3 format (pack5, unpack5, gemm5): hand-derived
bytes (tests/golden/base3_bytes.txt), the bijection between the 3^5 weight
patterns and the bytes 0..242, rejection of bytes 243..255, the projection
equal to the 2-bit format's oracle GEMM on the same ternary matrix, and the
closed forms x = ones and x = e_k.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
from packed_bit_gemv_tern_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "base3_bytes.txt")


def _golden():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                v = [int(s) for s in line.split()]
                out.append((v[0], v[1:]))
    return out


def test_hand_derived_bytes():
    for byte, w in _golden():
        t = np.zeros((1, 80), dtype=np.int8)
        t[0, :5] = w
        c = oracle.pack5(t)
        assert c[0, 0] == byte and np.all(c[0, 1:] == 121)
        assert list(oracle.unpack5(c, 80)[0, :5]) == w


def test_all_patterns_are_a_bijection_onto_0_242():
    pats = np.array(list(itertools.product((-1, 0, 1), repeat=5)), dtype=np.int8)  # 243 x 5
    t = np.zeros((243, 80), dtype=np.int8)
    t[:, :5] = pats
    c = oracle.pack5(t)
    assert sorted(c[:, 0].tolist()) == list(range(243))
    assert np.array_equal(oracle.unpack5(c, 80), t)


def test_invalid_bytes_and_shapes_rejected():
    scale = np.ones(1, dtype=np.float32)
    x = np.zeros((1, 80), dtype=np.uint16)
    for b in (243, 250, 255):
        c = np.full((1, 16), 121, dtype=np.uint8)
        c[0, 7] = b
        with pytest.raises(oracle.OracleError):
            oracle.unpack5(c, 80)
        with pytest.raises(oracle.OracleError):
            oracle.gemm5(c, scale, 80, x)
    with pytest.raises(oracle.OracleError):
        oracle.pack5(np.zeros((2, 64), dtype=np.int8))


@pytest.mark.parametrize("rows,k,m", [(7, 80, 1), (33, 320, 2), (20, 4160, 7)])
def test_projection_equals_the_two_bit_oracle(rows, k, m):
    """The same ternary matrix in both formats gives the same fp64 sums (both
    add in increasing k), so gemm5 equals gemm bit for bit."""
    rng = np.random.default_rng(rows + k + m)
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    x = synth.activations(rng, m, k)
    k2 = (k + 63) // 64 * 64
    t2 = np.zeros((rows, k2), dtype=np.int8)
    t2[:, :k] = t
    x2 = np.zeros((m, k2), dtype=np.uint16)
    x2[:, :k] = x
    assert np.array_equal(oracle.gemm5(oracle.pack5(t), scale, k, x), oracle.gemm(oracle.pack(t2), scale, k2, x2))


def test_closed_forms():
    rng = np.random.default_rng(5)
    rows, k = 29, 400
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    c = oracle.pack5(t)
    ones = np.full((1, k), 0x3F80, dtype=np.uint16)
    assert np.array_equal(oracle.gemm5(c, scale, k, ones)[0], scale.astype(np.float64) * t.astype(np.int64).sum(1))
    for j in (0, 4, 5, 399):
        e = np.zeros((1, k), dtype=np.uint16)
        e[0, j] = 0x3F80
        assert np.array_equal(oracle.gemm5(c, scale, k, e)[0], scale.astype(np.float64) * t[:, j])
