"""Pins for the oracle's RMSNorm prologue (orc_rmsnorm, rmsnorm_gemm), checked
against what the operation's definition fixes rather than against a retyped
formula: closed forms (constant rows, unit rows that make the norm the
identity and reduce the projection to the plain oracle GEMM and to a dense
numpy product), invariants (power-of-two scaling of a row, duplicating a
row's channels, power-of-two channel weights), the unit mean square of the
output, and rows so small that eps decides the factor.
"""
import numpy as np
import pytest

import oracle
from packed_bit_gemv_tern_b300 import synth


def _f64(bits):
    return synth.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16)).astype(np.float64)


def _bits(vals):
    return synth.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def _normal_rows(rng, m, k):
    return _bits(rng.standard_normal((m, k), dtype=np.float32))


@pytest.mark.parametrize("c", [3.0, -0.5, 96.0, 1.0 / 16])
def test_constant_row_normalises_to_sign(c):
    """x = c everywhere: mean x^2 = c^2, so xn = g * sign(c) up to eps and the
    bf16 rounding (|c| / sqrt(c^2 + 1e-6) rounds to 1 for these c), and the
    projection is scale[r] * rowsum[r] * g * sign(c)."""
    rng = np.random.default_rng(11)
    k, rows = 256, 40
    x = _bits(np.full((1, k), c))
    for gval in (1.0, 0.75, -2.0):
        g = np.full(k, gval, dtype=np.float32)
        xn, _ = oracle.rmsnorm(x, g, 1e-6)
        assert np.all(_f64(xn) == gval * np.sign(c))
        t = synth.ternary(rng, rows, k)
        scale = synth.scales(rng, rows)
        codes = oracle.pack(t)
        y = oracle.rmsnorm_gemm(codes, scale, k, x, g, 1e-6)
        rowsum = t.astype(np.int64).sum(axis=1)
        assert np.array_equal(y[0], scale.astype(np.float64) * rowsum * (gval * np.sign(c)))


def test_unit_rows_reduce_to_the_plain_projection():
    """Rows of +-1 with unit weights and eps = 0 have mean square exactly 1,
    so the norm is the identity: rmsnorm_gemm equals the plain oracle GEMM
    bit for bit, and a dense numpy product from the int8 matrix."""
    rng = np.random.default_rng(12)
    for m, k, rows in [(1, 64, 17), (3, 512, 33), (7, 4096, 9)]:
        x = _bits(np.where(rng.random((m, k)) < 0.5, -1.0, 1.0))
        g = np.ones(k, dtype=np.float32)
        xn, r = oracle.rmsnorm(x, g, 0.0)
        assert np.all(r == 1.0) and np.array_equal(xn, x)
        t = synth.ternary(rng, rows, k)
        scale = synth.scales(rng, rows)
        codes = oracle.pack(t)
        y = oracle.rmsnorm_gemm(codes, scale, k, x, g, 0.0)
        assert np.array_equal(y, oracle.gemm(codes, scale, k, x))
        dense = (_f64(x) @ t.astype(np.float64).T) * scale.astype(np.float64)[None, :]
        assert np.allclose(y, dense, rtol=0, atol=1e-9)
        # the gated pair on the same rows equals the plain gated pair
        tu = synth.ternary(rng, rows, k)
        su = synth.scales(rng, rows)
        cu = oracle.pack(tu)
        assert np.array_equal(oracle.rmsnorm_swiglu(codes, scale, cu, su, k, x, g, 0.0),
                              oracle.swiglu(codes, scale, cu, su, k, x))


@pytest.mark.parametrize("j", [-30, -7, 3, 40])
def test_power_of_two_scaling_leaves_the_output_unchanged(j):
    """With eps = 0, x -> 2^j x scales the root mean square by exactly 2^j
    and every rounding step commutes with a power-of-two factor, so xn is
    identical bit for bit."""
    rng = np.random.default_rng(13)
    x = _normal_rows(rng, 4, 1024)
    xs = _bits(_f64(x) * 2.0 ** j)
    assert np.array_equal(_f64(xs), _f64(x) * 2.0 ** j)  # the scaled rows are exact
    g = rng.uniform(0.5, 2.0, 1024).astype(np.float32)
    a, ra = oracle.rmsnorm(x, g, 0.0)
    b, rb = oracle.rmsnorm(xs, g, 0.0)
    assert np.array_equal(a, b)
    assert np.array_equal(rb.astype(np.float64), ra.astype(np.float64) * 2.0 ** -j)


@pytest.mark.parametrize("k", [64, 4096, 12288])
def test_unit_mean_square(k):
    """With unit weights and eps = 0 the output has mean square 1, up to the
    bf16 rounding of each element (relative 2^-9 at most, so 2^-8 on a
    square)."""
    rng = np.random.default_rng(14 + k)
    x = _normal_rows(rng, 5, k)
    xn, _ = oracle.rmsnorm(x, np.ones(k, dtype=np.float32), 0.0)
    ms = (_f64(xn) ** 2).mean(axis=1)
    assert np.all(np.abs(ms - 1.0) <= 2.0 ** -8), ms


def test_eps_decides_tiny_rows():
    """x = 2^-20 everywhere: mean square 2^-40, far below eps = 1e-6, so the
    factor is about 1 / sqrt(1e-6) and xn about 2^-20 * 1000; with eps = 0
    the row normalises to 1.  (eps outside the root, or scaled by K, gives a
    different value.)"""
    k = 512
    x = _bits(np.full((1, k), 2.0 ** -20))
    g = np.ones(k, dtype=np.float32)
    xn, r = oracle.rmsnorm(x, g, 1e-6)
    want = 2.0 ** -20 / np.sqrt(2.0 ** -40 + 1e-6)
    assert np.all(np.abs(_f64(xn) - want) <= 2.0 ** -8 * want)
    assert abs(float(r[0]) - 1.0 / np.sqrt(2.0 ** -40 + 1e-6)) <= 1e-6 * float(r[0])
    xn0, _ = oracle.rmsnorm(x, g, 0.0)
    assert np.all(_f64(xn0) == 1.0)


def test_duplicated_channels_keep_the_mean():
    """Concatenating a row with itself (and its weights) keeps the mean
    square, so each half of the result equals the single row's result: the
    divisor is the row's own channel count."""
    rng = np.random.default_rng(15)
    x = _normal_rows(rng, 3, 768)
    g = rng.uniform(0.25, 4.0, 768).astype(np.float32)
    a, ra = oracle.rmsnorm(x, g, 1e-6)
    b, rb = oracle.rmsnorm(np.concatenate([x, x], axis=1), np.concatenate([g, g]), 1e-6)
    assert np.array_equal(ra, rb)
    assert np.array_equal(b[:, :768], a) and np.array_equal(b[:, 768:], a)


def test_channel_weights_apply_per_channel_after_the_mean():
    """Power-of-two weights 2^e_k scale output k by exactly 2^e_k and leave
    every other channel and the row factor alone: the weight multiplies its
    own channel, after the mean square is taken."""
    rng = np.random.default_rng(16)
    k = 1024
    x = _normal_rows(rng, 2, k)
    e = rng.integers(-3, 4, k)
    g = (2.0 ** e).astype(np.float32)
    base, r0 = oracle.rmsnorm(x, np.ones(k, dtype=np.float32), 1e-6)
    scaled, r1 = oracle.rmsnorm(x, g, 1e-6)
    assert np.array_equal(r0, r1)
    assert np.array_equal(_f64(scaled), _f64(base) * (2.0 ** e)[None, :])


def test_c_composite_matches():
    rng = np.random.default_rng(17)
    k, rows = 256, 21
    x = _normal_rows(rng, 3, k)
    g = rng.uniform(0.5, 1.5, k).astype(np.float32)
    codes = oracle.pack(synth.ternary(rng, rows, k))
    scale = synth.scales(rng, rows)
    assert np.array_equal(oracle.rmsnorm_gemm_c(codes, scale, k, x, g, 1e-6),
                          oracle.rmsnorm_gemm(codes, scale, k, x, g, 1e-6))
