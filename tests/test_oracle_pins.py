"""Pins for the fp64 CPU oracle, checked against things other than itself:
hand-decoded words of the format, a hand-worked GEMV, dense brute force on
tiny inputs (numpy on the int8 matrix, never on the packed words), closed
forms (x = ones, x = e_k), exact-integer inputs, invariants, and SiLU
identities checked through scipy's independent logistic routine.
"""
import itertools
import os

import numpy as np
import pytest
import scipy.special

import oracle
from packed_bit_gemv_tern_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_words():
    out = []
    with open(os.path.join(GOLDEN, "format_words.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            word = int(parts[0], 16)
            vals = None if parts[1] == "invalid" else [int(v) for v in parts[1:]]
            out.append((word, vals))
    return out


def _x_f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _brute(t, scale, x_bits):
    """Dense reference from the int8 matrix: y[m, r] = scale[r] * sum_k t[r,k] x[m,k]."""
    return (_x_f64(x_bits) @ t.astype(np.float64).T) * scale.astype(np.float64)[None, :]


@pytest.mark.parametrize("word,vals", _golden_words())
def test_format_golden_words(word, vals):
    codes = np.zeros((1, 4), dtype=np.uint32)
    codes[0, 0] = word
    if vals is None:
        with pytest.raises(oracle.OracleError):
            oracle.unpack(codes, 64)
        with pytest.raises(oracle.OracleError):
            oracle.stats(codes, 64)
        with pytest.raises(oracle.OracleError):
            oracle.gemm(codes, np.ones(1, np.float32), 64, np.zeros((1, 64), np.uint16))
        return
    t = oracle.unpack(codes, 64)
    assert t[0, :16].tolist() == vals
    assert not t[0, 16:].any()
    # the oracle's own encoder reproduces the hand-written word
    assert int(oracle.pack(t)[0, 0]) == word


def test_gemv_worked_example():
    x = np.zeros(64, np.float32)
    x[:4] = [1.0, 7.0, 0.5, -2.0]
    x[4:16] = 100.0
    x[16:] = 0.25
    xb = synth.f32_to_bf16_bits(x)[None, :]
    rows = []
    with open(os.path.join(GOLDEN, "gemv_worked.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                p = line.split()
                rows.append(([int(w, 16) for w in p[1:5]], float(p[5]), float(p[6])))
    codes = np.array([r[0] for r in rows], dtype=np.uint32)
    scale = np.array([r[1] for r in rows], dtype=np.float32)
    y = oracle.gemm(codes, scale, 64, xb)[0]
    assert y.tolist() == [r[2] for r in rows]


@pytest.mark.parametrize("rows,k,m,seed", [(1, 64, 1, 0), (3, 64, 1, 1), (33, 128, 2, 2),
                                           (64, 256, 7, 3), (17, 192, 8, 4)])
def test_pack_roundtrip_and_bruteforce(rows, k, m, seed):
    rng = np.random.default_rng(seed)
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    x = synth.activations(rng, m, k)
    codes = oracle.pack(t)
    assert codes.shape == (rows, k // 16)
    assert np.array_equal(oracle.unpack(codes, k), t)
    y = oracle.gemm(codes, scale, k, x)
    np.testing.assert_allclose(y, _brute(t, scale, x), rtol=1e-12, atol=1e-14)


def test_all_ternary_patterns_of_eight():
    """Every one of the 3**8 sign patterns on 8 columns, placed at both ends of a
    word and straddling two words, against brute force."""
    pats = np.array(list(itertools.product((-1, 0, 1), repeat=8)), dtype=np.int8)
    rng = np.random.default_rng(7)
    x = synth.activations(rng, 2, 64)
    scale = synth.scales(rng, pats.shape[0])
    for off in (0, 8, 12, 56):
        t = np.zeros((pats.shape[0], 64), np.int8)
        t[:, off:off + 8] = pats
        codes = oracle.pack(t)
        y = oracle.gemm(codes, scale, 64, x)
        np.testing.assert_allclose(y, _brute(t, scale, x), rtol=1e-12, atol=1e-14)


def test_unit_vectors_pin_bit_order():
    rng = np.random.default_rng(11)
    rows, k = 8, 128
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    codes = oracle.pack(t)
    one = synth.f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    for kk in range(k):
        x = np.zeros((1, k), np.uint16)
        x[0, kk] = one
        y = oracle.gemm(codes, scale, k, x)[0]
        assert np.array_equal(y, scale.astype(np.float64) * t[:, kk])


def test_ones_closed_form_and_rowsum():
    rng = np.random.default_rng(12)
    rows, k = 40, 1024
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    codes = oracle.pack(t)
    ones = np.full((1, k), synth.f32_to_bf16_bits(np.array([1.0], np.float32))[0], np.uint16)
    y = oracle.gemm(codes, scale, k, ones)[0]
    rowsum_np = t.astype(np.int64).sum(axis=1)
    assert np.array_equal(y, scale.astype(np.float64) * rowsum_np)
    rowsum, counts = oracle.stats(codes, k)
    assert np.array_equal(rowsum, rowsum_np)
    assert counts.tolist() == [int((t == 0).sum()), int((t == 1).sum()), int((t == -1).sum())]
    assert counts.sum() == rows * k
    assert np.array_equal(rowsum, (t == 1).sum(1) - (t == -1).sum(1))


def test_zero_negation_and_exact_integers():
    rng = np.random.default_rng(13)
    rows, k = 24, 4096
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    codes = oracle.pack(t)
    assert not oracle.gemm(codes, scale, k, np.zeros((1, k), np.uint16)).any()
    x = synth.activations(rng, 1, k)
    y = oracle.gemm(codes, scale, k, x)
    y_neg = oracle.gemm(codes, scale, k, x ^ np.uint16(0x8000))
    assert np.array_equal(y_neg, -y)
    xi = synth.small_int_activations(rng, 3, k)
    yi = oracle.gemm(codes, scale, k, xi)
    dot = synth.bf16_bits_to_f32(xi).astype(np.int64) @ t.astype(np.int64).T
    assert np.array_equal(yi, dot.astype(np.float64) * scale.astype(np.float64)[None, :])


def test_swiglu_identities():
    rng = np.random.default_rng(14)
    rows, k, m = 32, 256, 3
    tg = synth.ternary(rng, rows, k)
    tu = synth.ternary(rng, rows, k)
    tg[5] = 0  # a gate row of zeros gives h = 0 whatever up is
    sg, su = synth.scales(rng, rows), synth.scales(rng, rows)
    x = synth.activations(rng, m, k)
    h = oracle.swiglu(oracle.pack(tg), sg, oracle.pack(tu), su, k, x)
    g, u = _brute(tg, sg, x), _brute(tu, su, x)
    np.testing.assert_allclose(h, g * scipy.special.expit(g) * u, rtol=1e-12, atol=1e-15)
    assert not h[:, 5].any()
    assert oracle.silu(0.0) == 0.0
    for z in (-3.0, -0.5, 0.25, 1.0, 7.5):
        assert oracle.silu(z) - oracle.silu(-z) == pytest.approx(z, rel=1e-15)
        assert oracle.silu(z) == pytest.approx(z * scipy.special.expit(z), rel=1e-14)
    assert oracle.silu(800.0) == 800.0
    assert oracle.silu(-800.0) == 0.0


def test_bf16_widening():
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x0000) == 0.0
    assert oracle.bf16_to_double(0x3F81) == 1.0 + 2.0 ** -7
    assert oracle.bf16_to_double(0x0001) == 2.0 ** -133
    assert oracle.bf16_to_double(0x7F7F) == (2 - 2.0 ** -7) * 2.0 ** 127


def test_bad_shapes_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.pack(np.zeros((2, 48), np.int8))
    bad = np.zeros((2, 64), np.int8)
    bad[1, 3] = 2
    with pytest.raises(oracle.OracleError):
        oracle.pack(bad)


def test_threaded_rows_match_serial():
    rng = np.random.default_rng(15)
    rows, k = 300, 512
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    codes = oracle.pack(t)
    x = synth.activations(rng, 2, k)
    y1 = oracle.gemm(codes, scale, k, x, threads=1)
    y4 = oracle.gemm(codes, scale, k, x, threads=4)
    assert np.array_equal(y1, y4)
    sub = [3, 77, 299]
    ys = oracle.gemm(codes, scale, k, x, rows_subset=sub)
    assert np.array_equal(ys[:, sub], y1[:, sub])
