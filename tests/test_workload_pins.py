"""Pins of the synthetic workload against figures printed on the Neutrino-1 8B
model page (geometry, byte budget, code mix)."""
import os

import numpy as np

from packed_bit_gemv_tern_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _figures():
    out = {}
    with open(os.path.join(GOLDEN, "neutrino_page_figures.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = [s.strip() for s in line.split("=")]
                out[k] = float(v) if "." in v else int(v)
    return out


def test_geometry_matches_page():
    fig = _figures()
    assert synth.LAYERS == fig["decoder_layers"]
    assert synth.HIDDEN == fig["hidden"]
    assert synth.FFN == fig["ffn"]
    assert synth.KV_ROWS == fig["kv_heads"] * fig["head_width"]
    assert synth.HIDDEN == fig["query_heads"] * fig["head_width"]
    n_linears = synth.LAYERS * len(synth.LAYER_LINEARS)
    assert n_linears == fig["coded_linears"]
    codes_per_layer = sum(r * k for _, r, k in synth.LAYER_LINEARS)
    coded = synth.LAYERS * codes_per_layer
    assert coded == 6_945_767_424  # "6.95B coded projection weights"
    # parameters = coded + two untied int8 vocab tensors + norm weights
    norm = synth.LAYERS * (2 * synth.HIDDEN + 2 * fig["head_width"]) + synth.HIDDEN
    assert synth.LAYERS * 4 + 1 == fig["norm_tensors"]
    assert coded + 2 * fig["vocab"] * fig["hidden"] + norm == fig["parameters"]
    # The page's coded lane spends 72,351,744 bytes per layer: exactly 3.0 bits
    # per weight.  This project's format spends 2 bits per weight.
    assert fig["coded_bytes_per_layer"] * 8 == 3 * codes_per_layer
    assert synth.LAYERS * codes_per_layer // 4 == 1_736_441_856


def test_generator_code_mix_matches_page():
    fig = _figures()
    rng = np.random.default_rng(123)
    n = 4_000_000
    t = synth.ternary(rng, 1000, n // 1000)
    for val, key in ((0, "zero_fraction"), (1, "plus_fraction"), (-1, "minus_fraction")):
        p = fig[key]
        frac = float((t == val).mean())
        sigma = (p * (1 - p) / n) ** 0.5
        assert abs(frac - p) < 5 * sigma, (val, frac, p)


def test_sweep_zero_fractions():
    zs = [synth.sweep_zero_fraction(l, n) for l in range(36) for n, _, _ in synth.LAYER_LINEARS]
    assert len(zs) == 252
    w = [r * k for l in range(36) for _, r, k in synth.LAYER_LINEARS]
    agg = sum(z * c for z, c in zip(zs, w)) / sum(w)
    assert abs(agg - 0.6263) < 0.005  # aggregate near the page's 62.63 %
    assert synth.sweep_zero_fraction(2, "gate") == 0.71
    assert synth.sweep_zero_fraction(2, "up") == 0.62
    assert synth.sweep_zero_fraction(0, "q") == 0.62


def test_bf16_rounding_helper():
    a = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 0.0], np.float32)
    b = synth.f32_to_bf16_bits(a)
    # ties to even: 1+2^-8 -> 1.0 ; 1+3*2^-8 -> 1+2^-6
    assert b.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000]
    assert synth.bf16_bits_to_f32(b).tolist() == [1.0, 1.0, 1.0 + 2**-6, -2.5, 0.0]
