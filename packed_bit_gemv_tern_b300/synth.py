"""Seeded synthetic inputs for the ternary linear layers.

This module only draws random numbers.  It holds none of the method's
arithmetic: no packing, decoding or accumulation.  Both the CUDA path and the
CPU oracle take their inputs from here, so the two see identical values.

What is drawn, and why it looks the way it does:

* ternary weights ``t`` (int8 in {-1, 0, +1}), i.i.d. per element with the
  code mix the Neutrino-1 8B model page reports for its coded lane
  ("Inside the coded lane": 62.63 % zero, 18.68 % plus, 18.69 % minus;
  early feed-forward gate/down layers at 70-72 % zero);
* one fp32 scale per output row, uniform on [0.005, 0.05];
* bf16 activations, round-to-nearest-even of N(0, 1) fp32 samples, returned as
  their raw uint16 bit patterns (the C boundary takes bf16 as uint16 bits).

Every draw uses ``numpy.random.default_rng(seed)`` (PCG64) so a seed fixes the
whole workload.
"""
from __future__ import annotations

import numpy as np

# Code mix of the whole coded lane ("Inside the coded lane").
P_ZERO = 0.6263
P_PLUS = 0.1868
P_MINUS = 0.1869

SCALE_LO = 0.005
SCALE_HI = 0.05


def ternary(rng: np.random.Generator, rows: int, k: int,
            p_zero: float = P_ZERO, p_plus: float | None = None) -> np.ndarray:
    """int8 [rows, k] with P(0)=p_zero, P(+1)=p_plus, P(-1)=rest.

    When ``p_plus`` is None the non-zero mass is split evenly.
    Drawn as uint32 uniforms thresholded at the cumulative probabilities.
    """
    if p_plus is None:
        p_plus = (1.0 - p_zero) / 2.0
    if not (0.0 <= p_zero <= 1.0 and 0.0 <= p_plus <= 1.0 - p_zero):
        raise ValueError("bad code probabilities")
    out = np.empty((rows, k), dtype=np.int8)
    if rows == 0 or k == 0:
        return out
    t0 = np.uint32(min(int(round(p_zero * 2**32)), 2**32 - 1))
    t1 = np.uint32(min(int(round((p_zero + p_plus) * 2**32)), 2**32 - 1))
    step = max(1, (1 << 24) // max(k, 1))  # bound the temporary to ~64 MB
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        u = rng.integers(0, 2**32, size=(r1 - r0, k), dtype=np.uint32)
        blk = out[r0:r1]
        blk[...] = -1
        blk[u < t1] = 1
        blk[u < t0] = 0
    return out


def scales(rng: np.random.Generator, rows: int,
           lo: float = SCALE_LO, hi: float = SCALE_HI) -> np.ndarray:
    """fp32 [rows], uniform on [lo, hi)."""
    return rng.uniform(lo, hi, size=rows).astype(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns.

    Inputs here are finite normal-distribution samples; NaN/Inf are not drawn.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(rng: np.random.Generator, m: int, k: int) -> np.ndarray:
    """bf16 bits [m, k] of N(0, 1) samples."""
    return f32_to_bf16_bits(rng.standard_normal((m, k), dtype=np.float32))


def outlier_activations(rng: np.random.Generator, m: int, k: int, magnitude: float,
                        n_outliers: int = 3, shared_channels: bool = False) -> np.ndarray:
    """bf16 bits [m, k]: N(0, 1) samples with ``n_outliers`` channels per row
    replaced by +-``magnitude`` (random sign).

    Decoder activations carry a few channels far above the rest; these rows
    put the row maximum ``magnitude`` above a bulk of unit scale.  With
    ``shared_channels`` every row uses the same outlier channels (fixed
    outlier dimensions), otherwise each row draws its own.
    """
    x = rng.standard_normal((m, k), dtype=np.float32)
    n = min(n_outliers, k)
    shared = rng.choice(k, size=n, replace=False)
    for i in range(m):
        ch = shared if shared_channels else rng.choice(k, size=n, replace=False)
        x[i, ch] = np.where(rng.random(n) < 0.5, -1.0, 1.0).astype(np.float32) * np.float32(magnitude)
    return f32_to_bf16_bits(x)


def far_bulk_activations(rng: np.random.Generator, m: int, k: int, bulk_log2: int) -> np.ndarray:
    """bf16 bits [m, k]: a bulk of N(0, 1) * 2**bulk_log2 with one element per
    row of magnitude 1 (the row maximum sits far above everything else)."""
    x = rng.standard_normal((m, k), dtype=np.float32) * np.float32(2.0 ** bulk_log2)
    for i in range(m):
        x[i, rng.integers(0, k)] = np.float32(1.0 if rng.random() < 0.5 else -1.0)
    return f32_to_bf16_bits(x)


def small_int_activations(rng: np.random.Generator, m: int, k: int,
                          lo: int = -2, hi: int = 2) -> np.ndarray:
    """bf16 bits [m, k] of integers in [lo, hi] (exact in bf16).

    With |partial sums| < 2**24 every fp32 summation order is exact, which lets
    a test demand bit-exact accumulators.
    """
    v = rng.integers(lo, hi + 1, size=(m, k)).astype(np.float32)
    return f32_to_bf16_bits(v)


class Linear:
    """One drawn ternary projection: t [rows, k] int8 and scale [rows] fp32."""

    def __init__(self, t: np.ndarray, scale: np.ndarray, name: str = ""):
        self.t = t
        self.scale = scale
        self.name = name

    @property
    def rows(self) -> int:
        return int(self.t.shape[0])

    @property
    def k(self) -> int:
        return int(self.t.shape[1])


def linear(rng: np.random.Generator, rows: int, k: int, p_zero: float = P_ZERO,
           p_plus: float | None = None, name: str = "") -> Linear:
    t = ternary(rng, rows, k, p_zero, p_plus)
    return Linear(t, scales(rng, rows), name)


# ---------------------------------------------------------------------------
# Workloads.  Shapes follow the Neutrino-1 8B spec table (36 decoder layers,
# hidden 4,096, gated feed-forward 12,288 with three linears per layer,
# grouped-query attention 32 query : 8 key-value heads of width 128, so
# q/o are 4096x4096 and k/v are 1024x4096).
# ---------------------------------------------------------------------------
HIDDEN = 4096
FFN = 12288
KV_ROWS = 1024
LAYERS = 36

# (name, rows, k) of the seven linears of one decoder layer, in call order.
LAYER_LINEARS = (
    ("q", HIDDEN, HIDDEN),
    ("k", KV_ROWS, HIDDEN),
    ("v", KV_ROWS, HIDDEN),
    ("o", HIDDEN, HIDDEN),
    ("gate", FFN, HIDDEN),
    ("up", FFN, HIDDEN),
    ("down", HIDDEN, FFN),
)


def sweep_zero_fraction(layer: int, name: str) -> float:
    """Zero fraction used for one linear of the 36-layer sweep.

    Attention projections: 0.62 at every depth.  The model page says the gate
    and down feed-forward projections reach 70-72 % zeros in layers 1-3; this
    workload reads that as 0.72 / 0.71 / 0.70 for layers 1 / 2 / 3 on gate and
    down, and 0.62 everywhere else (up included).
    """
    if name in ("gate", "down") and layer in (1, 2, 3):
        return {1: 0.72, 2: 0.71, 3: 0.70}[layer]
    return 0.62


WORKLOADS = {
    "c0": dict(desc="ternary GEMV M=1, 1024x4096 (k_proj shape)", seed=0),
    "c1": dict(desc="ternary GEMV M=1, 4096x4096 (q/o projection shape)", seed=1),
    "c2": dict(desc="M=1 down 4096x12288 (P0=0.71) + fused gate/up 2x12288x4096 SiLU(g)*u", seed=2),
    "c3": dict(desc="M=7 speculative-verify: gate/up 12288x4096 (fused SwiGLU) + down 4096x12288", seed=3),
    "c4": dict(desc="36-layer linear sweep at M=1, 252 linears, 6,945,767,424 codes", seed=4),
}
