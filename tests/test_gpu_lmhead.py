"""GPU parity of the int8 output head with the fused greedy choice
(tern_lmhead_argmax) against the oracle's i8_gemm and argmax, through the C
ABI.

Logits: |y - y_ref| <= max(1e-3 |y_ref|, E), where E bounds the kernel's
fp32 arithmetic: every product enters exactly (two e4m3 nibble terms per
weight times e4m3 activation terms), and each logit is a chain of at most
K/32 + 8 fp32 roundings of partial sums no larger than
sum_k (|w| + 128) |x| (the offset-binary nibbles), so
E = (K/32 + 8) 2^-24 scale sum_k (|w_k| + 128) |x_k|.
Index: bit-exact with the argmax of the kernel's own fp32 logits (lowest
index on ties), and equal to the oracle's unless the oracle's two best
logits are closer than the bound (then the kernel's choice must be within
the bound of the best).
Cases: the full 151,936 x 4,096 head at m = 1 and m = 7 (the verify pass),
planted ties, ragged row counts, other K, m up to 8, the final RMSNorm, and
activations with outlier channels (the two-band operand).
"""
import numpy as np
import pytest

import oracle
import packed_bit_gemv_tern_b300 as tern
from packed_bit_gemv_tern_b300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

THREADS = 16
HEAD_ROWS, HEAD_K = 151936, 4096


def _head(rng, rows, k):
    w = rng.integers(-128, 128, (rows, k), dtype=np.int16).astype(np.int8)
    scale = rng.uniform(0.5e-3, 2e-3, rows).astype(np.float32)
    return w, scale


def _dev_x(xb):
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).cuda().view(torch.bfloat16)


def _run(w, scale, xb, norm=None, eps=1e-6, dw=None):
    m, k = xb.shape
    dw = tern.I8Matrix.from_host(w, scale) if dw is None else dw
    logits = torch.full((m, w.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
    am = torch.full((m,), -1, dtype=torch.int32, device="cuda")
    g = None if norm is None else torch.from_numpy(norm).cuda()
    tern.tern_lmhead_argmax(dw, _dev_x(xb), m, logits, am, norm_w=g, eps=eps)
    torch.cuda.synchronize()
    assert tern.tern_last_device_error() == tern.TERN_OK
    return logits.cpu().numpy().astype(np.float64), am.cpu().numpy().astype(np.int64)


def _check(w, scale, xb, y, idx, xref=None, what=""):
    """xref: the bf16 activations the oracle should see (the normalised rows
    when the call normalises)."""
    xr = xb if xref is None else xref
    y_ref, a_ref = oracle.i8_gemm(w, scale, xr, threads=THREADS, with_abs=True)
    k = w.shape[1]
    xa = np.abs(synth.bf16_bits_to_f32(xr).astype(np.float64)).sum(axis=1)
    # scale * sum_k (|w| + 128) |x| per logit
    big = a_ref + 128.0 * xa[:, None] * np.abs(scale.astype(np.float64))[None, :]
    bound = np.maximum(1e-3 * np.abs(y_ref), (k / 32 + 8) * 2.0 ** -24 * big)
    err = np.abs(y - y_ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} logits outside the bound; "
                           f"worst ratio {(err / bound).max():.3f}")
    # the index is the first maximum of the kernel's own logits
    assert np.array_equal(idx, np.argmax(y, axis=1)), what
    ref_idx = oracle.argmax(y_ref)
    for i in range(y.shape[0]):
        if idx[i] != ref_idx[i]:
            top = y_ref[i, ref_idx[i]]
            assert top - y_ref[i, idx[i]] <= 2 * bound[i, ref_idx[i]], (what, i, idx[i], ref_idx[i])


@pytest.fixture(scope="module")
def full_head():
    rng = np.random.default_rng(9100)
    w, scale = _head(rng, HEAD_ROWS, HEAD_K)
    return w, scale, tern.I8Matrix.from_host(w, scale)


@pytest.mark.parametrize("m", [1, 7])
def test_full_head(full_head, m):
    w, scale, dw = full_head
    rng = np.random.default_rng(9200 + m)
    xb = synth.f32_to_bf16_bits(rng.standard_normal((m, HEAD_K), dtype=np.float32))
    y, idx = _run(w, scale, xb, dw=dw)
    _check(w, scale, xb, y, idx, what=f"head m={m}")


def test_planted_ties_take_the_lowest_row():
    """Three identical rows that beat every other row: the lowest wins, in
    every activation row."""
    rng = np.random.default_rng(9300)
    rows, k = 5000, 4096
    w, scale = _head(rng, rows, k)
    xb = synth.f32_to_bf16_bits(np.abs(rng.standard_normal((3, k), dtype=np.float32)) + np.float32(0.1))
    best = np.full(k, 127, dtype=np.int8)
    for r in (4321, 777, 4999):
        w[r] = best
        scale[r] = np.float32(1e-3)
    scale[:] = np.float32(1e-3)
    y, idx = _run(w, scale, xb)
    assert list(idx) == [777, 777, 777]
    _check(w, scale, xb, y, idx, what="ties")


@pytest.mark.parametrize("rows,k,m", [(1, 64, 1), (129, 4096, 2), (1000, 1024, 8), (3333, 8192, 3),
                                      (300, 12288, 7)])
def test_shapes(rows, k, m):
    rng = np.random.default_rng(9400 + rows + m)
    w, scale = _head(rng, rows, k)
    xb = synth.f32_to_bf16_bits(rng.standard_normal((m, k), dtype=np.float32) * np.float32(2.0))
    y, idx = _run(w, scale, xb)
    _check(w, scale, xb, y, idx, what=f"{rows}x{k} m={m}")


@pytest.mark.parametrize("m", [1, 7])
def test_final_norm(m):
    rng = np.random.default_rng(9500 + m)
    rows, k = 20000, 4096
    w, scale = _head(rng, rows, k)
    xb = synth.f32_to_bf16_bits(rng.standard_normal((m, k), dtype=np.float32) * np.float32(5.0))
    g = rng.uniform(0.5, 1.5, k).astype(np.float32)
    y, idx = _run(w, scale, xb, norm=g)
    xn, _ = oracle.rmsnorm(xb, g, float(np.float32(1e-6)))
    _check(w, scale, xb, y, idx, xref=xn, what=f"norm m={m}")


@pytest.mark.parametrize("m", [1, 3, 7])
def test_outlier_channels(m):
    rng = np.random.default_rng(9600 + m)
    rows, k = 4000, 4096
    w, scale = _head(rng, rows, k)
    for mag in (2.0 ** 10, 2.0 ** 15):
        xb = synth.outlier_activations(rng, m, k, mag)
        y, idx = _run(w, scale, xb)
        _check(w, scale, xb, y, idx, what=f"outliers 2^{int(np.log2(mag))} m={m}")
