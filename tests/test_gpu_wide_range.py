"""GPU parity on activations with a wide dynamic range, through the C ABI.

The tensor-core kernels feed the activations to the MMA as e4m3 terms under
power-of-two row scales, so their exactness depends on where each element
sits relative to the row maximum.  These rows put the maximum far above the
bulk: a few outlier channels at 2^7 .. 2^15 over N(0, 1) (per-row or shared
channels), and a unit maximum over a bulk at 2^-8 .. 2^-20.  Every element is
compared with the fp64 oracle at the same bar as the other parity tests:
|y - y_ref| <= max(1e-3 |y_ref|, 1e-4).
"""
import numpy as np
import pytest

import oracle
import packed_bit_gemv_tern_b300 as tern
from packed_bit_gemv_tern_b300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-3, 1e-4
THREADS = 8
MAGNITUDES = [2.0 ** 7, 2.0 ** 10, 2.0 ** 13, 2.0 ** 15]


def _close(y_gpu, y_ref, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bound = np.maximum(RTOL * np.abs(y_ref), ATOL)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                           f"max err {err.max():.3e}, worst ratio {(err / bound).max():.3f}")


def _dev_x(xb):
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).cuda().view(torch.bfloat16)


def _mat(rng, rows, k):
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    codes, rowsum = tern.tern_pack(t)
    return tern.TernMatrix.from_host(codes, scale, k, rowsum), codes, scale


def _x_cases(rng, m, k):
    cases = []
    for mag in MAGNITUDES:
        cases.append((f"outliers 2^{int(np.log2(mag))}", synth.outlier_activations(rng, m, k, mag)))
        cases.append((f"shared outliers 2^{int(np.log2(mag))}",
                      synth.outlier_activations(rng, m, k, mag, n_outliers=6, shared_channels=True)))
    for b in (-8, -14, -20):
        cases.append((f"bulk at 2^{b}", synth.far_bulk_activations(rng, m, k, b)))
    return cases


@pytest.mark.parametrize("rows,k", [(4096, 4096), (1024, 12288)])
def test_gemv_wide_range(rows, k):
    rng = np.random.default_rng(7000 + k)
    w, codes, scale = _mat(rng, rows, k)
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    for name, xb in _x_cases(rng, 1, k):
        tern.tern_gemv(w, _dev_x(xb), y)
        torch.cuda.synchronize()
        _close(y.cpu().numpy(), oracle.gemm(codes, scale, k, xb, threads=THREADS), f"gemv {rows}x{k} {name}")
    assert tern.tern_last_device_error() == tern.TERN_OK


@pytest.mark.parametrize("m", [2, 4, 7, 8])
@pytest.mark.parametrize("rows,k", [(1024, 4096), (512, 12288)])
def test_smallm_wide_range(m, rows, k):
    rng = np.random.default_rng(7100 + 10 * m + k)
    w, codes, scale = _mat(rng, rows, k)
    y = torch.empty((m, rows), dtype=torch.float32, device="cuda")
    for name, xb in _x_cases(rng, m, k):
        tern.tern_gemm_smallm(w, _dev_x(xb), m, y)
        torch.cuda.synchronize()
        _close(y.cpu().numpy(), oracle.gemm(codes, scale, k, xb, threads=THREADS),
               f"smallm m={m} {rows}x{k} {name}")


@pytest.mark.parametrize("m", [1, 7])
def test_swiglu_wide_range(m):
    rows, k = 768, 4096
    rng = np.random.default_rng(7200 + m)
    wg, cg, sg = _mat(rng, rows, k)
    wu, cu, su = _mat(rng, rows, k)
    h = torch.empty((m, rows), dtype=torch.float32, device="cuda")
    for name, xb in _x_cases(rng, m, k):
        tern.tern_gemm_smallm_swiglu(wg, wu, _dev_x(xb), m, h)
        torch.cuda.synchronize()
        _close(h.cpu().numpy(), oracle.swiglu(cg, sg, cu, su, k, xb, threads=THREADS), f"swiglu m={m} {name}")


def test_batched_wide_range():
    """One persistent launch over items of every activation class at once;
    the preparing launch picks one or two bands per item and chunk."""
    rng = np.random.default_rng(7300)
    specs = [(4096, 4096, 1), (1024, 12288, 1), (1024, 4096, 3), (512, 12288, 7), (640, 4096, 8)]
    items, refs = [], []
    for rows, k, m in specs:
        w, codes, scale = _mat(rng, rows, k)
        for name, xb in _x_cases(rng, m, k):
            y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
            items.append((w, None, _dev_x(xb), y, m))
            refs.append((f"batched {rows}x{k} m={m} {name}", codes, scale, k, xb))
    tern.tern_gemm_batched(items)
    torch.cuda.synchronize()
    assert tern.tern_last_device_error() == tern.TERN_OK
    for it, (what, codes, scale, k, xb) in zip(items, refs):
        _close(it[3].cpu().numpy(), oracle.gemm(codes, scale, k, xb, threads=THREADS), what)


def test_batched_outliers_in_one_chunk():
    """Outlier channels inside one K range only, so that a tile's chunks mix
    the one-band operand and the two-band one (which takes both operand
    buffers): m = 1 at K = 32768 (two chunks), m = 3 and 7 at K = 12288, and
    a SwiGLU pair; plus plain N(0, 1) items between them.  Two calls in a
    row, every element against the oracle."""
    rng = np.random.default_rng(7400)
    specs = [(1024, 32768, 1, False, (20000, 20006)), (300, 12288, 3, False, (5000, 5003)),
             (512, 12288, 7, False, (6000, 6004)), (640, 4096, 7, True, (100, 103)),
             (4096, 4096, 1, False, None), (1024, 12288, 7, False, None)]
    for call in range(2):
        items, refs = [], []
        for rows, k, m, sw, band in specs:
            w, codes, scale = _mat(rng, rows, k)
            x = rng.standard_normal((m, k), dtype=np.float32)
            if band is not None:
                ch = np.arange(band[0], band[1])
                x[:, ch] = np.where(rng.random((m, ch.size)) < 0.5, -1.0, 1.0).astype(np.float32) * np.float32(2.0 ** 14)
            xb = synth.f32_to_bf16_bits(x)
            y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
            if sw:
                wu, cu, su = _mat(rng, rows, k)
                items.append((w, wu, _dev_x(xb), y, m))
                refs.append((f"call {call} swiglu {rows}x{k} m={m}", lambda c=codes, s=scale, cu=cu, su=su, k=k, xb=xb:
                             oracle.swiglu(c, s, cu, su, k, xb, threads=THREADS)))
            else:
                items.append((w, None, _dev_x(xb), y, m))
                refs.append((f"call {call} {rows}x{k} m={m}", lambda c=codes, s=scale, k=k, xb=xb:
                             oracle.gemm(c, s, k, xb, threads=THREADS)))
        tern.tern_gemm_batched(items)
        torch.cuda.synchronize()
        assert tern.tern_last_device_error() == tern.TERN_OK
        for it, (what, ref) in zip(items, refs):
            _close(it[3].cpu().numpy(), ref(), what)
