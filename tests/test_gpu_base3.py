"""GPU parity of the base-3 format (tern5_gemm, tern5_unpack) against the
oracle's gemm5 and unpack5, through the C ABI: bit-exact unpack, products
element by element at the standard bar |y - y_ref| <= max(1e-3 |y_ref|,
1e-4) for m = 1 .. 8 over ragged row counts and the Neutrino widths padded
to a multiple of 80 (4160, 12320), integer activations bit-exact, and
invalid bytes (243..255) without a fault.
"""
import numpy as np
import pytest

import oracle
import packed_bit_gemv_tern_b300 as tern
from packed_bit_gemv_tern_b300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-3, 1e-4


def _dev_x(xb):
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).cuda().view(torch.bfloat16)


def _mat(rng, rows, k):
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    codes, _ = tern.tern5_pack(t)
    return tern.Tern5Matrix.from_host(codes, scale, k), codes, scale, t


def _close(y, ref, what):
    err = np.abs(y.astype(np.float64) - ref)
    bound = np.maximum(RTOL * np.abs(ref), ATOL)
    assert (err <= bound).all(), f"{what}: max ratio {(err / bound).max():.3f}"


@pytest.mark.parametrize("rows,k", [(1, 80), (129, 400), (1000, 4160), (300, 12320)])
def test_unpack_exact(rows, k):
    rng = np.random.default_rng(rows + k)
    w, codes, scale, t = _mat(rng, rows, k)
    out = torch.empty((rows, k), dtype=torch.int8, device="cuda")
    tern.tern5_unpack(w, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), t)


@pytest.mark.parametrize("m", [1, 2, 3, 5, 7, 8])
@pytest.mark.parametrize("rows,k", [(1, 80), (257, 4160), (4096, 4160), (1000, 12320)])
def test_gemm_parity(m, rows, k):
    rng = np.random.default_rng(10 * m + rows + k)
    w, codes, scale, _ = _mat(rng, rows, k)
    xb = synth.activations(rng, m, k)
    y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    if m * k * 2 > tern.TERN_MAX_X_BYTES:
        # the staged activations would not fit in shared memory: refused on
        # the host before any launch, y untouched
        with pytest.raises(tern.TernError) as e:
            tern.tern5_gemm(w, _dev_x(xb), m, y)
        assert e.value.status == tern.TERN_ERR_SHAPE
        torch.cuda.synchronize()
        assert torch.isnan(y).all()
        return
    tern.tern5_gemm(w, _dev_x(xb), m, y)
    torch.cuda.synchronize()
    _close(y.cpu().numpy(), oracle.gemm5(codes, scale, k, xb, threads=8), f"m={m} {rows}x{k}")


def test_integer_activations_bit_exact():
    rng = np.random.default_rng(3)
    rows, k, m = 512, 4160, 3
    w, codes, _, t = _mat(rng, rows, k)
    scale = np.ones(rows, dtype=np.float32)
    w = tern.Tern5Matrix.from_host(codes, scale, k)
    xi = rng.integers(-2, 3, (m, k)).astype(np.float32)
    xb = synth.f32_to_bf16_bits(xi)
    y = torch.empty((m, rows), dtype=torch.float32, device="cuda")
    tern.tern5_gemm(w, _dev_x(xb), m, y)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().astype(np.float64), oracle.gemm5(codes, scale, k, xb))


def test_invalid_bytes_do_not_fault():
    rng = np.random.default_rng(4)
    rows, k = 64, 400
    _, codes, scale, _ = _mat(rng, rows, k)
    codes = codes.copy()
    codes[3, 5] = 250
    codes[40, 0] = 255
    w = tern.Tern5Matrix.from_host(codes, scale, k)
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    tern.tern5_gemm(w, _dev_x(synth.activations(rng, 1, k)), 1, y)
    out = torch.empty((rows, k), dtype=torch.int8, device="cuda")
    tern.tern5_unpack(w, out)
    torch.cuda.synchronize()
    assert tern.tern_last_device_error() == tern.TERN_OK
    assert (out.cpu().numpy()[3, 25:30] == -2).all()
