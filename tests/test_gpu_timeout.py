"""The bounded device waits, run out on purpose (no fault, no hang).

Every mbarrier wait of the tensor-core kernels gives up after a bound of SM
cycles; the kernel then records TERN_ERR_TIMEOUT, stops every role, waits
(with the default bound) for its own copies and MMAs in flight, releases its
tensor memory and returns.  Here the bound is set to 64 cycles, shorter than
any DRAM round trip, so the first wait for a weight stage runs out in every
kernel family: the split-K single-call kernel (plain and SwiGLU), and the
persistent batched kernel with an in-kernel operand build (m = 1) and a
prepared one (m = 7).  Then the default bound is restored and the same calls
must give correct results on the same context.
"""
import numpy as np
import pytest

import oracle
import packed_bit_gemv_tern_b300 as tern
from packed_bit_gemv_tern_b300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _mat(rng, rows, k):
    t = synth.ternary(rng, rows, k)
    codes, rowsum = tern.tern_pack(t)
    sc = synth.scales(rng, rows)
    return tern.TernMatrix.from_host(codes, sc, k, rowsum), codes, sc


def _x(xb):
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).cuda().view(torch.bfloat16)


def _close(got, ref):
    err = np.abs(got.astype(np.float64) - ref)
    assert (err <= np.maximum(1e-3 * np.abs(ref), 1e-4)).all(), float(err.max())


def test_bounded_waits_run_out_and_the_context_survives():
    rng = np.random.default_rng(31)
    w, cw, sw = _mat(rng, 4096, 4096)
    wu, cu, su = _mat(rng, 4096, 4096)
    w7, c7, s7 = _mat(rng, 1024, 4096)
    x1, x7 = synth.activations(rng, 1, 4096), synth.activations(rng, 7, 4096)
    d1, d7 = _x(x1), _x(x7)
    y = torch.empty((1, 4096), device="cuda")
    h = torch.empty((7, 4096), device="cuda")
    yb = torch.empty((1, 4096), device="cuda")
    yb7 = torch.empty((7, 1024), device="cuda")
    torch.cuda.synchronize()
    assert tern.tern_last_device_error() == tern.TERN_OK

    def calls():
        yield "gemv", lambda: tern.tern_gemv(w, d1, y)
        yield "smallm_swiglu", lambda: tern.tern_gemm_smallm_swiglu(w, wu, d7, 7, h)
        yield "batched", lambda: tern.tern_gemm_batched([(w, None, d1, yb, 1), (w7, None, d7, yb7, 7)])

    tern.tern_set_wait_limit(64)
    try:
        for name, fn in calls():
            fn()
            assert tern.tern_last_device_error() == tern.TERN_ERR_TIMEOUT, name
    finally:
        tern.tern_set_wait_limit(0)
    for name, fn in calls():
        fn()
        assert tern.tern_last_device_error() == tern.TERN_OK, name
    _close(y.cpu().numpy(), oracle.gemm(cw, sw, 4096, x1, threads=8))
    _close(h.cpu().numpy(), oracle.swiglu(cw, sw, cu, su, 4096, x7, threads=8))
    _close(yb.cpu().numpy(), oracle.gemm(cw, sw, 4096, x1, threads=8))
    _close(yb7.cpu().numpy(), oracle.gemm(c7, s7, 4096, x7, threads=8))
