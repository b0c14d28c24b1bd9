"""GPU parity of the RMSNorm prologue (tern_gemm_batched_rmsnorm) against the
oracle's rmsnorm_gemm / rmsnorm_swiglu, through the C ABI.

Shapes follow the Neutrino-1 linears the norm precedes or shares a launch
with: q/k/v-like 4096 x 4096 at m = 1, the gate/up pair 12288 x 4096 and the
down projection 4096 x 12288 at m = 1 (decode) and m = 7 (verification).
Large items are compared on sampled rows (the oracle's rows_subset), every
activation row and every sampled output against the standard bar
|y - y_ref| <= max(1e-3 |y_ref|, 1e-4).  Also: items with and without a norm
in one launch, K split into two chunks at m = 1 (the mean square spans
both), outlier channels that need the two-band operand after the norm, rows
where eps decides the factor, and eps = 0.
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


def _close(y_gpu, y_ref, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bound = np.maximum(RTOL * np.abs(y_ref), ATOL)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                           f"max err {err.max():.3e}, worst ratio {(err / bound).max():.3f}")


def _dev_x(xb):
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).cuda().view(torch.bfloat16)


def _dev_g(g):
    return torch.from_numpy(np.ascontiguousarray(g, dtype=np.float32)).cuda()


def _mat(rng, rows, k, p_zero=synth.P_ZERO):
    t = synth.ternary(rng, rows, k, p_zero=p_zero)
    scale = synth.scales(rng, rows)
    codes, rowsum = tern.tern_pack(t)
    return tern.TernMatrix.from_host(codes, scale, k, rowsum), codes, scale


def _weights(rng, k, spikes=0):
    g = rng.uniform(0.5, 1.5, k).astype(np.float32)
    if spikes:
        g[rng.choice(k, spikes, replace=False)] = np.float32(64.0)
    return g


def _x(rng, m, k):
    return synth.f32_to_bf16_bits(rng.standard_normal((m, k), dtype=np.float32) * np.float32(3.0))


def _rows(rng, rows, n=384):
    return None if rows <= n else np.sort(rng.choice(rows, n, replace=False))


class _Batch:
    """Items for one call, each with its oracle reference."""

    def __init__(self):
        self.items, self.norms, self.refs = [], [], []

    def add(self, rng, rows, k, m, swiglu=False, norm=True, x=None, g=None, eps_ref=1e-6, p_zero=synth.P_ZERO):
        w, codes, scale = _mat(rng, rows, k, p_zero)
        xb = _x(rng, m, k) if x is None else x
        g = _weights(rng, k) if (norm and g is None) else g
        y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
        sub = _rows(rng, rows)
        eps = float(np.float32(eps_ref))
        if swiglu:
            wu, cu, su = _mat(rng, rows, k, p_zero)
            self.items.append((w, wu, _dev_x(xb), y, m))
            if norm:
                ref = lambda: oracle.rmsnorm_swiglu(codes, scale, cu, su, k, xb, g, eps, THREADS, sub)
            else:
                ref = lambda: oracle.swiglu(codes, scale, cu, su, k, xb, THREADS, sub)
        else:
            self.items.append((w, None, _dev_x(xb), y, m))
            if norm:
                ref = lambda: oracle.rmsnorm_gemm(codes, scale, k, xb, g, eps, THREADS, sub)
            else:
                ref = lambda: oracle.gemm(codes, scale, k, xb, THREADS, sub)
        self.norms.append(_dev_g(g) if norm else None)
        self.refs.append((f"{rows}x{k} m={m}{' swiglu' if swiglu else ''}{' norm' if norm else ''}", sub, ref))

    def run_and_check(self, eps=1e-6):
        tern.tern_gemm_batched_rmsnorm(self.items, self.norms, eps)
        torch.cuda.synchronize()
        assert tern.tern_last_device_error() == tern.TERN_OK
        for it, (what, sub, ref) in zip(self.items, self.refs):
            y = it[3].cpu().numpy()
            want = ref()
            _close(y if sub is None else y[:, sub], want if sub is None else want[:, sub], what)


def test_rmsnorm_decode_shapes():
    """m = 1: q/k/v-like, the gate/up pair and down, each behind a norm."""
    rng = np.random.default_rng(8100)
    b = _Batch()
    for _ in range(3):
        b.add(rng, 4096, 4096, 1)
    b.add(rng, 12288, 4096, 1, swiglu=True)
    b.add(rng, 4096, 12288, 1)
    b.run_and_check()


@pytest.mark.parametrize("m", [2, 7, 8])
def test_rmsnorm_verify_shapes(m):
    """m >= 2 (the preparing kernel normalises): gate/up pair and down."""
    rng = np.random.default_rng(8200 + m)
    b = _Batch()
    b.add(rng, 12288, 4096, m, swiglu=True)
    b.add(rng, 4096, 12288, m)
    b.add(rng, 1024, 4096, m)
    b.run_and_check()


def test_rmsnorm_mixed_with_plain_items():
    """Items with and without a norm in one launch, m = 1 and m = 7, sharing
    one activation buffer as q, k and v do."""
    rng = np.random.default_rng(8300)
    b = _Batch()
    x1 = _x(rng, 1, 4096)
    g1 = _weights(rng, 4096)
    for norm in (True, False, True):
        b.add(rng, 1024, 4096, 1, x=x1, g=g1 if norm else None, norm=norm)
    x7 = _x(rng, 7, 4096)
    b.add(rng, 640, 4096, 7, x=x7, norm=False)
    b.add(rng, 640, 4096, 7, x=x7, g=g1)
    b.add(rng, 512, 4096, 3, swiglu=True, norm=False)
    b.run_and_check()


def test_rmsnorm_two_chunks_at_m1():
    """K = 32768 at m = 1 takes two K chunks: each chunk's build uses the
    whole row's mean square."""
    rng = np.random.default_rng(8400)
    b = _Batch()
    b.add(rng, 512, 32768, 1)
    b.add(rng, 256, 32768, 2)
    b.run_and_check()


def test_rmsnorm_outlier_channels():
    """Channel weights of 64 on a few channels make outliers after the norm,
    so chunks need the two-band operand, rebuilt from x with the row factor."""
    rng = np.random.default_rng(8500)
    b = _Batch()
    for m, rows, k in [(1, 1024, 4096), (1, 512, 12288), (7, 512, 4096), (3, 300, 12288)]:
        b.add(rng, rows, k, m, g=_weights(rng, k, spikes=4))
    b.add(rng, 640, 4096, 7, swiglu=True, g=_weights(rng, 4096, spikes=3))
    b.run_and_check()


@pytest.mark.parametrize("eps", [0.0, 1e-6, 1e-2])
def test_rmsnorm_eps_values(eps):
    """eps = 0, the page's 1e-6, and a large eps, on ordinary rows and on
    tiny rows where eps decides the factor."""
    rng = np.random.default_rng(8600 + int(eps * 1e6))
    b = _Batch()
    tiny1 = synth.f32_to_bf16_bits(rng.standard_normal((1, 4096), dtype=np.float32) * np.float32(2.0 ** -12))
    tiny7 = synth.f32_to_bf16_bits(rng.standard_normal((7, 4096), dtype=np.float32) * np.float32(2.0 ** -12))
    b.add(rng, 1024, 4096, 1, eps_ref=eps)
    b.add(rng, 1024, 4096, 1, x=tiny1, eps_ref=eps)
    b.add(rng, 512, 4096, 7, x=tiny7, eps_ref=eps)
    b.run_and_check(eps)
