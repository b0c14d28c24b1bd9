"""tern_gemm_batched_noalloc against the existing tern_gemm_batched: the same
bytes for the same batch over two calls in a row (with new activations for
the second, so stale scratch would show), a batch whose two launch groups
both prepare activations in the one array, and an oversize batch rejected
before anything runs.  The file is named to be collected last: it must pass
both alone and after every other test in one process.

Callers that cannot allocate device memory (a serving engine that has
reserved the GPU's memory for its own pools, code that may not call
cudaMalloc) use the no-alloc entry point; these tests hold it to the
allocating one, bit for bit."""
import ctypes

import numpy as np
import pytest

import packed_bit_gemv_tern_b300 as tern
from packed_bit_gemv_tern_b300 import synth

torch = pytest.importorskip("torch")

# (rows, k, m, swiglu): plain GEMVs and small-M products, SwiGLU pairs, K over
# several chunks, ragged rows and short K
SPECS = [(4096, 4096, 1, False), (640, 4096, 7, True), (4096, 12288, 7, False), (300, 12288, 3, False),
         (33, 192, 8, True), (200, 8256, 2, False), (1, 64, 5, False), (12288, 4096, 8, True)]


def _weights(rng):
    out = []
    for rows, k, m, sw in SPECS:
        def one():
            t = synth.ternary(rng, rows, k)
            codes, rowsum = tern.tern_pack(t)
            return tern.TernMatrix.from_host(codes, synth.scales(rng, rows), k, rowsum)
        out.append((one(), one() if sw else None))
    return out


def _xs(rng):
    return [torch.from_numpy(synth.activations(rng, m, k).view(np.int16)).cuda().view(torch.bfloat16)
            for rows, k, m, sw in SPECS]


def _ys(fill):
    return [torch.full((m, rows), fill, dtype=torch.float32, device="cuda") for rows, k, m, sw in SPECS]


def _items(ws, xs, ys):
    return [(w, up, x, y, m) for (w, up), x, y, (rows, k, m, sw) in zip(ws, xs, ys, SPECS)]


@pytest.mark.gpu
def test_noalloc_matches_batched_over_two_calls():
    rng = np.random.default_rng(2024)
    ws = _weights(rng)
    xa, xb = _xs(rng), _xs(rng)
    ref_a, ref_b = _ys(0.0), _ys(0.0)
    tern.tern_gemm_batched(_items(ws, xa, ref_a))
    tern.tern_gemm_batched(_items(ws, xb, ref_b))
    torch.cuda.synchronize()
    assert tern.tern_last_device_error() == tern.TERN_OK
    got_a, got_b = _ys(float("nan")), _ys(float("nan"))
    # back to back on one stream: the second call rewrites the same scratch
    tern.tern_gemm_batched_noalloc(_items(ws, xa, got_a))
    tern.tern_gemm_batched_noalloc(_items(ws, xb, got_b))
    torch.cuda.synchronize()
    assert tern.tern_last_device_error() == tern.TERN_OK
    for i, spec in enumerate(SPECS):
        assert torch.equal(got_a[i].view(torch.int32), ref_a[i].view(torch.int32)), ("first call", spec)
        assert torch.equal(got_b[i].view(torch.int32), ref_b[i].view(torch.int32)), ("second call", spec)


@pytest.mark.gpu
def test_noalloc_two_launch_groups_share_the_array():
    """130 small items with m >= 2 take two launch groups, and each group's
    activation-preparing launch writes the array from offset 0: the second
    must not overwrite it while the first group's persistent kernel still
    reads it.  Two calls in a row, compared bit for bit with
    tern_gemm_batched, which is itself checked against the oracle."""
    import oracle
    rng = np.random.default_rng(2026)
    specs = [(64 + 32 * (i % 4), 64 * (1 + i % 8), 2 + i % 7) for i in range(130)]
    ws, cs = [], []
    for rows, k, m in specs:
        t = synth.ternary(rng, rows, k)
        codes, rowsum = tern.tern_pack(t)
        sc = synth.scales(rng, rows)
        ws.append(tern.TernMatrix.from_host(codes, sc, k, rowsum))
        cs.append((codes, sc))

    def xs():
        return [synth.activations(rng, m, k) for rows, k, m in specs]

    def run(fn, xb):
        ys = [torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda") for rows, k, m in specs]
        items = [(w, None, torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16), y, m)
                 for w, x, y, (rows, k, m) in zip(ws, xb, ys, specs)]
        assert tern.tern_gemm_batched_launches(items) == 4  # two groups, each with a preparing launch
        fn(items)
        torch.cuda.synchronize()
        assert tern.tern_last_device_error() == tern.TERN_OK
        return ys

    xa, xb = xs(), xs()
    ref_a, ref_b = run(tern.tern_gemm_batched, xa), run(tern.tern_gemm_batched, xb)
    got_a, got_b = run(tern.tern_gemm_batched_noalloc, xa), run(tern.tern_gemm_batched_noalloc, xb)
    for i, (rows, k, m) in enumerate(specs):
        assert torch.equal(got_a[i].view(torch.int32), ref_a[i].view(torch.int32)), ("first call", i)
        assert torch.equal(got_b[i].view(torch.int32), ref_b[i].view(torch.int32)), ("second call", i)
    for i in (0, 63, 64, 65, 129):  # items on both sides of the group boundary
        codes, sc = cs[i]
        ref = oracle.gemm(codes, sc, specs[i][1], xb[i], threads=4)
        got = got_b[i].cpu().numpy().astype(np.float64)
        assert (np.abs(got - ref) <= np.maximum(1e-3 * np.abs(ref), 1e-4)).all(), i


@pytest.mark.gpu
def test_noalloc_oversize_launches_nothing():
    rng = np.random.default_rng(2025)
    t = synth.ternary(rng, 64, 12288)
    codes, rowsum = tern.tern_pack(t)
    w = tern.TernMatrix.from_host(codes, synth.scales(rng, 64), 12288, rowsum)
    x = torch.zeros((8, 12288), dtype=torch.bfloat16, device="cuda")
    ys = [torch.full((8, 64), 7.0, device="cuda") for _ in range(24)]
    with pytest.raises(tern.TernError) as e:
        tern.tern_gemm_batched_noalloc([(w, None, x, y, 8) for y in ys])
    assert e.value.status == tern.TERN_ERR_SHAPE
    torch.cuda.synchronize()
    assert all(bool((y == 7.0).all()) for y in ys)


def test_noalloc_size_check_on_host():
    """The scratch limit is enforced before any CUDA call (fake pointers,
    never dereferenced): 24 items of m = 8, k = 12288 need about 9.4 MB."""
    from packed_bit_gemv_tern_b300 import build
    build.build()
    lib = tern.load()
    w = tern.CMatrix(64, 12288, 0x1000, 0x2000, None)
    arr = (tern.CBatchItem * 24)()
    for i in range(24):
        arr[i].w, arr[i].up, arr[i].x, arr[i].y, arr[i].m = ctypes.addressof(w), None, 0x3000, 0x4000, 8
    assert lib.tern_gemm_batched_noalloc(ctypes.cast(arr, ctypes.c_void_p), 24, None) == tern.TERN_ERR_SHAPE
    assert lib.tern_gemm_batched_noalloc(None, 0, None) == tern.TERN_OK
    assert lib.tern_gemm_batched_noalloc(None, -1, None) == tern.TERN_ERR_SHAPE
    assert lib.tern_gemm_batched_noalloc(None, 2, None) == tern.TERN_ERR_NULL
