"""GPU parity: every device entry point against the fp64 CPU oracle, through
the C ABI, on the same seeded inputs.

Bar: decode is bit-exact; outputs satisfy |y - y_ref| <= max(1e-3 |y_ref|, 1e-4)
element by element; integer-valued activations give bit-exact results.
"""
import numpy as np
import pytest

import oracle
import packed_bit_gemv_tern_b300 as tern
from packed_bit_gemv_tern_b300 import synth, workloads

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


def _mat(t, scale):
    codes, rowsum = tern.tern_pack(t)
    return tern.TernMatrix.from_host(codes, scale, t.shape[1], rowsum), codes


def _guarded_out(m, rows):
    """Output with a sentinel guard band after it; returns (full, view)."""
    full = torch.full((m * rows + 64,), 12345.0, dtype=torch.float32, device="cuda")
    return full, full[: m * rows].view(m, rows)


def _guard_ok(full, m, rows):
    tail = full[m * rows:].cpu().numpy()
    assert np.all(tail == 12345.0), "kernel wrote past the end of its output"


SHAPES = [(1, 64), (3, 128), (33, 192), (64, 4096), (100, 1024), (257, 320), (1024, 4096)]


@pytest.mark.parametrize("rows,k", SHAPES + [(5, 12288)])
def test_unpack_bit_exact(rows, k):
    rng = np.random.default_rng(rows * 31 + k)
    t = synth.ternary(rng, rows, k)
    w, codes = _mat(t, synth.scales(rng, rows))
    out = torch.zeros((rows, k), dtype=torch.int8, device="cuda")
    tern.tern_unpack(w, out)
    got = out.cpu().numpy()
    assert np.array_equal(got, oracle.unpack(codes, k))
    assert np.array_equal(got, t)


@pytest.mark.parametrize("rows,k", SHAPES + [(4096, 12288), (12288, 4096)])
def test_gemv_matches_oracle(rows, k):
    rng = np.random.default_rng(rows + 7 * k)
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    w, codes = _mat(t, scale)
    xb = synth.activations(rng, 1, k)
    full, y = _guarded_out(1, rows)
    tern.tern_gemv(w, _dev_x(xb), y)
    torch.cuda.synchronize()
    ref = oracle.gemm(codes, scale, k, xb, threads=THREADS)
    _close(y.cpu().numpy(), ref, f"gemv {rows}x{k}")
    _guard_ok(full, 1, rows)
    assert tern.tern_last_device_error() == tern.TERN_OK


@pytest.mark.parametrize("rows,k", [(33, 192), (4096, 4096), (1000, 12288)])
def test_gemv_exact_integer_activations(rows, k):
    """x in {-2..2}: every fp32 partial sum is an exact integer, so the GPU must
    equal fl32(scale * exact sum) bit for bit."""
    rng = np.random.default_rng(99 + rows)
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    w, codes = _mat(t, scale)
    xb = synth.small_int_activations(rng, 1, k)
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    tern.tern_gemv(w, _dev_x(xb), y)
    ref = oracle.gemm(codes, scale, k, xb, threads=THREADS)
    assert np.array_equal(y.cpu().numpy(), ref.astype(np.float32))


def test_gemv_closed_forms():
    rows, k = 300, 4096
    rng = np.random.default_rng(5)
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    w, codes = _mat(t, scale)
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    ones = np.full((1, k), 0x3F80, np.uint16)
    tern.tern_gemv(w, _dev_x(ones), y)
    rowsum = t.astype(np.int64).sum(1)
    assert np.array_equal(y.cpu().numpy()[0], (scale.astype(np.float64) * rowsum).astype(np.float32))
    tern.tern_gemv(w, _dev_x(np.zeros((1, k), np.uint16)), y)
    assert not y.cpu().numpy().any()
    for kk in (0, 15, 16, 63, 64, 4095):
        e = np.zeros((1, k), np.uint16)
        e[0, kk] = 0x3F80
        tern.tern_gemv(w, _dev_x(e), y)
        assert np.array_equal(y.cpu().numpy()[0], scale * t[:, kk].astype(np.float32))


@pytest.mark.parametrize("rows,k", [(1, 64), (33, 192), (512, 4096), (12288, 4096)])
def test_swiglu_matches_oracle(rows, k):
    rng = np.random.default_rng(3 * rows + k)
    tg, tu = synth.ternary(rng, rows, k), synth.ternary(rng, rows, k)
    tg[0] = 0
    sg, su = synth.scales(rng, rows), synth.scales(rng, rows)
    wg, cg = _mat(tg, sg)
    wu, cu = _mat(tu, su)
    xb = synth.activations(rng, 1, k)
    full, h = _guarded_out(1, rows)
    tern.tern_gemv_swiglu(wg, wu, _dev_x(xb), h)
    ref = oracle.swiglu(cg, sg, cu, su, k, xb, threads=THREADS)
    got = h.cpu().numpy()
    _close(got, ref, f"swiglu {rows}x{k}")
    assert got[0, 0] == 0.0
    _guard_ok(full, 1, rows)


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("rows,k", [(33, 192), (1024, 4096), (300, 12288)])
def test_smallm_matches_oracle(m, rows, k):
    rng = np.random.default_rng(m * 1000 + rows + k)
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    w, codes = _mat(t, scale)
    xb = synth.activations(rng, m, k)
    full, y = _guarded_out(m, rows)
    tern.tern_gemm_smallm(w, _dev_x(xb), m, y)
    ref = oracle.gemm(codes, scale, k, xb, threads=THREADS)
    _close(y.cpu().numpy(), ref, f"smallm m={m} {rows}x{k}")
    _guard_ok(full, m, rows)


@pytest.mark.parametrize("m", [1, 4, 7, 8])
def test_smallm_swiglu_matches_oracle(m):
    rows, k = 640, 4096
    rng = np.random.default_rng(77 + m)
    tg, tu = synth.ternary(rng, rows, k), synth.ternary(rng, rows, k)
    sg, su = synth.scales(rng, rows), synth.scales(rng, rows)
    wg, cg = _mat(tg, sg)
    wu, cu = _mat(tu, su)
    xb = synth.activations(rng, m, k)
    full, h = _guarded_out(m, rows)
    tern.tern_gemm_smallm_swiglu(wg, wu, _dev_x(xb), m, h)
    ref = oracle.swiglu(cg, sg, cu, su, k, xb, threads=THREADS)
    _close(h.cpu().numpy(), ref, f"smallm_swiglu m={m}")
    _guard_ok(full, m, rows)


def test_smallm_exact_integer():
    rows, k, m = 777, 12288, 7
    rng = np.random.default_rng(8)
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    w, codes = _mat(t, scale)
    xb = synth.small_int_activations(rng, m, k)
    y = torch.empty((m, rows), dtype=torch.float32, device="cuda")
    tern.tern_gemm_smallm(w, _dev_x(xb), m, y)
    ref = oracle.gemm(codes, scale, k, xb, threads=THREADS)
    assert np.array_equal(y.cpu().numpy(), ref.astype(np.float32))


def test_k_zero_gives_zero_and_empty_rows():
    rows = 10
    scale = torch.rand(rows, device="cuda")
    codes = torch.zeros((rows, 0), dtype=torch.int32, device="cuda")
    w = tern.TernMatrix(codes, scale, 0)
    y = torch.full((1, rows), 7.0, device="cuda")
    x = torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda")
    tern.tern_gemv(w, x, y)
    assert not y.cpu().numpy().any()
    empty = tern.TernMatrix(torch.zeros((0, 4), dtype=torch.int32, device="cuda"),
                            torch.zeros(0, device="cuda"), 64)
    tern.tern_gemv(empty, x, torch.zeros(0, device="cuda"))


def test_invalid_code_does_not_fault():
    rows, k = 64, 256
    codes = np.full((rows, k // 16), 0xAAAAAAAA, np.uint32)  # every field is 10
    w = tern.TernMatrix.from_host(codes, np.ones(rows, np.float32), k)
    y = torch.empty((1, rows), device="cuda")
    x = _dev_x(synth.activations(np.random.default_rng(1), 1, k))
    tern.tern_gemv(w, x, y)
    out = torch.empty((rows, k), dtype=torch.int8, device="cuda")
    tern.tern_unpack(w, out)
    assert tern.tern_last_device_error() == tern.TERN_OK
    assert (out.cpu().numpy() == -2).all()


def test_side_stream_and_reuse():
    rows, k = 2048, 4096
    rng = np.random.default_rng(21)
    t = synth.ternary(rng, rows, k)
    scale = synth.scales(rng, rows)
    w, codes = _mat(t, scale)
    xb = synth.activations(rng, 1, k)
    s = torch.cuda.Stream()
    y = torch.empty((1, rows), device="cuda")
    x = _dev_x(xb)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(3):
            tern.tern_gemv(w, x, y, stream=s)
    s.synchronize()
    _close(y.cpu().numpy(), oracle.gemm(codes, scale, k, xb, threads=THREADS), "side stream")


def _run_step(wl, api):
    """One step of a workload: through tern_gemm_batched as bench.py times it by
    default (one persistent launch per group, after an activation-preparing
    launch), or one tern_* call per linear."""
    if api == "batched":
        workloads.run_batched(workloads.batch_of(wl.calls))
    else:
        workloads.run_calls(wl.calls)
    torch.cuda.synchronize()
    assert tern.tern_last_device_error() == tern.TERN_OK


@pytest.mark.parametrize("api", ["batched", "calls"])
@pytest.mark.parametrize("name", ["c0", "c1", "c2", "c3"])
def test_bench_workloads_full_size(name, api):
    """The benchmark's own workloads at full size, in both launch
    configurations bench.py can time; every distinct matrix checked against
    the oracle element by element."""
    wl = workloads.build(name, rotate_bytes=1, distinct=1)
    _run_step(wl, api)
    for c, h in zip(wl.calls, wl.host):
        lin = h["lin"]
        codes = oracle.pack(lin.t)
        if c.up is not None:
            up = h["up"]
            ref = oracle.swiglu(codes, lin.scale, oracle.pack(up.t), up.scale, lin.k, h["x_bits"],
                                threads=THREADS)
        else:
            ref = oracle.gemm(codes, lin.scale, lin.k, h["x_bits"], threads=THREADS)
        _close(c.y.cpu().numpy(), ref, f"{name}:{c.name}")


@pytest.mark.parametrize("api", ["batched", "calls"])
def test_sweep_sampled_rows(api):
    """Two layers of the 36-layer sweep (all seven shapes, the layer-1 code
    mix), sampled rows of every linear against the oracle."""
    wl = workloads.build("c4", layers=2)
    _run_step(wl, api)
    rng = np.random.default_rng(0)
    for c, h in zip(wl.calls, wl.host):
        lin = h["lin"]
        rows = np.sort(rng.choice(lin.rows, size=64, replace=False))
        codes = oracle.pack(lin.t)
        ref = oracle.gemm(codes, lin.scale, lin.k, h["x_bits"], threads=THREADS, rows_subset=rows)
        _close(c.y.cpu().numpy()[:, rows], ref[:, rows], c.name)


def _item(rng, rows, k, m, swiglu=False, p_zero=synth.P_ZERO, int_x=False):
    """One batched item with its oracle reference (float64)."""
    t = synth.ternary(rng, rows, k, p_zero)
    sc = synth.scales(rng, rows)
    w, codes = _mat(t, sc)
    up = upc = su = None
    if swiglu:
        tu = synth.ternary(rng, rows, k, p_zero)
        su = synth.scales(rng, rows)
        up, upc = _mat(tu, su)
    xb = synth.small_int_activations(rng, m, k) if int_x else synth.activations(rng, m, k)
    full, y = _guarded_out(m, rows)
    if swiglu:
        ref = oracle.swiglu(codes, sc, upc, su, k, xb, threads=THREADS)
    else:
        ref = oracle.gemm(codes, sc, k, xb, threads=THREADS)
    return (w, up, _dev_x(xb), y, m), ref, full


def test_batched_mixed_items():
    """One batched call over plain GEMVs, SwiGLU pairs and small-M products of
    several shapes (ragged rows, K spanning several 4096-code chunks, short
    rows), each element checked against the oracle."""
    rng = np.random.default_rng(404)
    specs = [(4096, 4096, 1, False), (1024, 4096, 1, False), (257, 320, 1, False), (640, 4096, 1, True),
             (300, 12288, 3, False), (4096, 12288, 7, False), (130, 4096, 7, True), (1, 64, 1, False),
             (33, 192, 8, True), (12288, 4096, 1, True), (200, 8256, 2, False)]
    made = [_item(rng, r, k, m, sw) for (r, k, m, sw) in specs]
    tern.tern_gemm_batched([mi[0] for mi in made])
    torch.cuda.synchronize()
    assert tern.tern_last_device_error() == tern.TERN_OK
    for (spec, (it, ref, full)) in zip(specs, made):
        rows, k, m, sw = spec
        _close(it[3].cpu().numpy(), ref, f"batched {spec}")
        _guard_ok(full, m, rows)


def test_batched_one_stage_chunks_in_one_cta():
    """A CTA whose run is three one-stage tiles of one item (257 x 320) ahead
    of a SwiGLU pair: the issuers of a later tile reach their waits while the
    staging warps still build the first tile's operand, so every buffer wait
    must be for the right phase (a parity wait issued a phase early returns
    at once).  Run three times; every element against the oracle."""
    rng = np.random.default_rng(409)
    for _ in range(3):
        made = [_item(rng, 257, 320, 1), _item(rng, 640, 4096, 1, swiglu=True)]
        tern.tern_gemm_batched([mi[0] for mi in made])
        torch.cuda.synchronize()
        assert tern.tern_last_device_error() == tern.TERN_OK
        for it, ref, full in made:
            _close(it[3].cpu().numpy(), ref, "one-stage chunks")


def test_batched_exact_integers_and_many_items():
    """More items than one launch carries (split over several launches),
    integer activations: every result bit-exact."""
    rng = np.random.default_rng(405)
    made = [_item(rng, 128 + 64 * (i % 5), 4096 if i % 3 else 12288, 1 + (i % 8), swiglu=(i % 4 == 0), int_x=True)
            for i in range(150)]
    # two persistent launches, each after an activation-preparing launch
    assert tern.tern_gemm_batched_launches([mi[0] for mi in made]) == 4
    tern.tern_gemm_batched([mi[0] for mi in made])
    torch.cuda.synchronize()
    for i, (it, ref, full) in enumerate(made):
        if it[1] is None:
            assert np.array_equal(it[3].cpu().numpy(), ref.astype(np.float32)), i
        else:
            _close(it[3].cpu().numpy(), ref, f"swiglu item {i}")


def test_batched_empty_and_degenerate():
    rng = np.random.default_rng(406)
    it, ref, full = _item(rng, 100, 256, 2)
    kzero = tern.TernMatrix(torch.zeros((5, 0), dtype=torch.int32, device="cuda"), torch.ones(5, device="cuda"), 0)
    y0 = torch.full((1, 5), 3.0, device="cuda")
    empty = tern.TernMatrix(torch.zeros((0, 4), dtype=torch.int32, device="cuda"), torch.zeros(0, device="cuda"), 64)
    tern.tern_gemm_batched([])
    tern.tern_gemm_batched([it, (kzero, None, torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda"), y0, 1),
                            (empty, None, None, None, 1)])
    torch.cuda.synchronize()
    _close(it[3].cpu().numpy(), ref, "batched small")
    assert not y0.cpu().numpy().any()
    with pytest.raises(tern.TernError) as e:
        tern.tern_gemm_batched([(it[0], None, it[2], it[3], 9)])
    assert e.value.status == tern.TERN_ERR_M_RANGE
