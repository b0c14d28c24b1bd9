"""Host-side tests of the C ABI (no GPU needed): the library loads, exports
every symbol include/tern.h declares, packs and validates exactly like the
oracle's independent encoder, and rejects bad arguments before launching
anything."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import packed_bit_gemv_tern_b300 as tern
from packed_bit_gemv_tern_b300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^TERN_API[^(]*?\b(tern\d*_\w+)\s*\(", src, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    from packed_bit_gemv_tern_b300 import build
    build.build()
    return tern.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(tern.ABI_FUNCTIONS) <= set(names)
    assert tern.tern_abi_version() == 2


def test_header_constants_match_binding():
    """Every TERN_* integer constant of include/tern.h has the same value in
    the Python binding."""
    src = open(os.path.join(ROOT, "include", "tern.h")).read()
    defs = dict(re.findall(r"^#define\s+(TERN_\w+)\s+(\d+)\s*$", src, flags=re.M))
    enums = dict(re.findall(r"\b(TERN_\w+)\s*=\s*(\d+)", src))
    both = {**defs, **enums}
    assert "TERN_NOALLOC_WS_BYTES" in both and "TERN_MAX_X_BYTES" in both
    for name, val in both.items():
        if hasattr(tern, name):
            assert getattr(tern, name) == int(val), name
    for name in ("TERN_NOALLOC_WS_BYTES", "TERN_MAX_X_BYTES", "TERN_MAX_M", "TERN_ERR_TIMEOUT"):
        assert hasattr(tern, name), name


def test_status_strings(lib):
    for s in range(10):
        assert tern.tern_status_str(s)
    assert "unknown" in tern.tern_status_str(99)


@pytest.mark.parametrize("rows,k,seed", [(1, 64, 0), (7, 128, 1), (33, 4096, 2), (5, 12288, 3), (0, 64, 4), (3, 0, 5)])
def test_pack_matches_oracle_encoder(lib, rows, k, seed):
    rng = np.random.default_rng(seed)
    t = synth.ternary(rng, rows, k)
    codes, rowsum = tern.tern_pack(t)
    if rows and k:
        assert np.array_equal(codes, oracle.pack(t))
    orc_rowsum, orc_counts = oracle.stats(codes, k) if rows else (np.zeros(0), np.zeros(3))
    assert np.array_equal(rowsum, orc_rowsum.astype(np.int32))
    counts = tern.tern_validate(codes, k, rowsum)
    assert counts.tolist() == [int((t == 0).sum()), int((t == 1).sum()), int((t == -1).sum())]
    if rows:
        assert counts.tolist() == orc_counts.tolist()


def test_pack_rejects(lib):
    with pytest.raises(tern.TernError) as e:
        tern.tern_pack(np.zeros((2, 48), np.int8))
    assert e.value.status == tern.TERN_ERR_SHAPE
    bad = np.zeros((2, 64), np.int8)
    bad[1, 5] = -2
    with pytest.raises(tern.TernError) as e:
        tern.tern_pack(bad)
    assert e.value.status == tern.TERN_ERR_VALUE


def test_validate_rejects(lib):
    rng = np.random.default_rng(9)
    t = synth.ternary(rng, 4, 128)
    codes, rowsum = tern.tern_pack(t)
    bad = codes.copy()
    bad[2, 3] |= np.uint32(0x2 << 10)
    bad[2, 3] &= ~np.uint32(0x1 << 10)
    with pytest.raises(tern.TernError) as e:
        tern.tern_validate(bad, 128)
    assert e.value.status == tern.TERN_ERR_BADCODE
    rs = rowsum.copy()
    rs[1] += 1
    with pytest.raises(tern.TernError) as e:
        tern.tern_validate(codes, 128, rs)
    assert e.value.status == tern.TERN_ERR_ROWSUM


def _mat(rows, k, codes=0x1000, scale=0x2000):
    return tern.CMatrix(rows, k, codes, scale, None)


def _call(lib, name, *args):
    return getattr(lib, name)(*args)


def test_device_entry_points_reject_before_launch(lib):
    """Every case fails a host check, so nothing reaches the GPU (or the
    missing GPU).  Pointers are fake but never dereferenced."""
    ok_m = _mat(4, 64)
    x, y = ctypes.c_void_p(0x3000), ctypes.c_void_p(0x4000)
    ref = ctypes.byref
    assert lib.tern_gemv(None, x, y, None) == tern.TERN_ERR_NULL
    assert lib.tern_gemv(ref(_mat(4, 48)), x, y, None) == tern.TERN_ERR_SHAPE
    assert lib.tern_gemv(ref(_mat(-1, 64)), x, y, None) == tern.TERN_ERR_SHAPE
    assert lib.tern_gemv(ref(_mat(4, 64, codes=0x1004)), x, y, None) == tern.TERN_ERR_ALIGN
    assert lib.tern_gemv(ref(_mat(4, 64, scale=0x2002)), x, y, None) == tern.TERN_ERR_ALIGN
    assert lib.tern_gemv(ref(_mat(4, 64, codes=0)), x, y, None) == tern.TERN_ERR_NULL
    assert lib.tern_gemv(ref(ok_m), None, y, None) == tern.TERN_ERR_NULL
    assert lib.tern_gemv(ref(ok_m), x, None, None) == tern.TERN_ERR_NULL
    assert lib.tern_gemv(ref(ok_m), ctypes.c_void_p(0x3008), y, None) == tern.TERN_ERR_ALIGN
    assert lib.tern_gemv(ref(ok_m), x, ctypes.c_void_p(0x4002), None) == tern.TERN_ERR_ALIGN
    big = _mat(4, 98368)  # 2*k > TERN_MAX_X_BYTES
    assert lib.tern_gemv(ref(big), x, y, None) == tern.TERN_ERR_SHAPE
    # small-M range and limits
    for m in (0, 9, -1):
        assert lib.tern_gemm_smallm(ref(ok_m), x, m, y, None) == tern.TERN_ERR_M_RANGE
    assert lib.tern_gemm_smallm(ref(_mat(4, 12352)), x, 8, y, None) == tern.TERN_ERR_SHAPE
    # SwiGLU pair mismatch / missing up
    assert lib.tern_gemv_swiglu(ref(ok_m), None, x, y, None) == tern.TERN_ERR_NULL
    assert lib.tern_gemv_swiglu(ref(ok_m), ref(_mat(5, 64)), x, y, None) == tern.TERN_ERR_SHAPE
    assert lib.tern_gemv_swiglu(ref(ok_m), ref(_mat(4, 128)), x, y, None) == tern.TERN_ERR_SHAPE
    assert lib.tern_gemm_smallm_swiglu(ref(ok_m), ref(ok_m), x, 9, y, None) == tern.TERN_ERR_M_RANGE
    # unpack
    assert lib.tern_unpack(ref(ok_m), None, None) == tern.TERN_ERR_NULL
    assert lib.tern_unpack(ref(ok_m), ctypes.c_void_p(0x5001), None) == tern.TERN_ERR_ALIGN
    # batched: bad count / NULL array / a bad item rejects the whole batch
    assert lib.tern_gemm_batched(None, -1, None) == tern.TERN_ERR_SHAPE
    assert lib.tern_gemm_batched(None, 0, None) == tern.TERN_OK
    assert lib.tern_gemm_batched(None, 2, None) == tern.TERN_ERR_NULL
    good = _mat(4, 64)
    arr = (tern.CBatchItem * 2)()
    arr[0].w, arr[0].up, arr[0].x, arr[0].y, arr[0].m = ctypes.addressof(good), None, 0x3000, 0x4000, 1
    bad = _mat(4, 48)
    arr[1].w, arr[1].up, arr[1].x, arr[1].y, arr[1].m = ctypes.addressof(bad), None, 0x3000, 0x4000, 1
    assert lib.tern_gemm_batched(ctypes.cast(arr, ctypes.c_void_p), 2, None) == tern.TERN_ERR_SHAPE
    arr[1].w, arr[1].m = ctypes.addressof(good), 0
    assert lib.tern_gemm_batched(ctypes.cast(arr, ctypes.c_void_p), 2, None) == tern.TERN_ERR_M_RANGE
    arr[1].m, arr[1].up = 1, ctypes.addressof(_mat(5, 64))
    assert lib.tern_gemm_batched(ctypes.cast(arr, ctypes.c_void_p), 2, None) == tern.TERN_ERR_SHAPE
    arr[1].up, arr[1].x = None, 0x3004
    assert lib.tern_gemm_batched(ctypes.cast(arr, ctypes.c_void_p), 2, None) == tern.TERN_ERR_ALIGN
    # batched with an RMSNorm: the item checks first, then the norm arguments
    arr[1].x = 0x3000
    pa = ctypes.cast(arr, ctypes.c_void_p)
    norms = (ctypes.c_void_p * 2)(0x6000, None)
    pn = ctypes.cast(norms, ctypes.c_void_p)
    f = lib.tern_gemm_batched_rmsnorm
    assert f(None, None, ctypes.c_float(1e-6), 0, None) == tern.TERN_OK
    assert f(None, pn, ctypes.c_float(1e-6), -1, None) == tern.TERN_ERR_SHAPE
    assert f(pa, None, ctypes.c_float(1e-6), 2, None) == tern.TERN_ERR_NULL
    for eps in (-1e-6, float("nan"), float("inf")):
        assert f(pa, pn, ctypes.c_float(eps), 2, None) == tern.TERN_ERR_VALUE
    norms[1] = 0x6004
    assert f(pa, pn, ctypes.c_float(1e-6), 2, None) == tern.TERN_ERR_ALIGN
    arr[1].m = 9  # a bad item is reported before the norm arguments
    assert f(pa, None, ctypes.c_float(-1.0), 2, None) == tern.TERN_ERR_M_RANGE
    arr[1].m = 1
    # base-3 format: shape, pointers and alignment before a launch
    c5 = tern.C5Matrix(4, 160, 0x7000, 0x7100)
    assert lib.tern5_gemm(None, x, 1, y, None) == tern.TERN_ERR_NULL
    assert lib.tern5_gemm(ref(tern.C5Matrix(4, 150, 0x7000, 0x7100)), x, 1, y, None) == tern.TERN_ERR_SHAPE
    assert lib.tern5_gemm(ref(c5), x, 0, y, None) == tern.TERN_ERR_M_RANGE
    assert lib.tern5_gemm(ref(c5), x, 9, y, None) == tern.TERN_ERR_M_RANGE
    assert lib.tern5_gemm(ref(tern.C5Matrix(4, 160, 0x7008, 0x7100)), x, 1, y, None) == tern.TERN_ERR_ALIGN
    assert lib.tern5_gemm(ref(c5), ctypes.c_void_p(0x3008), 1, y, None) == tern.TERN_ERR_ALIGN
    assert lib.tern5_gemm(ref(c5), x, 1, None, None) == tern.TERN_ERR_NULL
    assert lib.tern5_gemm(ref(tern.C5Matrix(4, 24640, 0x7000, 0x7100)), x, 4, y, None) == tern.TERN_ERR_SHAPE
    assert lib.tern5_unpack(ref(c5), None, None) == tern.TERN_ERR_NULL
    assert lib.tern5_gemm(ref(tern.C5Matrix(0, 160, None, None)), None, 1, None, None) == tern.TERN_OK
    # int8 head: every argument is checked before a launch
    h = tern.CI8Matrix(10, 128, 0x7000, 0x7100)
    lg, am = ctypes.c_void_p(0x8000), ctypes.c_void_p(0x9000)
    f = lib.tern_lmhead_argmax
    e6 = ctypes.c_float(1e-6)
    assert f(None, x, 1, None, e6, lg, am, None) == tern.TERN_ERR_NULL
    assert f(ref(h), None, 1, None, e6, lg, am, None) == tern.TERN_ERR_NULL
    assert f(ref(h), x, 1, None, e6, lg, None, None) == tern.TERN_ERR_NULL
    assert f(ref(tern.CI8Matrix(0, 128, 0x7000, 0x7100)), x, 1, None, e6, lg, am, None) == tern.TERN_ERR_SHAPE
    assert f(ref(tern.CI8Matrix(10, 96, 0x7000, 0x7100)), x, 1, None, e6, lg, am, None) == tern.TERN_ERR_SHAPE
    assert f(ref(tern.CI8Matrix(10, 24576, 0x7000, 0x7100)), x, 8, None, e6, lg, am, None) == tern.TERN_ERR_SHAPE
    for m in (0, 9):
        assert f(ref(h), x, m, None, e6, lg, am, None) == tern.TERN_ERR_M_RANGE
    assert f(ref(tern.CI8Matrix(10, 128, 0x7008, 0x7100)), x, 1, None, e6, lg, am, None) == tern.TERN_ERR_ALIGN
    assert f(ref(h), ctypes.c_void_p(0x3008), 1, None, e6, lg, am, None) == tern.TERN_ERR_ALIGN
    assert f(ref(h), x, 1, ctypes.c_void_p(0x6004), e6, lg, am, None) == tern.TERN_ERR_ALIGN
    assert f(ref(h), x, 1, None, e6, lg, ctypes.c_void_p(0x9002), None) == tern.TERN_ERR_ALIGN
    assert f(ref(h), x, 1, None, ctypes.c_float(-1.0), lg, am, None) == tern.TERN_ERR_VALUE
    # empty problems succeed without a launch, with NULL pointers
    empty = tern.CMatrix(0, 64, None, None, None)
    assert lib.tern_gemv(ref(empty), None, None, None) == tern.TERN_OK
    assert lib.tern_gemm_smallm(ref(empty), None, 3, None, None) == tern.TERN_OK
    assert lib.tern_gemv_swiglu(ref(empty), ref(empty), None, None, None) == tern.TERN_OK
    assert lib.tern_unpack(ref(empty), None, None) == tern.TERN_OK


def test_batched_launch_plan(lib):
    """Launch count of tern_gemm_batched: 128 items or 144 weight matrices per
    launch, k == 0 items on a launch of their own, rows == 0 items on none, and
    one activation-preparing launch per group that holds an item with m >= 2."""
    keep = []

    def arr(spec):
        a = (tern.CBatchItem * len(spec))()
        for i, sp in enumerate(spec):
            rows, k, sw = sp[:3]
            w = _mat(rows, k)
            keep.append(w)
            a[i].w = ctypes.addressof(w)
            if sw:
                u = _mat(rows, k)
                keep.append(u)
                a[i].up = ctypes.addressof(u)
            a[i].x, a[i].y, a[i].m = 0x3000, 0x4000, sp[3] if len(sp) > 3 else 1
        return a

    cases = [([(4096, 4096, 0)] * 128, 1), ([(4096, 4096, 0)] * 129, 2), ([(64, 4096, 1)] * 72, 1),
             ([(64, 4096, 1)] * 73, 2), ([(0, 64, 0)] * 5, 0), ([(4, 0, 0)] * 3, 3),
             ([(4, 0, 0), (4096, 4096, 0), (0, 4, 0)], 2), ([(4096, 4096, 0)] * 252, 2),
             ([(4096, 4096, 0)] * 257, 3), ([(4096, 4096, 0)] * 100 + [(64, 4096, 1)] * 30, 2),
             ([(4096, 4096, 0, 7)], 2), ([(12288, 4096, 1, 7), (4096, 12288, 0, 7)] * 4, 2),
             ([(4096, 4096, 0, 2)] + [(4096, 4096, 0)] * 200, 3), ([(4, 0, 0, 7), (0, 64, 0, 3)], 1)]
    for spec, want in cases:
        assert tern.tern_gemm_batched_launches(arr(spec)) == want, (len(spec), want)
    assert lib.tern_gemm_batched_launches(None, 0) == 0
    assert lib.tern_gemm_batched_launches(None, 3) == -tern.TERN_ERR_NULL
    assert lib.tern_gemm_batched_launches(None, -1) == -tern.TERN_ERR_SHAPE


@pytest.mark.parametrize("rows,k,seed", [(1, 80, 0), (7, 400, 1), (33, 4160, 2)])
def test_base3_pack_matches_oracle_encoder(lib, rows, k, seed):
    rng = np.random.default_rng(seed)
    t = synth.ternary(rng, rows, k)
    codes, rowsum = tern.tern5_pack(t)
    assert np.array_equal(codes, oracle.pack5(t))
    assert np.array_equal(rowsum, t.astype(np.int64).sum(axis=1))


def test_base3_pack_rejects(lib):
    with pytest.raises(tern.TernError) as e:
        tern.tern5_pack(np.zeros((2, 64), dtype=np.int8))
    assert e.value.status == tern.TERN_ERR_SHAPE
    bad = np.zeros((1, 80), dtype=np.int8)
    bad[0, 17] = 2
    with pytest.raises(tern.TernError) as e:
        tern.tern5_pack(bad)
    assert e.value.status == tern.TERN_ERR_VALUE
