"""Python binding of the ternary packed-weight linear-layer library (``libtern.so``).

Argument marshalling only: every device step runs in the CUDA kernels behind
the C ABI declared in ``include/tern.h``.  PyTorch supplies device memory and
streams.  The library is loaded on first use; if it is missing (not built)
every call raises -- there is no CPU fallback.

Names follow the C ABI: ``tern_pack``, ``tern_validate``, ``tern_unpack``,
``tern_gemv``, ``tern_gemv_swiglu``, ``tern_gemm_smallm``,
``tern_gemm_smallm_swiglu``, ``tern_last_device_error``, ``tern_status_str``,
``tern_abi_version``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtern.so")

TERN_OK = 0
TERN_ERR_NULL = 1
TERN_ERR_SHAPE = 2
TERN_ERR_ALIGN = 3
TERN_ERR_BADCODE = 4
TERN_ERR_ROWSUM = 5
TERN_ERR_M_RANGE = 6
TERN_ERR_CUDA = 7
TERN_ERR_TIMEOUT = 8
TERN_ERR_VALUE = 9
TERN_MAX_X_BYTES = 196608
TERN_MAX_M = 8
TERN_NOALLOC_WS_BYTES = 4194304

ABI_FUNCTIONS = (
    "tern_pack", "tern_validate", "tern_unpack", "tern_gemv", "tern_gemv_swiglu",
    "tern_gemm_smallm", "tern_gemm_smallm_swiglu", "tern_gemm_batched", "tern_gemm_batched_launches",
    "tern_gemm_batched_noalloc", "tern_gemm_batched_rmsnorm", "tern_lmhead_argmax",
    "tern5_pack", "tern5_unpack", "tern5_gemm",
    "tern_last_device_error", "tern_set_wait_limit",
    "tern_status_str", "tern_abi_version",
)


class TernError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: status {status} ({_status_text(status)})")


class CMatrix(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("k", ctypes.c_int32), ("codes", ctypes.c_void_p),
                ("scale", ctypes.c_void_p), ("rowsum", ctypes.c_void_p)]


class CI8Matrix(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("k", ctypes.c_int32), ("w", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class C5Matrix(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("k", ctypes.c_int32), ("codes", ctypes.c_void_p),
                ("scale", ctypes.c_void_p)]


class CBatchItem(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("up", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("m", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Load ``libtern.so`` (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"libtern.so not found at {p}; build it with "
                              "`python -m packed_bit_gemv_tern_b300.build`")
        lib = ctypes.CDLL(p)
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        sig = {
            "tern_pack": [vp, i32, i32, vp, vp],
            "tern_validate": [vp, i32, i32, vp, vp],
            "tern_unpack": [vp, vp, vp],
            "tern_gemv": [vp, vp, vp, vp],
            "tern_gemv_swiglu": [vp, vp, vp, vp, vp],
            "tern_gemm_smallm": [vp, vp, i32, vp, vp],
            "tern_gemm_smallm_swiglu": [vp, vp, vp, i32, vp, vp],
            "tern_gemm_batched": [vp, i32, vp],
            "tern_gemm_batched_launches": [vp, i32],
            "tern_gemm_batched_noalloc": [vp, i32, vp],
            "tern_gemm_batched_rmsnorm": [vp, vp, ctypes.c_float, i32, vp],
            "tern_lmhead_argmax": [vp, vp, i32, vp, ctypes.c_float, vp, vp, vp],
            "tern5_pack": [vp, i32, i32, vp, vp],
            "tern5_unpack": [vp, vp, vp],
            "tern5_gemm": [vp, vp, i32, vp, vp],
            "tern_last_device_error": [vp],
            "tern_set_wait_limit": [ctypes.c_int64],
            "tern_status_str": [ctypes.c_int],
            "tern_abi_version": [],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        lib.tern_status_str.restype = ctypes.c_char_p
        lib.tern_set_wait_limit.restype = None
        lib.tern_abi_version.restype = ctypes.c_int32
        _lib = lib
        return lib


def _status_text(status: int) -> str:
    try:
        return load().tern_status_str(int(status)).decode()
    except Exception:  # pragma: no cover - library missing
        return "?"


def _check(status: int, what: str):
    if status != TERN_OK:
        raise TernError(status, what)


def _np_ptr(a):
    return None if a is None else a.ctypes.data


# ---------------------------------------------------------------------------
# Host packer / validator
# ---------------------------------------------------------------------------

def tern_pack(t: np.ndarray):
    """int8 [rows, k] -> (codes uint32 [rows, k//16], rowsum int32 [rows])."""
    t = np.ascontiguousarray(t, dtype=np.int8)
    rows, k = t.shape
    codes = np.zeros((rows, max(k // 16, 0)), dtype=np.uint32)
    rowsum = np.zeros(rows, dtype=np.int32)
    _check(load().tern_pack(_np_ptr(t), rows, k, _np_ptr(codes), _np_ptr(rowsum)), "tern_pack")
    return codes, rowsum


def tern_validate(codes: np.ndarray, k: int, rowsum: np.ndarray | None = None):
    """Returns counts int64 [3] = (zeros, plus, minus); raises TernError on a bad code / rowsum."""
    codes = np.ascontiguousarray(codes, dtype=np.uint32)
    rows = codes.shape[0]
    counts = np.zeros(3, dtype=np.int64)
    rs = None if rowsum is None else np.ascontiguousarray(rowsum, dtype=np.int32)
    _check(load().tern_validate(_np_ptr(codes), rows, k, _np_ptr(rs), _np_ptr(counts)), "tern_validate")
    return counts


# ---------------------------------------------------------------------------
# Device side
# ---------------------------------------------------------------------------

class TernMatrix:
    """A packed ternary matrix resident on the GPU (torch tensors own the memory)."""

    def __init__(self, codes, scale, k: int, rowsum=None):
        self.codes = codes    # torch.int32 view of the uint32 words, [rows, k//16]
        self.scale = scale    # torch.float32 [rows]
        self.rowsum = rowsum  # torch.int32 [rows] or None
        self.rows = int(scale.shape[0])
        self.k = int(k)
        self._c = CMatrix(self.rows, self.k, codes.data_ptr() if codes.numel() else None,
                          scale.data_ptr() if scale.numel() else None,
                          rowsum.data_ptr() if rowsum is not None and rowsum.numel() else None)

    @classmethod
    def from_host(cls, codes: np.ndarray, scale: np.ndarray, k: int, rowsum: np.ndarray | None = None,
                  device="cuda"):
        import torch
        c = torch.from_numpy(np.ascontiguousarray(codes, np.uint32).view(np.int32)).to(device)
        s = torch.from_numpy(np.ascontiguousarray(scale, np.float32)).to(device)
        r = None if rowsum is None else torch.from_numpy(np.ascontiguousarray(rowsum, np.int32)).to(device)
        return cls(c, s, k, r)

    @property
    def packed_bytes(self) -> int:
        return self.rows * self.k // 4

    def ref(self):
        return ctypes.byref(self._c)


class I8Matrix:
    """An int8 matrix with per-row fp32 scales resident on the GPU (the
    output head); torch tensors own the memory."""

    def __init__(self, w, scale):
        self.w = w            # torch.int8 [rows, k]
        self.scale = scale    # torch.float32 [rows]
        self.rows, self.k = int(w.shape[0]), int(w.shape[1])
        self._c = CI8Matrix(self.rows, self.k, w.data_ptr() if w.numel() else None,
                            scale.data_ptr() if scale.numel() else None)

    @classmethod
    def from_host(cls, w: np.ndarray, scale: np.ndarray, device="cuda"):
        import torch
        return cls(torch.from_numpy(np.ascontiguousarray(w, np.int8)).to(device),
                   torch.from_numpy(np.ascontiguousarray(scale, np.float32)).to(device))

    @property
    def packed_bytes(self) -> int:
        return self.rows * self.k

    def ref(self):
        return ctypes.byref(self._c)


class Tern5Matrix:
    """A base-3 packed matrix (five weights per byte) resident on the GPU."""

    def __init__(self, codes, scale, k: int):
        self.codes = codes    # torch.uint8 [rows, k//5]
        self.scale = scale    # torch.float32 [rows]
        self.rows, self.k = int(scale.shape[0]), int(k)
        self._c = C5Matrix(self.rows, self.k, codes.data_ptr() if codes.numel() else None,
                           scale.data_ptr() if scale.numel() else None)

    @classmethod
    def from_host(cls, codes: np.ndarray, scale: np.ndarray, k: int, device="cuda"):
        import torch
        return cls(torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).to(device),
                   torch.from_numpy(np.ascontiguousarray(scale, np.float32)).to(device), k)

    @property
    def packed_bytes(self) -> int:
        return self.rows * self.k // 5

    def ref(self):
        return ctypes.byref(self._c)


def tern5_pack(t: np.ndarray):
    """int8 [rows, k] (k % 80 == 0) -> (uint8 codes [rows, k//5], int32 rowsum [rows])."""
    t = np.ascontiguousarray(t, dtype=np.int8)
    rows, k = t.shape
    codes = np.zeros((rows, k // 5), dtype=np.uint8)
    rowsum = np.zeros(rows, dtype=np.int32)
    _check(load().tern5_pack(_np_ptr(t), rows, k, _np_ptr(codes), _np_ptr(rowsum)), "tern5_pack")
    return codes, rowsum


def tern5_unpack(w: "Tern5Matrix", t_out, stream=None):
    _check(load().tern5_unpack(w.ref(), _dptr(t_out), _stream_handle(stream)), "tern5_unpack")


def tern5_gemm(w: "Tern5Matrix", x, m: int, y, stream=None):
    _check(load().tern5_gemm(w.ref(), _dptr(x), int(m), _dptr(y), _stream_handle(stream)), "tern5_gemm")


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dptr(t):
    return None if t is None or t.numel() == 0 else t.data_ptr()


def tern_unpack(w: TernMatrix, t_out, stream=None):
    _check(load().tern_unpack(w.ref(), _dptr(t_out), _stream_handle(stream)), "tern_unpack")


def tern_gemv(w: TernMatrix, x, y, stream=None):
    _check(load().tern_gemv(w.ref(), _dptr(x), _dptr(y), _stream_handle(stream)), "tern_gemv")


def tern_gemv_swiglu(gate: TernMatrix, up: TernMatrix, x, h, stream=None):
    _check(load().tern_gemv_swiglu(gate.ref(), up.ref(), _dptr(x), _dptr(h), _stream_handle(stream)),
           "tern_gemv_swiglu")


def tern_gemm_smallm(w: TernMatrix, x, m: int, y, stream=None):
    _check(load().tern_gemm_smallm(w.ref(), _dptr(x), int(m), _dptr(y), _stream_handle(stream)),
           "tern_gemm_smallm")


def tern_gemm_smallm_swiglu(gate: TernMatrix, up: TernMatrix, x, m: int, h, stream=None):
    _check(load().tern_gemm_smallm_swiglu(gate.ref(), up.ref(), _dptr(x), int(m), _dptr(h),
                                          _stream_handle(stream)), "tern_gemm_smallm_swiglu")


def batch_items(items):
    """ctypes array for tern_gemm_batched from (w, up, x, y, m) tuples; up may be None.

    The returned array references the TernMatrix structs, which must stay alive."""
    arr = (CBatchItem * len(items))()
    for i, (w, up, x, y, m) in enumerate(items):
        arr[i].w = ctypes.addressof(w._c)
        arr[i].up = ctypes.addressof(up._c) if up is not None else None
        arr[i].x = _dptr(x)
        arr[i].y = _dptr(y)
        arr[i].m = int(m)
    return arr


def tern_gemm_batched(items, stream=None):
    """items: sequence of (w, up, x, y, m) tuples, or an array from batch_items()."""
    arr = items if isinstance(items, ctypes.Array) else batch_items(items)
    _check(load().tern_gemm_batched(ctypes.cast(arr, ctypes.c_void_p) if len(arr) else None, len(arr),
                                    _stream_handle(stream)), "tern_gemm_batched")


def tern_gemm_batched_noalloc(items, stream=None):
    """tern_gemm_batched with its scratch in a fixed module-scope array of
    TERN_NOALLOC_WS_BYTES instead of a library-allocated workspace."""
    arr = items if isinstance(items, ctypes.Array) else batch_items(items)
    _check(load().tern_gemm_batched_noalloc(ctypes.cast(arr, ctypes.c_void_p) if len(arr) else None, len(arr),
                                            _stream_handle(stream)), "tern_gemm_batched_noalloc")


def tern_gemm_batched_rmsnorm(items, norm_w, eps: float = 1e-6, stream=None):
    """tern_gemm_batched with an RMSNorm ahead of each item whose entry in
    norm_w (a sequence of device fp32 [k] tensors or None, one per item) is
    not None."""
    arr = items if isinstance(items, ctypes.Array) else batch_items(items)
    if len(norm_w) != len(arr):
        raise ValueError("norm_w needs one entry per item")
    ptrs = (ctypes.c_void_p * max(1, len(arr)))()
    for i, g in enumerate(norm_w):
        ptrs[i] = None if g is None else _dptr(g)
    _check(load().tern_gemm_batched_rmsnorm(ctypes.cast(arr, ctypes.c_void_p) if len(arr) else None,
                                            ctypes.cast(ptrs, ctypes.c_void_p), ctypes.c_float(eps), len(arr),
                                            _stream_handle(stream)), "tern_gemm_batched_rmsnorm")


def tern_lmhead_argmax(w: I8Matrix, x, m: int, logits, argmax, norm_w=None, eps: float = 1e-6, stream=None):
    """Output-head logits [m, rows] and the per-row greedy choice argmax [m]
    (int32 tensor), with an optional RMSNorm of x first."""
    _check(load().tern_lmhead_argmax(w.ref(), _dptr(x), int(m), _dptr(norm_w), ctypes.c_float(eps), _dptr(logits),
                                     _dptr(argmax), _stream_handle(stream)), "tern_lmhead_argmax")


def tern_gemm_batched_launches(items) -> int:
    """Kernel launches tern_gemm_batched makes for these items (host only)."""
    arr = items if isinstance(items, ctypes.Array) else batch_items(items)
    n = int(load().tern_gemm_batched_launches(ctypes.cast(arr, ctypes.c_void_p) if len(arr) else None, len(arr)))
    if n < 0:
        raise TernError(-n, "tern_gemm_batched_launches")
    return n


def tern_last_device_error(stream=None) -> int:
    return int(load().tern_last_device_error(_stream_handle(stream)))


def tern_set_wait_limit(cycles: int = 0):
    """Bound of the kernels' device-side waits for later launches, in SM
    cycles (0 restores the default); a diagnostic for the time-out path."""
    load().tern_set_wait_limit(int(cycles))


def tern_status_str(status: int) -> str:
    return load().tern_status_str(int(status)).decode()


def tern_abi_version() -> int:
    return int(load().tern_abi_version())
