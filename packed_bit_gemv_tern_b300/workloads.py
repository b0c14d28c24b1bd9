"""Device-resident workloads for the benchmark and the tests.

Weights are drawn with :mod:`synth` (seeded), packed on the host with the
library's own ``tern_pack`` and copied to the GPU once.  Each workload is a
list of calls that make up one step; ``run_calls`` issues them on a stream.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import (TernMatrix, batch_items, synth, tern_gemm_batched, tern_gemm_smallm, tern_gemm_smallm_swiglu, tern_gemv,
               tern_gemv_swiglu, tern_pack)

MiB = 1 << 20


@dataclasses.dataclass
class Call:
    kind: str                 # gemv | swiglu | smallm | smallm_swiglu
    w: TernMatrix
    x: object                 # torch bf16 tensor [m, k]
    y: object                 # torch fp32 tensor [m, rows]
    m: int = 1
    up: TernMatrix | None = None
    name: str = ""

    @property
    def packed_bytes(self) -> int:
        return self.w.packed_bytes + (self.up.packed_bytes if self.up is not None else 0)

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes a perfect kernel moves: packed codes + scales + x + y."""
        mats = [self.w] + ([self.up] if self.up is not None else [])
        b = sum(w.packed_bytes + 4 * w.rows for w in mats)
        return b + 2 * self.m * self.w.k + 4 * self.m * self.w.rows


def device_matrix(lin: synth.Linear, device="cuda") -> TernMatrix:
    codes, rowsum = tern_pack(lin.t)
    return TernMatrix.from_host(codes, lin.scale, lin.k, rowsum, device=device)


def run_call(c: Call, stream=None):
    if c.kind == "gemv":
        tern_gemv(c.w, c.x, c.y, stream)
    elif c.kind == "swiglu":
        tern_gemv_swiglu(c.w, c.up, c.x, c.y, stream)
    elif c.kind == "smallm":
        tern_gemm_smallm(c.w, c.x, c.m, c.y, stream)
    elif c.kind == "smallm_swiglu":
        tern_gemm_smallm_swiglu(c.w, c.up, c.x, c.m, c.y, stream)
    else:
        raise ValueError(c.kind)


def run_calls(calls, stream=None):
    """Issue every call of a step as its own single-call launch."""
    for c in calls:
        run_call(c, stream)


def batch_of(calls):
    """The calls of a step as one tern_gemm_batched item array (independent items)."""
    return batch_items([(c.w, c.up, c.x, c.y, c.m) for c in calls])


def run_batched(batch, stream=None):
    """Issue a step through the persistent batched entry point."""
    tern_gemm_batched(batch, stream)


def _x(rng, m, k, device):
    import torch
    xb = synth.activations(rng, m, k)
    return torch.from_numpy(xb.view(np.int16)).to(device).view(torch.bfloat16), xb


def _y(m, rows, device):
    import torch
    return torch.empty((m, rows), dtype=torch.float32, device=device)


class Workload:
    """Calls of one step plus the host copies the tests need for the oracle."""

    def __init__(self, name: str, desc: str):
        self.name = name
        self.desc = desc
        self.calls: list[Call] = []
        self.host = []  # per call: dict(lin=..., up=..., x_bits=...)
        self.distinct = 0
        self.x_flat = None  # every call's x, contiguous (bf16)
        self.y_flat = None  # every call's y, contiguous (fp32)

    @property
    def packed_bytes(self) -> int:
        return sum(c.packed_bytes for c in self.calls)

    @property
    def algorithmic_bytes(self) -> int:
        return sum(c.algorithmic_bytes for c in self.calls)


def build(name: str, device="cuda", rotate_bytes: int = 400 * MiB, seed_offset: int = 0,
          distinct: int | None = None, layers: int | None = None) -> Workload:
    """Build workload c0..c4.

    c0/c1/c2/c3 repeat their unit over distinct device buffers until the
    packed weights of one step reach ``rotate_bytes`` (more than three times
    the 126 MB L2), so every call streams from HBM.  ``distinct`` seeded draws
    are made and reused across the buffers (the copies are separate
    allocations).  c4 is the 36-layer sweep, 1.74 GB per step by itself.
    """
    spec = synth.WORKLOADS[name]
    seed = spec["seed"] + 1000 * seed_offset
    rng = np.random.default_rng(seed)
    wl = Workload(name, spec["desc"])

    def units_for(unit_bytes):
        return max(1, -(-rotate_bytes // unit_bytes))

    if name in ("c0", "c1"):
        rows = 1024 if name == "c0" else 4096
        k = 4096
        n = units_for(rows * k // 4)
        nd = min(n, distinct or 16)
        lins = [synth.linear(rng, rows, k, name=f"{name}.{i}") for i in range(nd)]
        dms = [device_matrix(l, device) for l in lins]
        for i in range(n):
            j = i % nd
            w = dms[j] if i < nd else _clone(dms[j])
            x, xb = _x(rng, 1, k, device)
            wl.calls.append(Call("gemv", w, x, _y(1, rows, device), name=lins[j].name))
            wl.host.append(dict(lin=lins[j], x_bits=xb))
        wl.distinct = nd
    elif name == "c2":
        # early-layer code mix P(0)=0.71, P(+1)=P(-1)=0.145 for all three
        unit = (4096 * 12288 + 2 * 12288 * 4096) // 4
        n = units_for(unit)
        nd = min(n, distinct or 4)
        units = []
        for i in range(nd):
            down = synth.linear(rng, 4096, 12288, p_zero=0.71, name=f"down.{i}")
            gate = synth.linear(rng, 12288, 4096, p_zero=0.71, name=f"gate.{i}")
            up = synth.linear(rng, 12288, 4096, p_zero=0.71, name=f"up.{i}")
            units.append((down, gate, up, device_matrix(down, device), device_matrix(gate, device),
                          device_matrix(up, device)))
        for i in range(n):
            down, gate, up, dd, dg, du = units[i % nd]
            if i >= nd:
                dd, dg, du = _clone(dd), _clone(dg), _clone(du)
            x, xb = _x(rng, 1, 4096, device)
            wl.calls.append(Call("swiglu", dg, x, _y(1, 12288, device), up=du, name=gate.name))
            wl.host.append(dict(lin=gate, up=up, x_bits=xb))
            x2, xb2 = _x(rng, 1, 12288, device)
            wl.calls.append(Call("gemv", dd, x2, _y(1, 4096, device), name=down.name))
            wl.host.append(dict(lin=down, x_bits=xb2))
        wl.distinct = nd
    elif name == "c3":
        m = 7
        unit = (2 * 12288 * 4096 + 4096 * 12288) // 4
        n = units_for(unit)
        nd = min(n, distinct or 4)
        units = []
        for i in range(nd):
            gate = synth.linear(rng, 12288, 4096, name=f"gate.{i}")
            up = synth.linear(rng, 12288, 4096, name=f"up.{i}")
            down = synth.linear(rng, 4096, 12288, name=f"down.{i}")
            units.append((gate, up, down, device_matrix(gate, device), device_matrix(up, device),
                          device_matrix(down, device)))
        for i in range(n):
            gate, up, down, dg, du, dd = units[i % nd]
            if i >= nd:
                dg, du, dd = _clone(dg), _clone(du), _clone(dd)
            x, xb = _x(rng, m, 4096, device)
            wl.calls.append(Call("smallm_swiglu", dg, x, _y(m, 12288, device), m=m, up=du, name=gate.name))
            wl.host.append(dict(lin=gate, up=up, x_bits=xb))
            x2, xb2 = _x(rng, m, 12288, device)
            wl.calls.append(Call("smallm", dd, x2, _y(m, 4096, device), m=m, name=down.name))
            wl.host.append(dict(lin=down, x_bits=xb2))
        wl.distinct = nd
    elif name == "c4":
        nl = synth.LAYERS if layers is None else layers
        for layer in range(nl):
            for lname, rows, k in synth.LAYER_LINEARS:
                z = synth.sweep_zero_fraction(layer, lname)
                lin = synth.linear(rng, rows, k, p_zero=z, name=f"L{layer}.{lname}")
                x, xb = _x(rng, 1, k, device)
                wl.calls.append(Call("gemv", device_matrix(lin, device), x, _y(1, rows, device), name=lin.name))
                wl.host.append(dict(lin=lin, x_bits=xb))
        wl.distinct = len(wl.calls)
    else:
        raise ValueError(name)
    _pack_io(wl, device)
    return wl


def _pack_io(wl: Workload, device):
    """Place every call's x in one bf16 buffer and every y in one fp32 buffer
    (each call keeps a view), so a step's inputs and outputs move between host
    and device as one copy each.  Views stay 128-byte aligned: m*k is a
    multiple of 64 elements."""
    import torch
    nx = sum(c.x.numel() for c in wl.calls)
    ny = sum(c.y.numel() for c in wl.calls)
    xf = torch.empty(nx, dtype=torch.bfloat16, device=device)
    yf = torch.zeros(ny, dtype=torch.float32, device=device)
    ox = oy = 0
    for c in wl.calls:
        n = c.x.numel()
        xf[ox:ox + n].copy_(c.x.reshape(-1))
        c.x = xf[ox:ox + n].view(c.x.shape)
        ox += n
        n = c.y.numel()
        c.y = yf[oy:oy + n].view(c.y.shape)
        oy += n
    wl.x_flat, wl.y_flat = xf, yf


def io_copy(wl: Workload):
    """A second set of activation and output buffers for the calls of `wl`
    (same weights, same shapes and layout as wl.x_flat / wl.y_flat) and the
    batch that uses them, so a caller can prepare one step's inputs while
    another step runs.  Returns (x_flat, y_flat, batch, items)."""
    import torch
    xf = torch.empty_like(wl.x_flat)
    yf = torch.zeros_like(wl.y_flat)
    items, ox, oy = [], 0, 0
    for c in wl.calls:
        nx, ny = c.x.numel(), c.y.numel()
        items.append((c.w, c.up, xf[ox:ox + nx].view(c.x.shape), yf[oy:oy + ny].view(c.y.shape), c.m))
        ox += nx
        oy += ny
    return xf, yf, batch_items(items), items


def _clone(w: TernMatrix) -> TernMatrix:
    return TernMatrix(w.codes.clone(), w.scale.clone(), w.k, None if w.rowsum is None else w.rowsum.clone())


def layer_sweep(device="cuda", layers: int | None = None, distinct_layers: int = 4, seed: int = 4242):
    """The decode sweep in dependency order: per layer four launch groups,
    q|k|v, o, the gate/up pair (fused SwiGLU) and down, each one
    tern_gemm_batched call, so a token is 4 * layers launch groups in stream
    order.  ``distinct_layers`` layers of weights (about 46 MB each, more than
    the 126 MB L2 together) are drawn and reused cyclically over the layers.
    Returns (groups, packed_bytes_per_token, buffers): groups is the list of
    item arrays in call order; buffers keeps every tensor alive."""
    nl = synth.LAYERS if layers is None else layers
    rng = np.random.default_rng(seed)
    shapes = dict((n, (r, k)) for n, r, k in synth.LAYER_LINEARS)
    mats = []
    for _ in range(distinct_layers):
        d = {}
        for name, (rows, k) in shapes.items():
            d[name] = device_matrix(synth.linear(rng, rows, k, name=name), device)
        mats.append(d)
    groups, buffers, packed = [], [], 0
    for layer in range(nl):
        d = mats[layer % distinct_layers]
        plan = [[("q", None), ("k", None), ("v", None)], [("o", None)], [("gate", "up")], [("down", None)]]
        for grp in plan:
            items = []
            for name, up in grp:
                w = d[name]
                x, _ = _x(rng, 1, w.k, device)
                y = _y(1, w.rows, device)
                items.append((w, d[up] if up else None, x, y, 1))
                buffers += [x, y]
                packed += w.packed_bytes + (d[up].packed_bytes if up else 0)
            groups.append(batch_items(items))
    buffers.append(mats)
    return groups, packed, buffers
