"""Seeded synthetic KV records (input generation only).

Builds ``records.c`` with gcc on first use (in-tree, ``workload/_build/``) and
fills host-pool rows through it.  Values are bf16 N(0,1) draws, keyed by
(layer, request, position) so that any row can be regenerated on its own.
"""
import ctypes
import os
import statistics
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "records.c")
_OUT = os.path.join(_HERE, "_build", "libwlrecords.so")
_lib = None
_table = None

POISON = 0xA5  # fill byte of host rows that no one has written yet


def build():
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    if os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    tmp = _OUT + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-Wall", "-shared", "-fPIC", "-o", tmp,
                           _SRC, "-lpthread"])
    os.replace(tmp, _OUT)
    return _OUT


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.wl_fill_records.restype = ctypes.c_int32
        lib.wl_fill_records.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int32, ctypes.c_uint64, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                                        ctypes.c_int32]
        _lib = lib
    return _lib


def f32_to_bf16_rne(x):
    """bf16 bits of float32 values, round to nearest even (NaN not expected)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def normal_table():
    """65536 bf16 values: the N(0,1) quantile at (u + 0.5) / 65536."""
    global _table
    if _table is None:
        nd = statistics.NormalDist()
        q = np.array([nd.inv_cdf((u + 0.5) / 65536.0) for u in range(65536)], dtype=np.float64)
        _table = np.ascontiguousarray(f32_to_bf16_rne(q.astype(np.float32)))
    return _table


def threads():
    return max(1, min(32, os.cpu_count() or 1))


def fill(dst_ptr, n_rows, row_stride, rec, seed, layer, req, pos0):
    """Write records for positions pos0..pos0+n_rows-1 at dst_ptr (row stride)."""
    t = normal_table()
    e = _load().wl_fill_records(ctypes.c_void_p(dst_ptr), n_rows, row_stride, rec, seed, layer,
                                req, pos0, ctypes.c_void_p(t.ctypes.data), threads())
    if e:
        raise ValueError("bad record-fill arguments")


def records(w, layer, req, positions):
    """Records of the given positions as a numpy uint8 array [n][rec]."""
    positions = [int(p) for p in positions]
    out = np.empty((len(positions), w.rec), dtype=np.uint8)
    for i, p in enumerate(positions):
        fill(out[i].ctypes.data, 1, w.rec, w.rec, w.seed, layer, req, p)
    return out


def fill_host_pool(w, geometry, layers=None):
    """Fill rows [0, L_ctx) of every (layer, request) unit; poison the rest.

    ``geometry(l)`` gives layer l's (address of row (0, 0), request stride,
    row stride) in bytes: row (l, r, p) lives at addr + r*req_stride +
    p*row_stride.
    """
    layers = range(w.L) if layers is None else layers
    for l in layers:
        base, req_stride, row_stride = geometry(l)
        for r in range(w.R):
            unit = base + r * req_stride
            fill(unit, w.L_ctx, row_stride, w.rec, w.seed, l, r, 0)
            if row_stride == w.rec and w.P > w.L_ctx:
                ctypes.memset(unit + w.L_ctx * w.rec, POISON, (w.P - w.L_ctx) * w.rec)
            else:
                for p in range(w.L_ctx, w.P):
                    ctypes.memset(unit + p * row_stride, POISON, w.rec)


def new_token_records(w):
    """KV of each decode step's new token: uint8 [steps][L][R][rec] (write-through only)."""
    if not w.write_through:
        return None
    out = np.empty((w.steps, w.L, w.R, w.rec), dtype=np.uint8)
    for l in range(w.L):
        for r in range(w.R):
            for t in range(w.steps):
                fill(out[t, l, r].ctypes.data, 1, w.rec, w.rec, w.seed, l, r, w.L_ctx + t)
    return out
