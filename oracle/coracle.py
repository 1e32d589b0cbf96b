"""ctypes front end of the plain C oracle -- TEST INFRASTRUCTURE ONLY.

Builds ``hisparse_oracle.c`` with gcc (in-tree, ``oracle/_build/``) and wraps
one layer's state in numpy arrays so tests can read every field directly.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hisparse_oracle.c")
_OUT = os.path.join(_HERE, "_build", "libhisparse_oracle.so")
_lib = None

ERR_RANGE = 1
ERR_DUP = 2


def build():
    """Compile the C oracle (plain -O2, single-threaded)."""
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    if os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    tmp = _OUT + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-Wall", "-shared", "-fPIC", "-o", tmp, _SRC])
    os.replace(tmp, _OUT)
    return _OUT


class _Layer(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int32), ("k", ctypes.c_int32), ("B", ctypes.c_int32),
        ("P", ctypes.c_int64), ("rec", ctypes.c_int32),
        ("slot_pos", ctypes.c_void_p), ("lru", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p), ("miss_count", ctypes.c_void_p),
        ("unit_err", ctypes.c_void_p), ("hot", ctypes.c_void_p),
        ("host", ctypes.c_void_p), ("host_req_stride", ctypes.c_int64),
        ("host_split", ctypes.c_int64), ("host_tail", ctypes.c_void_p),
        ("plan_pos", ctypes.c_void_p), ("plan_slot", ctypes.c_void_p),
        ("plan_count", ctypes.c_void_p), ("mark", ctypes.c_void_p),
        ("mark_gen", ctypes.c_int32), ("hit", ctypes.c_void_p),
        ("misses", ctypes.c_void_p), ("ev", ctypes.c_void_p),
        ("first", ctypes.c_void_p), ("host_row_stride", ctypes.c_int64),
    ]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER(_Layer)
        vp = ctypes.c_void_p
        lib.hso_reset_unit.argtypes = [P, ctypes.c_int32]
        lib.hso_resolve_unit.argtypes = [P, ctypes.c_int32, vp, ctypes.c_int32, ctypes.c_int32, vp]
        lib.hso_resolve_unit.restype = ctypes.c_int32
        lib.hso_resolve_layer.argtypes = [P, vp, vp, ctypes.c_int32, ctypes.c_int32, vp]
        lib.hso_resolve_layer.restype = ctypes.c_int32
        lib.hso_resolve_layer_res.argtypes = [P, vp, vp, vp, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp]
        lib.hso_resolve_layer_res.restype = ctypes.c_int32
        lib.hso_resolve_unit_res.argtypes = [P, ctypes.c_int32, vp, ctypes.c_int32,
                                             ctypes.c_int32, vp, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, vp]
        lib.hso_resolve_unit_res.restype = ctypes.c_int32
        lib.hso_short_lookup_unit.argtypes = [P, ctypes.c_int32, vp, ctypes.c_int32,
                                              ctypes.c_int32, vp, ctypes.c_int32, ctypes.c_int32,
                                              vp]
        lib.hso_short_lookup_unit.restype = ctypes.c_int32
        lib.hso_set_newest_rows.argtypes = [P, vp, ctypes.c_int32]
        lib.hso_writeback.argtypes = [P, vp, ctypes.c_int32]
        lib.hso_writeback.restype = ctypes.c_int32
        lib.hso_replay.argtypes = [P, P, ctypes.c_int32]
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


class OracleLayer:
    """One layer of the C oracle for R requests.

    ``host`` is a read-only view of this layer's host pool rows [0, host_split)
    given either as a numpy uint8 array [R][rows][rec] or as a raw address plus
    request stride; rows [host_split, P) live in ``host_tail``, owned here and
    initialised to ``poison``.  ``keep_bytes=False`` keeps metadata only.
    """

    def __init__(self, R, k, B, P, rec, host=None, host_ptr=None, host_req_stride=0,
                 host_split=None, keep_bytes=True, metadata=True, poison=0xA5):
        if B < k:
            raise ValueError("B must be >= k")
        self.R, self.k, self.B, self.P, self.rec = R, k, B, P, rec
        self.host_split = P if host_split is None else host_split
        self._host_keep = host
        host_row_stride = 0
        if host is not None:
            host_ptr = host.ctypes.data
            host_req_stride = host.strides[0]
            host_row_stride = host.strides[1]
            if host.strides[2] != 1:
                raise ValueError("host rows must be contiguous bytes")
        m = metadata
        self.slot_pos = np.full((R, B), -1, np.int32) if m else None
        self.lru = np.tile(np.arange(B, dtype=np.int16), (R, 1)) if m else None
        self.page_table = np.full((R, P), -1, np.int32) if m else None
        self.miss_count = np.zeros(R, np.int32)
        self.unit_err = np.zeros(R, np.int32)
        self.hot = np.zeros((R, B + 1, rec), np.uint8) if keep_bytes else None
        tail_rows = P - self.host_split
        self.host_tail = np.full((R, tail_rows, rec), poison, np.uint8) if tail_rows else None
        self.plan_pos = np.zeros((R, k), np.int32)
        self.plan_slot = np.zeros((R, k), np.int32)
        self.plan_count = np.zeros(R, np.int32)
        self._mark = np.zeros(P, np.int32) if m else None
        self._hit = np.zeros(B, np.uint8)
        self._misses = np.zeros(k, np.int32)
        self._ev = np.zeros(B, np.int16)
        self._first = np.zeros(P, np.int32) if m else None
        self._s = _Layer(R, k, B, P, rec, _p(self.slot_pos), _p(self.lru), _p(self.page_table),
                         _p(self.miss_count), _p(self.unit_err), _p(self.hot),
                         ctypes.c_void_p(host_ptr) if host_ptr else None, host_req_stride,
                         self.host_split, _p(self.host_tail), _p(self.plan_pos),
                         _p(self.plan_slot), _p(self.plan_count), _p(self._mark), 0,
                         _p(self._hit), _p(self._misses), _p(self._ev), _p(self._first),
                         host_row_stride)
        self._lib = _load()

    def reset(self, r=None):
        for rr in (range(self.R) if r is None else [r]):
            self._lib.hso_reset_unit(ctypes.byref(self._s), rr)

    def admit(self, r, n, io=True):
        """Admission of unit r with its first n positions preloaded (reading
        R16 of oracle/tiny.py: the state resolving positions 0..n-1 in order
        from the reset state gives), as consecutive lists of k."""
        if not 0 <= n <= min(self.B, self.P):
            raise ValueError("preload length outside [0, min(B, P)]")
        self._lib.hso_reset_unit(ctypes.byref(self._s), r)
        out = np.empty(self.k, np.int32)
        pos, cnt = [], 0
        for c0 in range(0, n, self.k):
            chunk = np.full(self.k, -1, np.int32)
            m = min(n, c0 + self.k) - c0
            chunk[:m] = np.arange(c0, c0 + m, dtype=np.int32)
            e = self._lib.hso_resolve_unit(ctypes.byref(self._s), r, _p(chunk), -1,
                                           int(bool(io)), _p(out))
            assert e == 0
            cnt += int(self.plan_count[r])
        self.miss_count[r] = 0
        self.plan_count[r] = 0
        return cnt

    def preload_bytes(self, r, n):
        """A shared-index layer's side of an admission: its slots move in
        lockstep with the anchor's, so slot s < n holds its own host row s."""
        for s in range(n):
            self.hot[r, s] = self._host_keep[r, s] if s < self.host_split else self.host_tail[r, s - self.host_split]

    def resolve(self, sel, newest=None, num_reqs=None, io=True, res_blocks=None, res_tok=1,
                union=False):
        """sel int32 [R][k]; newest int32 [R] or None; res_blocks int32
        [R][nblk] (resident block table, -1 = not resident) or None; union:
        repeated positions share their first reference's row.
        Returns (out [R][k], err)."""
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        nr = self.R if num_reqs is None else num_reqs
        out = np.full((self.R, self.k), -1, np.int32)
        nw = None if newest is None else np.ascontiguousarray(newest, dtype=np.int32)
        if res_blocks is None and not union:
            e = self._lib.hso_resolve_layer(ctypes.byref(self._s), _p(sel), _p(nw), nr,
                                            int(bool(io)), _p(out))
        else:
            rb = None if res_blocks is None else np.ascontiguousarray(res_blocks, dtype=np.int32)
            e = self._lib.hso_resolve_layer_res(ctypes.byref(self._s), _p(sel), _p(nw), _p(rb),
                                                0 if rb is None else rb.shape[1], int(res_tok),
                                                int(bool(union)), nr, int(bool(io)), _p(out))
        return out, e

    def resolve_with_seq_lens(self, sel, newest, prev, seq_lens, num_reqs=None, io=True,
                              res_blocks=None, res_tok=1, union=False):
        """One layer-step where each request carries its sequence length
        (reading R17 of oracle/tiny.py): a request with seq_len <= B grows its
        buffer by its previous token (a one-entry resolve of ``prev[r]`` when
        it is >= 0, whose record the write-back has just stored; otherwise
        its miss count and plan are 0) and then looks its selections up by
        position; a longer one is resolved as usual.  The write-back itself
        (``writeback``) comes first, as for any step.  Returns (out, err)."""
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        nr = self.R if num_reqs is None else num_reqs
        out = np.full((self.R, self.k), -1, np.int32)
        rb = None if res_blocks is None else np.ascontiguousarray(res_blocks, dtype=np.int32)
        nblk = 0 if rb is None else rb.shape[1]
        err = 0
        grow = np.full(self.k, -1, np.int32)
        scratch = np.empty(self.k, np.int32)
        for r in range(nr):
            nw = -1 if newest is None else int(newest[r])
            blk = None if rb is None else rb[r]
            if int(seq_lens[r]) <= self.B:
                if prev is not None and int(prev[r]) >= 0:
                    grow[0] = int(prev[r])
                    e = self._lib.hso_resolve_unit_res(ctypes.byref(self._s), r, _p(grow), -1,
                                                       int(bool(io)), None, 0, 1, 0,
                                                       _p(scratch))
                    assert e == 0, "the previous token is a valid one-entry selection"
                else:
                    self.miss_count[r] = 0
                    self.plan_count[r] = 0
                row = np.ascontiguousarray(sel[r])
                o = np.empty(self.k, np.int32)
                err |= self._lib.hso_short_lookup_unit(ctypes.byref(self._s), r, _p(row), nw,
                                                       int(seq_lens[r]), _p(blk), nblk,
                                                       int(res_tok), _p(o))
                out[r] = o
            else:
                row = np.ascontiguousarray(sel[r])
                o = np.empty(self.k, np.int32)
                err |= self._lib.hso_resolve_unit_res(ctypes.byref(self._s), r, _p(row), nw,
                                                      int(bool(io)), _p(blk), nblk, int(res_tok),
                                                      int(bool(union)), _p(o))
                out[r] = o
        return out, err

    def set_newest_rows(self, rows, num_reqs=None):
        rows = np.ascontiguousarray(rows, dtype=np.uint8)
        self._lib.hso_set_newest_rows(ctypes.byref(self._s), _p(rows),
                                      self.R if num_reqs is None else num_reqs)

    def writeback(self, pos, num_reqs=None):
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        e = self._lib.hso_writeback(ctypes.byref(self._s), _p(pos),
                                    self.R if num_reqs is None else num_reqs)
        if e:
            raise ValueError("write-back position outside the model-owned rows")

    def replay_into(self, follower, num_reqs=None):
        """Copy this (anchor) layer's last plan into ``follower``'s hot rows."""
        self._lib.hso_replay(ctypes.byref(self._s), ctypes.byref(follower._s),
                             self.R if num_reqs is None else num_reqs)

    def host_row(self, r, p):
        """This model's view of host row (r, p)."""
        if p >= self.host_split:
            return self.host_tail[r, p - self.host_split]
        if self._host_keep is not None:
            return self._host_keep[r, p]
        raise ValueError("host rows given by address only")
