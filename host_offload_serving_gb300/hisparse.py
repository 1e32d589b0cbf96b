"""Python binding of the C ABI in ``include/hisparse.h`` (argument marshalling only).

Every function keeps the C name and takes plain integers for pointers and
streams (``tensor.data_ptr()``, ``torch.cuda.Stream.cuda_stream``).  Nothing
here computes any part of RESOLVE: all of it runs in ``libhisparse.so``.  If the
library cannot be built or loaded the import fails -- there is no fallback.
"""
import ctypes
import os

from . import _build

OK, EINVAL, EBOUND, ENOMEM, ECUDA, EROLE = 0, -1, -2, -3, -4, -5
ERR_RANGE, ERR_DUP = 1, 2
RECORD_PLAN, SKIP_IO, FROM_MIRROR, UNION, WITH_SHARED = 1, 2, 4, 8, 16
LOOKUP_PAGE_TABLE, LOOKUP_HASH = 0, 1
HOST_HUGE, HOST_PINNED = 0, 1

_i32, _i64, _u32, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p


class Config(ctypes.Structure):
    _fields_ = [("num_requests", _i32), ("num_layers", _i32), ("top_k", _i32),
                ("buffer_slots", _i32), ("host_rows", _i64), ("record_bytes", _i32),
                ("ctas_per_request", _i32), ("replay_ctas", _i32), ("lookup", _i32),
                ("anchor_of", _vp)]


class LayerBuffers(ctypes.Structure):
    _fields_ = [("host_pool", _vp), ("host_req_stride", _i64), ("host_row_stride", _i64),
                ("hot", _vp), ("hot_req_stride", _i64), ("hot_row_stride", _i64),
                ("mirror", _vp)]


class Info(ctypes.Structure):
    _fields_ = [("ctas_per_request", _i32), ("threads_per_cta", _i32), ("smem_bytes", _i32),
                ("hash_capacity", _i32), ("replay_ctas", _i32), ("sm_count", _i32),
                ("metadata_bytes", _i64), ("lookup", _i32)]


# (name, restype, argtypes) of every exported symbol, in header order
SIGNATURES = [
    ("hisparse_init", _i32, [ctypes.POINTER(Config), ctypes.POINTER(LayerBuffers),
                             ctypes.POINTER(_vp)]),
    ("hisparse_destroy", _i32, [_vp]),
    ("hisparse_resolve", _i32, [_vp, _i32, _vp, _vp, _vp, _vp, _u32, _vp]),
    ("hisparse_resolve_step", _i32, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _u32, _vp]),
    ("hisparse_resolve_resident", _i32, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp,
                                         _u32, _vp]),
    ("hisparse_resolve_ex", _i32, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _u32, _vp]),
    ("hisparse_admit", _i32, [_vp, _i32, _vp, _i32, _vp, _vp]),
    ("hisparse_writeback", _i32, [_vp, _i32, _vp, _vp, _vp, _vp]),
    ("hisparse_prefetch_plan", _i32, [_vp, _i32, _i32, _vp, _vp]),
    ("hisparse_copy", _i32, [_vp, _vp, _i64, _vp]),
    ("hisparse_copy_miss_counts", _i32, [_vp, _i32, _vp, _vp]),
    ("hisparse_get_status", _i32, [_vp, ctypes.POINTER(_u32), _vp]),
    ("hisparse_export_state", _i32, [_vp, _i32, _vp, _vp, _vp, _vp]),
    ("hisparse_import_state", _i32, [_vp, _i32, _vp, _vp, _vp, _vp]),
    ("hisparse_export_plan", _i32, [_vp, _i32, _vp, _vp, _vp]),
    ("hisparse_reset", _i32, [_vp, _i32, _vp]),
    ("hisparse_set_l2_persisting", _i32, [_vp, _i64]),
    ("hisparse_get_info", _i32, [_vp, ctypes.POINTER(Info)]),
    ("hisparse_host_alloc", _i32, [ctypes.c_size_t, ctypes.POINTER(_vp)]),
    ("hisparse_host_free", _i32, [_vp]),
    ("hisparse_host_alloc_kind", _i32, [ctypes.c_size_t, _i32, ctypes.POINTER(_vp)]),
    ("hisparse_host_hugepage_bytes", _i32, [_vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]),
    ("hisparse_last_cuda_error", _i32, []),
    ("hisparse_strerror", ctypes.c_char_p, [_i32]),
]

_lib = None


def load(path=None):
    """Build (if stale) and load libhisparse.so; raises if that is impossible."""
    global _lib
    if _lib is None:
        path = path or _build.build()
        lib = ctypes.CDLL(path)
        for name, res, args in SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def library_path():
    return os.path.abspath(load()._name)


class HiSparseError(RuntimeError):
    def __init__(self, code, what):
        lib = load()
        msg = lib.hisparse_strerror(code).decode()
        if code == ECUDA:
            msg += f" (cudaError {lib.hisparse_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [{code}]")
        self.code = code


def check(code, what):
    if code != OK:
        raise HiSparseError(code, what)
    return code


# ---- thin same-name wrappers ---------------------------------------------
def hisparse_init(cfg, layers):
    h = _vp()
    arr = (LayerBuffers * len(layers))(*layers)
    rc = load().hisparse_init(ctypes.byref(cfg), arr, ctypes.byref(h))
    return rc, h.value


def hisparse_destroy(h):
    return load().hisparse_destroy(h)


def hisparse_resolve(h, layer, d_sel, d_num_reqs, d_newest, d_out, flags, stream):
    return load().hisparse_resolve(h, layer, d_sel, d_num_reqs, d_newest, d_out, flags, stream)


def hisparse_resolve_step(h, layer, d_sel, d_num_reqs, d_newest, d_prev_pos, d_new_rows, d_out,
                          flags, stream):
    return load().hisparse_resolve_step(h, layer, d_sel, d_num_reqs, d_newest, d_prev_pos,
                                        d_new_rows, d_out, flags, stream)


class ResolveOptions(ctypes.Structure):
    """hisparse_resolve_options."""
    _fields_ = [("d_prev_pos", ctypes.c_void_p), ("d_new_rows", ctypes.c_void_p),
                ("d_res_blocks", ctypes.c_void_p), ("res_max_blocks", ctypes.c_int32),
                ("res_block_tokens", ctypes.c_int32), ("sel_block_tokens", ctypes.c_int32),
                ("d_seq_lens", ctypes.c_void_p)]


def hisparse_resolve_ex(h, layer, d_sel, d_num_reqs, d_newest, opt, d_out, flags, stream):
    return load().hisparse_resolve_ex(h, layer, d_sel, d_num_reqs, d_newest,
                                      ctypes.addressof(opt) if opt is not None else None, d_out,
                                      flags, stream)


def hisparse_resolve_resident(h, layer, d_sel, d_num_reqs, d_newest, d_prev_pos, d_new_rows,
                              d_res_blocks, res_max_blocks, res_block_tokens, d_out, flags,
                              stream):
    return load().hisparse_resolve_resident(h, layer, d_sel, d_num_reqs, d_newest, d_prev_pos,
                                            d_new_rows, d_res_blocks, res_max_blocks,
                                            res_block_tokens, d_out, flags, stream)


def hisparse_writeback(h, layer, d_pos, d_new_rows, d_num_reqs, stream):
    return load().hisparse_writeback(h, layer, d_pos, d_new_rows, d_num_reqs, stream)


def hisparse_prefetch_plan(h, anchor_layer, follower_layer, d_num_reqs, stream):
    return load().hisparse_prefetch_plan(h, anchor_layer, follower_layer, d_num_reqs, stream)


def hisparse_copy(dst, src, nbytes, stream):
    return load().hisparse_copy(dst, src, nbytes, stream)


def hisparse_copy_miss_counts(h, layer, d_dst, stream):
    return load().hisparse_copy_miss_counts(h, layer, d_dst, stream)


def hisparse_get_status(h, unit_err_ptr=None):
    f = _u32()
    rc = load().hisparse_get_status(h, ctypes.byref(f), unit_err_ptr)
    return rc, f.value


def hisparse_export_state(h, layer, slot_pos, lru, page_table, miss_counts):
    return load().hisparse_export_state(h, layer, slot_pos, lru, page_table, miss_counts)


def hisparse_import_state(h, layer, slot_pos, lru, page_table, miss_counts):
    return load().hisparse_import_state(h, layer, slot_pos, lru, page_table, miss_counts)


def hisparse_export_plan(h, layer, count, pos, slot):
    return load().hisparse_export_plan(h, layer, count, pos, slot)


def hisparse_reset(h, layer, stream):
    return load().hisparse_reset(h, layer, stream)


def hisparse_set_l2_persisting(h, nbytes):
    return load().hisparse_set_l2_persisting(h, nbytes)


def hisparse_get_info(h):
    info = Info()
    rc = load().hisparse_get_info(h, ctypes.byref(info))
    return rc, info


def hisparse_host_alloc(nbytes):
    p = _vp()
    rc = load().hisparse_host_alloc(nbytes, ctypes.byref(p))
    return rc, p.value


def hisparse_host_alloc_kind(nbytes, kind):
    p = _vp()
    rc = load().hisparse_host_alloc_kind(nbytes, kind, ctypes.byref(p))
    return rc, p.value


def hisparse_host_free(p):
    return load().hisparse_host_free(p)


def hisparse_host_hugepage_bytes(p, nbytes):
    v = ctypes.c_size_t()
    rc = load().hisparse_host_hugepage_bytes(p, nbytes, ctypes.byref(v))
    return rc, v.value


def hisparse_admit(h, layer, d_reqs, n, d_preload, stream):
    return load().hisparse_admit(h, layer, d_reqs, n, d_preload, stream)
