"""The C ABI library on a machine without a GPU: it loads, exports every
declared symbol, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

from host_offload_serving_gb300 import hisparse as H

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "hisparse.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hisparse_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = H.load()
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    bound = {n for n, _, _ in H.SIGNATURES}
    assert set(names) == bound, set(names) ^ bound


# Wrappers that return the C function's out-parameters instead of taking them.
_OUT_PARAMS = {"hisparse_init": 1, "hisparse_get_status": 1, "hisparse_get_info": 1,
               "hisparse_host_alloc": 1, "hisparse_host_alloc_kind": 1,
               "hisparse_host_hugepage_bytes": 1}


def declared_arity():
    """Number of parameters of every function in include/hisparse.h."""
    src = open(os.path.join(ROOT, "include", "hisparse.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(hisparse_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_arity_matches_the_header():
    """Every C function's argtypes and every same-name Python wrapper take
    the parameters the header declares (wrappers that return out-parameters
    take that many fewer)."""
    import inspect
    arity = declared_arity()
    for name, _, args in H.SIGNATURES:
        assert len(args) == arity[name], (name, len(args), arity[name])
        fn = getattr(H, name, None)
        if fn is None:
            continue
        n = len(inspect.signature(fn).parameters)
        assert n + _OUT_PARAMS.get(name, 0) == arity[name], (name, n, arity[name])


def test_strerror_and_codes():
    lib = H.load()
    assert lib.hisparse_strerror(0) == b"ok"
    for code in (H.EINVAL, H.EBOUND, H.ENOMEM, H.ECUDA, H.EROLE):
        assert lib.hisparse_strerror(code) not in (b"ok", b"unknown error")
    assert lib.hisparse_strerror(-99) == b"unknown error"


def _cfg(R=2, L=1, k=4, B=8, P=100, rec=1152, cs=0, rc=0, lookup=0, anchor=None):
    arr = None
    if anchor is not None:
        arr = (ctypes.c_int32 * len(anchor))(*anchor)
    c = H.Config(R, L, k, B, P, rec, cs, rc, lookup, ctypes.cast(arr, ctypes.c_void_p) if arr else None)
    c._keep = arr
    return c


def _bufs(L=1, host=0x1000, hot=0x2000, rs=1152 * 100, row=1152, hrs=1152 * 9, hrow=1152):
    return [H.LayerBuffers(host, rs, row, hot, hrs, hrow, None) for _ in range(L)]


@pytest.mark.parametrize("kw,bufkw,code", [
    (dict(B=2, k=4), {}, H.EBOUND),                     # B < k
    (dict(B=40000, k=4), {}, H.EBOUND),                 # int16 LRU order
    (dict(rec=1000), dict(row=1008, hrow=1008), H.EINVAL),  # record not a multiple of 16
    (dict(R=0), {}, H.EINVAL),
    (dict(R=9000), {}, H.EBOUND),
    (dict(P=0), {}, H.EINVAL),
    (dict(cs=17), {}, H.EBOUND),
    (dict(lookup=7), {}, H.EINVAL),
    (dict(L=3, anchor=[-1, 0, 1]), dict(L=3), H.EROLE),   # anchor of an anchor
    (dict(L=2, anchor=[1, 1]), dict(L=2), H.EROLE),       # own anchor
    (dict(L=2, anchor=[-1, 5]), dict(L=2), H.EROLE),      # out of range
    ({}, dict(host=0x1004), H.EINVAL),                   # misaligned host pool
    ({}, dict(hot=0), H.EINVAL),                         # NULL hot buffer
    ({}, dict(row=1000), H.EINVAL),                      # row stride < record
    ({}, dict(rs=1152 * 100 + 8), H.EINVAL),             # stride not a multiple of 16
])
def test_init_rejects_on_host(kw, bufkw, code):
    L = kw.get("L", 1)
    rc, h = H.hisparse_init(_cfg(**kw), _bufs(**bufkw) if "L" in bufkw else _bufs(L=L, **bufkw))
    assert rc == code and h is None


def test_init_without_gpu_reports_cuda_error_not_crash():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = H.hisparse_init(_cfg(), _bufs())
    assert rc in (H.ECUDA, H.EINVAL) and h is None


def test_calls_on_null_handle_are_rejected():
    lib = H.load()
    assert lib.hisparse_resolve(None, 0, 1, None, None, 1, 0, None) == H.EINVAL
    assert lib.hisparse_writeback(None, 0, 1, None, None, None) == H.EINVAL
    assert lib.hisparse_prefetch_plan(None, 0, 1, None, None) == H.EINVAL
    assert lib.hisparse_reset(None, 0, None) == H.EINVAL
    assert lib.hisparse_destroy(None) == H.EINVAL
    f = ctypes.c_uint32()
    assert lib.hisparse_get_status(None, ctypes.byref(f), None) == H.EINVAL
    assert H.hisparse_host_alloc(0)[0] == H.EINVAL


def test_hugepage_query_on_ordinary_memory():
    a = np.zeros(1 << 20, np.uint8)
    rc, huge = H.hisparse_host_hugepage_bytes(a.ctypes.data, a.nbytes)
    assert rc == H.OK and 0 <= huge <= a.nbytes


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes mirrors of the header's structs have the C sizes and offsets
    (compiled with the host C compiler against include/hisparse.h)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    prog = tmp_path / "layout.c"
    prog.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "hisparse.h"\n'
        "int main(void) {\n"
        '  printf("%zu %zu %zu %zu\\n", sizeof(hisparse_resolve_options),'
        " offsetof(hisparse_resolve_options, d_res_blocks),"
        " offsetof(hisparse_resolve_options, res_max_blocks),"
        " offsetof(hisparse_resolve_options, sel_block_tokens));\n"
        '  printf("%zu %zu %zu\\n", sizeof(hisparse_config), sizeof(hisparse_layer_buffers),'
        " sizeof(hisparse_info));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.check_call([cc, "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)])
    got = subprocess.check_output([str(exe)], text=True).split("\n")
    o = H.ResolveOptions
    assert [int(x) for x in got[0].split()] == [ctypes.sizeof(o), o.d_res_blocks.offset,
                                                o.res_max_blocks.offset,
                                                o.sel_block_tokens.offset]
    assert [int(x) for x in got[1].split()] == [ctypes.sizeof(H.Config),
                                                ctypes.sizeof(H.LayerBuffers),
                                                ctypes.sizeof(H.Info)]


def test_resolve_ex_without_a_handle_is_rejected():
    o = H.ResolveOptions(None, None, 0x1000, 4, 64, 1)
    assert H.hisparse_resolve_ex(None, 0, 0x10, None, None, o, 0x20, 0, None) == H.EINVAL
    assert H.hisparse_resolve_ex(None, 0, 0x10, None, None, None, 0x20, 0, None) == H.EINVAL


def test_copy_argument_checks_need_no_gpu():
    """hisparse_copy refuses bad sizes and alignments before touching CUDA;
    zero bytes is a no-op.  A shared-layer replay on no handle is refused."""
    lib = H.load()
    assert H.hisparse_copy(0x1000, 0x2000, 24, None) == H.EINVAL      # not a multiple of 16
    assert H.hisparse_copy(0x1008, 0x2000, 32, None) == H.EINVAL      # misaligned destination
    assert H.hisparse_copy(0x1000, 0x2004, 32, None) == H.EINVAL      # misaligned source
    assert H.hisparse_copy(None, 0x2000, 32, None) == H.EINVAL
    assert H.hisparse_copy(0x1000, 0x2000, -16, None) == H.EINVAL
    assert H.hisparse_copy(0x1000, 0x2000, 0, None) == H.OK
    assert lib.hisparse_prefetch_plan(None, 0, -1, None, None) == H.EINVAL
