"""The C ABI on the host (no GPU): the library loads, exports what include/dgc.h declares, and
rejects bad arguments synchronously before it makes any CUDA call.

Every rejected call below breaks at least one host-side rule, so nothing reaches the device even
where a GPU is present.
"""
import ctypes
import math
import os
import re

import pytest

import sparsified_gradient_compression_gb300 as dgc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    dgc.build()
    return dgc.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "dgc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dgc_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert len(names) >= 12
    for name in names:
        assert hasattr(L, name), name


def test_status_strings(L):
    assert dgc.dgc_status_string(0) == "ok"
    assert "malformed" in dgc.dgc_status_string(dgc.ECORRUPT)
    assert dgc.dgc_status_string(12345) == "unknown status"


P = dgc.make_params


def test_workspace_and_bounds_queries(L):
    p = P(sparsity=0.999)
    assert dgc.dgc_compress_max_out(1_048_576, 1, p) == 1049 + 1  # sum of ceilings + slack
    assert dgc.dgc_compress_max_out(1000, 1, P(sparsity=0.0)) == 1000
    assert dgc.dgc_compress_max_out(1000, 1, P(sparsity=1.0)) == 0
    assert dgc.dgc_compress_max_out(1000, 3, P(mode=dgc.SELECT_ADACOMP, bin_size=7)) == 1000
    ps = P(mode=dgc.SELECT_SAMPLED, sparsity=0.999, reselect_factor=1.3)
    assert dgc.dgc_compress_max_out(1 << 30, 1, ps) >= int(1.3 * 1073742)
    w1 = dgc.dgc_compress_workspace(1 << 20, 1, p)
    w2 = dgc.dgc_compress_workspace(1 << 21, 1, p)
    assert 8 * (1 << 20) < w1 < w2  # candidate slots and list: 8 bytes per entry
    assert dgc.dgc_encode_max_bytes(10, 1000) == 32 + 6 * 10 + 2
    assert dgc.dgc_encode_max_bytes(0, 200000) == 32 + 6 * 3 + 2
    assert dgc.dgc_decode_workspace([32, 40, 44], 100) > 0


@pytest.mark.parametrize("sizes", [[31], [33], [32 + 6], [32 + 6 + 2 + 6], [0]])
def test_decode_rejects_impossible_sizes(L, sizes):
    with pytest.raises(dgc.DGCError) as e:
        dgc.dgc_decode_workspace(sizes, 100)
    assert e.value.code == dgc.ECORRUPT


FAKE = 1 << 40  # aligned non-null address that is never dereferenced


def _compress(L, n=1024, nseg=1, params=None, g=FAKE, u=FAKE, v=FAKE, seg=FAKE, out_idx=FAKE,
              out_val=FAKE, cap=None, count=FAKE, status=FAKE, ws=FAKE, ws_bytes=None):
    params = params or P()

    def query(f):
        try:
            return f(n, nseg, params)
        except dgc.DGCError:
            return 0

    cap = query(dgc.dgc_compress_max_out) if cap is None else cap
    ws_bytes = query(dgc.dgc_compress_workspace) if ws_bytes is None else ws_bytes
    return L.dgc_compress(g, u, v, n, seg, nseg, ctypes.byref(params), out_idx, out_val, cap,
                          count, None, status, ws, ws_bytes, None)


@pytest.mark.parametrize("case,code", [
    (dict(n=-1), dgc.EINVAL),
    (dict(n=2**32), dgc.EUNSUPPORTED),
    (dict(nseg=0), dgc.EINVAL),
    (dict(params=P(sparsity=1.5)), dgc.EINVAL),
    (dict(params=P(sparsity=float("nan"))), dgc.EINVAL),
    (dict(params=P(momentum=float("inf"))), dgc.EINVAL),
    (dict(params=P(mode=7)), dgc.EINVAL),
    (dict(params=P(mode=dgc.SELECT_SAMPLED, sample_ratio=0.0)), dgc.EINVAL),
    (dict(params=P(mode=dgc.SELECT_SAMPLED, sample_ratio=1e-12)), dgc.EINVAL),
    (dict(params=P(mode=dgc.SELECT_SAMPLED, reselect_factor=0.5)), dgc.EINVAL),
    (dict(params=P(mode=dgc.SELECT_ADACOMP, bin_size=0)), dgc.EINVAL),
    (dict(g=None), dgc.EINVAL),
    (dict(g=FAKE + 4), dgc.EINVAL),
    (dict(u=FAKE + 8), dgc.EINVAL),
    (dict(v=FAKE + 12), dgc.EINVAL),
    (dict(seg=None), dgc.EINVAL),
    (dict(count=None), dgc.EINVAL),
    (dict(status=None), dgc.EINVAL),
    (dict(ws=None), dgc.EINVAL),
    (dict(ws=FAKE + 16), dgc.EINVAL),
    (dict(ws_bytes=100), dgc.EINVAL),
    (dict(cap=1, params=P(sparsity=0.5)), dgc.ECAPACITY),
    (dict(out_idx=None), dgc.EINVAL),
])
def test_compress_rejects_on_host(L, case, code):
    assert _compress(L, **case) == code


def test_encode_and_decode_reject_on_host(L):
    ws = dgc.dgc_encode_workspace(10)
    e = L.dgc_encode
    assert e(FAKE, FAKE, FAKE, -1, 100, FAKE, 100, FAKE, FAKE, FAKE, ws, None) == dgc.EINVAL
    assert e(FAKE, FAKE, FAKE, 10, 2**32, FAKE, 100, FAKE, FAKE, FAKE, ws, None) == dgc.EUNSUPPORTED
    assert e(FAKE, FAKE, FAKE, 10, 100, FAKE + 4, 100, FAKE, FAKE, FAKE, ws, None) == dgc.EINVAL
    assert e(FAKE, FAKE, None, 10, 100, FAKE, 100, FAKE, FAKE, FAKE, ws, None) == dgc.EINVAL
    assert e(FAKE, FAKE, FAKE, 10, 100, FAKE, 100, FAKE, FAKE, FAKE, ws - 1, None) == dgc.EINVAL
    d = L.dgc_decode_accumulate
    ptrs = (ctypes.c_void_p * 1)(FAKE)
    good = (ctypes.c_uint64 * 1)(40)
    bad = (ctypes.c_uint64 * 1)(37)
    cast = lambda a: ctypes.cast(a, ctypes.c_void_p)  # noqa: E731
    wsb = dgc.dgc_decode_workspace([40], 100)
    assert d(cast(ptrs), cast(bad), 1, FAKE, 100, 0, FAKE, FAKE, wsb, None) == dgc.ECORRUPT
    assert d(cast(ptrs), cast(good), 1, FAKE, 100, 0, FAKE, FAKE, wsb - 1, None) == dgc.EINVAL
    assert d(cast(ptrs), cast(good), 1, None, 100, 0, FAKE, FAKE, wsb, None) == dgc.EINVAL
    ptrs_mis = (ctypes.c_void_p * 1)(FAKE + 4)
    assert d(cast(ptrs_mis), cast(good), 1, FAKE, 100, 0, FAKE, FAKE, wsb, None) == dgc.EINVAL
    assert d(cast(ptrs), cast(good), -1, FAKE, 100, 0, FAKE, FAKE, wsb, None) == dgc.EINVAL


def test_decode_apply_rejects_on_host(L):
    d = L.dgc_decode_apply
    ptrs = (ctypes.c_void_p * 1)(FAKE)
    good = (ctypes.c_uint64 * 1)(40)
    bad = (ctypes.c_uint64 * 1)(37)
    cast = lambda a: ctypes.cast(a, ctypes.c_void_p)  # noqa: E731
    wsb = dgc.dgc_decode_workspace([40], 100)
    for lr in (-0.0, -1.0, math.inf, -math.inf, math.nan):  # lr must be finite, sign bit clear
        assert d(cast(ptrs), cast(good), 1, FAKE, 100, lr, FAKE, FAKE, wsb, None) == dgc.EINVAL
    assert d(cast(ptrs), cast(bad), 1, FAKE, 100, 0.5, FAKE, FAKE, wsb, None) == dgc.ECORRUPT
    assert d(cast(ptrs), cast(good), 1, FAKE, 100, 0.5, FAKE, FAKE, wsb - 1, None) == dgc.EINVAL
    assert d(cast(ptrs), cast(good), 1, None, 100, 0.5, FAKE, FAKE, wsb, None) == dgc.EINVAL
    assert d(cast(ptrs), cast(good), 1, FAKE, 2**32, 0.5, FAKE, FAKE, wsb, None) == dgc.EUNSUPPORTED


def test_quant_entry_points_reject_on_host(L):
    cast = lambda a: ctypes.cast(a, ctypes.c_void_p)  # noqa: E731
    ews = dgc.dgc_encode_workspace(10)
    e = L.dgc_encode_quant
    for alpha, bits in ((0.0, 8), (-1.0, 16), (math.inf, 8), (math.nan, 8), (1.0, 4), (1.0, 32)):
        assert e(FAKE, FAKE, FAKE, 10, 100, alpha, bits, None, FAKE, 100, FAKE, FAKE, FAKE, ews,
                 None) == dgc.EINVAL
    # the size fixes T for a known width: 16-bit messages are 32 + 4T bytes
    sizes = (ctypes.c_uint64 * 1)(33)
    out = ctypes.c_size_t(0)
    w = L.dgc_decode_workspace_quant
    assert w(1, cast(sizes), 100, 16, ctypes.byref(out)) == dgc.ECORRUPT
    assert w(1, cast(sizes), 100, 12, ctypes.byref(out)) == dgc.EINVAL
    assert dgc.dgc_decode_workspace_quant([40], 100, 16) > 0   # T = 2
    assert dgc.dgc_decode_workspace_quant([42], 100, 8) > 0    # T = 3: 35 -> 36, + 6
    ptrs = (ctypes.c_void_p * 1)(FAKE)
    good = (ctypes.c_uint64 * 1)(40)
    wsb = dgc.dgc_decode_workspace_quant([40], 100, 16)
    d, a = L.dgc_decode_accumulate_quant, L.dgc_decode_apply_quant
    for bits, alpha in ((12, 1.0), (16, 0.0), (16, math.nan)):
        assert d(cast(ptrs), cast(good), 1, bits, alpha, FAKE, 100, 0, FAKE, FAKE, wsb,
                 None) == dgc.EINVAL
        assert a(cast(ptrs), cast(good), 1, bits, alpha, FAKE, 100, 0.5, FAKE, FAKE, wsb,
                 None) == dgc.EINVAL
    assert a(cast(ptrs), cast(good), 1, 16, 1.0, FAKE, 100, -0.0, FAKE, FAKE, wsb,
             None) == dgc.EINVAL
    many = (ctypes.c_void_p * 65537)(*([FAKE] * 65537))
    many_sizes = (ctypes.c_uint64 * 65537)(*([40] * 65537))
    assert d(cast(many), cast(many_sizes), 65537, 16, 1.0, FAKE, 100, 0, FAKE, FAKE, 1 << 30,
             None) == dgc.EUNSUPPORTED


def test_l2_fetch_granularity_rejects_out_of_range(L):
    assert L.dgc_set_l2_fetch_granularity(-1) == dgc.EINVAL
    assert L.dgc_set_l2_fetch_granularity(129) == dgc.EINVAL


def _oracle_struct(name):
    import oracle
    return getattr(oracle, name)


@pytest.mark.parametrize("cname,py,header", [
    ("dgc_params", lambda: dgc.dgc_params, "include/dgc.h"),
    ("dgc_seg_stats", lambda: dgc.dgc_seg_stats, "include/dgc.h"),
    ("orc_params", lambda: _oracle_struct("Params"), "oracle/dgc_oracle.h"),
    ("orc_seg_stats", lambda: _oracle_struct("SegStats"), "oracle/dgc_oracle.h")])
def test_binding_structs_match_the_header(tmp_path, cname, py, header):
    # the C compiler's layout of the header's struct against the ctypes copy in the library's
    # binding (and in the oracle's test wrapper): the same size and every field at the same offset
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    py = py()
    inc, hname = os.path.split(os.path.join(ROOT, header))
    names = [f[0] for f in py._fields_]
    src = tmp_path / "layout.c"
    src.write_text(
        f'#include <stdio.h>\n#include <stddef.h>\n#include "{hname}"\nint main(void) {{\n'
        f'    printf("%zu\\n", sizeof({cname}));\n'
        + "".join(f'    printf("%zu\\n", offsetof({cname}, {n}));\n' for n in names)
        + "    return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", inc, str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(py)
    assert got[1:] == [getattr(py, n).offset for n in names]
