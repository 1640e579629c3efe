"""Python binding of libdgc, the GB300 (sm_103a) DGC gradient compressor.

Argument marshalling only: every function below has the name of a C entry point declared in
``include/dgc.h``, turns torch tensors into device pointers, passes the current CUDA stream, and
raises :class:`DGCError` when the C call returns a nonzero status. All arithmetic runs in the
CUDA kernels of ``libdgc.so``; there is no CPU path. If the library has not been built, loading
it fails with an error that says so (call :func:`build`).
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB, build

__all__ = [
    "DGCError", "build", "lib", "dgc_params", "dgc_seg_stats", "make_params",
    "dgc_compress_workspace", "dgc_compress_max_out", "dgc_compress", "dgc_compress_noalloc",
    "dgc_encode_max_bytes", "dgc_encode_workspace", "dgc_encode",
    "dgc_decode_workspace", "dgc_decode_accumulate", "dgc_decode_apply",
    "dgc_decode_workspace_bound", "dgc_decode_accumulate_dev", "dgc_decode_apply_dev",
    "dgc_encode_quant", "dgc_decode_workspace_quant", "dgc_decode_accumulate_quant",
    "dgc_decode_apply_quant", "dgc_compress_shared", "dgc_sum_shared_workspace",
    "dgc_sum_shared",
    "dgc_read_status", "dgc_status_string", "dgc_launch_count", "dgc_selftest_wait_timeout",
    "dgc_set_l2_fetch_granularity",
    "dgc_profile_stream_pass",
    "SELECT_EXACT", "SELECT_SAMPLED", "SELECT_ADACOMP", "FLAG_MASK_MOMENTUM",
]

OK, EINVAL, ECAPACITY, ECUDA, ETIMEOUT, ECORRUPT, EUNSUPPORTED = 0, -1, -2, -3, -4, -5, -6
SELECT_EXACT, SELECT_SAMPLED, SELECT_ADACOMP = 0, 1, 2
FLAG_MASK_MOMENTUM = 1


class dgc_params(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_uint32),
        ("flags", ctypes.c_uint32),
        ("sparsity", ctypes.c_double),
        ("momentum", ctypes.c_float),
        ("clip_norm", ctypes.c_float),
        ("sample_ratio", ctypes.c_double),
        ("reselect_factor", ctypes.c_double),
        ("seed", ctypes.c_uint64),
        ("bin_size", ctypes.c_uint32),
        ("leak", ctypes.c_float),
    ]


class dgc_seg_stats(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_uint64),
        ("candidates", ctypes.c_uint64),
        ("sent", ctypes.c_uint64),
        ("thresh_key", ctypes.c_uint32),
        ("sample_key", ctypes.c_uint32),
        ("reselected", ctypes.c_uint32),
        ("clip_scale", ctypes.c_float),
        ("clip_sumsq", ctypes.c_double),
    ]


STATS_BYTES = ctypes.sizeof(dgc_seg_stats)


class DGCError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {_status_text(code)} ({code})")


_lib = None


def lib():
    """The loaded libdgc.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"libdgc.so is not built ({LIB}); run "
                               "sparsified_gradient_compression_gb300.build()")
        L = ctypes.CDLL(LIB)
        i32, i64, u32, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        P = ctypes.POINTER
        L.dgc_compress_workspace.argtypes = [i64, i32, P(dgc_params), P(sz)]
        L.dgc_compress_max_out.argtypes = [i64, i32, P(dgc_params), P(i64)]
        L.dgc_compress.argtypes = [vp, vp, vp, i64, vp, i32, P(dgc_params), vp, vp, i64, vp, vp,
                                   vp, vp, sz, vp]
        L.dgc_compress_noalloc.argtypes = [vp, vp, vp, i64, vp, i32, P(dgc_params), vp, vp, i64,
                                           vp, vp, vp, vp]
        L.dgc_encode_max_bytes.argtypes = [i64, i64, P(u64)]
        L.dgc_encode_workspace.argtypes = [i64, P(sz)]
        L.dgc_encode.argtypes = [vp, vp, vp, i64, i64, vp, u64, vp, vp, vp, sz, vp]
        L.dgc_decode_workspace.argtypes = [i32, vp, i64, P(sz)]
        L.dgc_decode_accumulate.argtypes = [vp, vp, i32, vp, i64, i32, vp, vp, sz, vp]
        L.dgc_decode_apply.argtypes = [vp, vp, i32, vp, i64, ctypes.c_float, vp, vp, sz, vp]
        L.dgc_decode_workspace_bound.argtypes = [i32, vp, i64, P(sz)]
        L.dgc_decode_accumulate_dev.argtypes = [vp, vp, vp, i32, vp, i64, i32, vp, vp, sz, vp]
        L.dgc_decode_apply_dev.argtypes = [vp, vp, vp, i32, vp, i64, ctypes.c_float, vp, vp, sz,
                                           vp]
        f32 = ctypes.c_float
        L.dgc_encode_quant.argtypes = [vp, vp, vp, i64, i64, f32, i32, vp, vp, u64, vp, vp, vp,
                                       sz, vp]
        L.dgc_decode_workspace_quant.argtypes = [i32, vp, i64, i32, P(sz)]
        L.dgc_decode_accumulate_quant.argtypes = [vp, vp, i32, i32, f32, vp, i64, i32, vp, vp, sz,
                                                  vp]
        L.dgc_decode_apply_quant.argtypes = [vp, vp, i32, i32, f32, vp, i64, f32, vp, vp, sz, vp]
        L.dgc_compress_shared.argtypes = [vp, vp, vp, i64, vp, i32, P(dgc_params), vp, vp, i64,
                                          vp, vp, vp, sz, vp]
        L.dgc_sum_shared_workspace.argtypes = [i32, P(sz)]
        L.dgc_sum_shared.argtypes = [vp, i32, vp, i64, vp, vp, vp, sz, vp]
        L.dgc_read_status.argtypes = [vp, vp]
        L.dgc_status_string.argtypes = [ctypes.c_int]
        L.dgc_status_string.restype = ctypes.c_char_p
        L.dgc_launch_count.argtypes = []
        L.dgc_launch_count.restype = u64
        L.dgc_set_l2_fetch_granularity.argtypes = [i32]
        L.dgc_set_l2_fetch_granularity.restype = ctypes.c_int
        L.dgc_selftest_wait_timeout.argtypes = [vp, u32, vp]
        L.dgc_profile_stream_pass.argtypes = [vp, vp]
        L.dgc_profile_stream_pass.restype = None
        for f in ("dgc_compress_workspace", "dgc_compress_max_out", "dgc_compress",
                  "dgc_compress_noalloc",
                  "dgc_encode_max_bytes", "dgc_encode_workspace", "dgc_encode",
                  "dgc_decode_workspace", "dgc_decode_accumulate", "dgc_decode_apply",
                  "dgc_decode_workspace_bound", "dgc_decode_accumulate_dev",
                  "dgc_decode_apply_dev",
                  "dgc_encode_quant", "dgc_decode_workspace_quant",
                  "dgc_decode_accumulate_quant", "dgc_decode_apply_quant",
                  "dgc_compress_shared", "dgc_sum_shared_workspace", "dgc_sum_shared",
                  "dgc_read_status",
                  "dgc_selftest_wait_timeout"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _status_text(code: int) -> str:
    try:
        return lib().dgc_status_string(int(code)).decode()
    except Exception:  # the library itself failed to load
        return "status"


def _check(rc: int, where: str) -> int:
    if rc != OK:
        raise DGCError(rc, where)
    return rc


def _ptr(t) -> int | None:
    """Device (or host) address of a tensor, or an int address passed through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_params(mode=SELECT_EXACT, sparsity=0.999, momentum=0.9, clip_norm=0.0,
                mask_momentum=True, sample_ratio=0.01, reselect_factor=1.3, seed=0,
                bin_size=1000, leak=0.0) -> dgc_params:
    return dgc_params(int(mode), FLAG_MASK_MOMENTUM if mask_momentum else 0, float(sparsity),
                      float(momentum), float(clip_norm), float(sample_ratio),
                      float(reselect_factor), int(seed) & (2**64 - 1), int(bin_size),
                      float(leak))


# --------------------------------------------------------------------------- compressor
def dgc_compress_workspace(n: int, nseg: int, params: dgc_params) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().dgc_compress_workspace(int(n), int(nseg), ctypes.byref(params),
                                        ctypes.byref(out)), "dgc_compress_workspace")
    return out.value


def dgc_compress_max_out(n: int, nseg: int, params: dgc_params) -> int:
    out = ctypes.c_int64(0)
    _check(lib().dgc_compress_max_out(int(n), int(nseg), ctypes.byref(params), ctypes.byref(out)),
           "dgc_compress_max_out")
    return out.value


def dgc_compress(g, u, v, seg_off, params: dgc_params, out_idx, out_val, out_count, stats,
                 status, ws, n: int | None = None, out_cap: int | None = None,
                 ws_bytes: int | None = None, stream=None) -> int:
    """g, u, v: float32 CUDA tensors of n entries; seg_off: int64 CUDA tensor (nseg+1);
    out_idx (int32/uint32), out_val (float32): CUDA tensors of out_cap entries; out_count: int64
    CUDA tensor (1); stats: uint8 CUDA tensor of nseg * STATS_BYTES or None; status: int32 CUDA
    tensor (1); ws: uint8 CUDA tensor."""
    n = g.numel() if n is None else n
    nseg = seg_off.numel() - 1 if hasattr(seg_off, "numel") else None
    out_cap = out_idx.numel() if out_cap is None else out_cap
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    return _check(lib().dgc_compress(_ptr(g), _ptr(u), _ptr(v), int(n), _ptr(seg_off), int(nseg),
                                     ctypes.byref(params), _ptr(out_idx), _ptr(out_val),
                                     int(out_cap), _ptr(out_count), _ptr(stats), _ptr(status),
                                     _ptr(ws), int(ws_bytes), _stream(stream)), "dgc_compress")


def dgc_compress_noalloc(g, u, v, seg_off, params: dgc_params, out_idx, out_val, out_count,
                         stats, status, n: int | None = None, out_cap: int | None = None,
                         stream=None) -> int:
    """dgc_compress without a caller workspace, for callers that cannot allocate device memory
    (the library's own 16 MiB scratch per GPU; see include/dgc.h for the limit and rules)."""
    n = g.numel() if n is None else n
    nseg = seg_off.numel() - 1
    out_cap = out_idx.numel() if out_cap is None else out_cap
    return _check(lib().dgc_compress_noalloc(_ptr(g), _ptr(u), _ptr(v), int(n), _ptr(seg_off),
                                             int(nseg), ctypes.byref(params), _ptr(out_idx),
                                             _ptr(out_val), int(out_cap), _ptr(out_count),
                                             _ptr(stats), _ptr(status), _stream(stream)),
                  "dgc_compress_noalloc")


# -------------------------------------------------------------------------------- codec
def dgc_encode_max_bytes(max_count: int, n: int) -> int:
    out = ctypes.c_uint64(0)
    _check(lib().dgc_encode_max_bytes(int(max_count), int(n), ctypes.byref(out)),
           "dgc_encode_max_bytes")
    return out.value


def dgc_encode_workspace(max_count: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().dgc_encode_workspace(int(max_count), ctypes.byref(out)), "dgc_encode_workspace")
    return out.value


def dgc_encode(idx, val, count, n: int, out, out_bytes, status, ws, max_count: int | None = None,
               out_cap: int | None = None, ws_bytes: int | None = None, stream=None) -> int:
    max_count = idx.numel() if max_count is None else max_count
    out_cap = out.numel() * out.element_size() if out_cap is None else out_cap
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    return _check(lib().dgc_encode(_ptr(idx), _ptr(val), _ptr(count), int(max_count), int(n),
                                   _ptr(out), int(out_cap), _ptr(out_bytes), _ptr(status),
                                   _ptr(ws), int(ws_bytes), _stream(stream)), "dgc_encode")


def dgc_decode_workspace(stream_bytes, n: int) -> int:
    W = len(stream_bytes)
    arr = (ctypes.c_uint64 * max(W, 1))(*[int(b) for b in stream_bytes])
    out = ctypes.c_size_t(0)
    _check(lib().dgc_decode_workspace(W, ctypes.cast(arr, ctypes.c_void_p), int(n),
                                      ctypes.byref(out)), "dgc_decode_workspace")
    return out.value


def dgc_decode_accumulate(streams, stream_bytes, dense, n: int, accumulate: bool, status, ws,
                          ws_bytes: int | None = None, stream=None) -> int:
    """streams: list of device addresses or uint8 CUDA tensors; stream_bytes: list of sizes."""
    W = len(stream_bytes)
    ptrs = (ctypes.c_void_p * max(W, 1))(*[_ptr(s) for s in streams])
    sizes = (ctypes.c_uint64 * max(W, 1))(*[int(b) for b in stream_bytes])
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    return _check(lib().dgc_decode_accumulate(ctypes.cast(ptrs, ctypes.c_void_p),
                                              ctypes.cast(sizes, ctypes.c_void_p), W,
                                              _ptr(dense), int(n), int(bool(accumulate)),
                                              _ptr(status), _ptr(ws), int(ws_bytes),
                                              _stream(stream)), "dgc_decode_accumulate")


def dgc_decode_apply(streams, stream_bytes, w, n: int, lr: float, status, ws,
                     ws_bytes: int | None = None, stream=None) -> int:
    """w <- fma(-lr, ordered sum of the decoded messages, w); streams as for decode."""
    W = len(stream_bytes)
    ptrs = (ctypes.c_void_p * max(W, 1))(*[_ptr(s) for s in streams])
    sizes = (ctypes.c_uint64 * max(W, 1))(*[int(b) for b in stream_bytes])
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    return _check(lib().dgc_decode_apply(ctypes.cast(ptrs, ctypes.c_void_p),
                                         ctypes.cast(sizes, ctypes.c_void_p), W, _ptr(w), int(n),
                                         float(lr), _ptr(status), _ptr(ws), int(ws_bytes),
                                         _stream(stream)), "dgc_decode_apply")


def dgc_decode_workspace_bound(max_bytes, n: int) -> int:
    """Workspace of the _dev decoders for W messages of at most max_bytes[w] bytes each."""
    W = len(max_bytes)
    arr = (ctypes.c_uint64 * max(W, 1))(*[int(b) for b in max_bytes])
    out = ctypes.c_size_t(0)
    _check(lib().dgc_decode_workspace_bound(W, ctypes.cast(arr, ctypes.c_void_p), int(n),
                                            ctypes.byref(out)), "dgc_decode_workspace_bound")
    return out.value


def dgc_decode_accumulate_dev(streams, stream_bytes, max_bytes, dense, n: int, accumulate: bool,
                              status, ws, ws_bytes: int | None = None, stream=None) -> int:
    """streams: device addresses or uint8 CUDA tensors; stream_bytes: a CUDA tensor of W 8-byte
    sizes (int64 or uint64, e.g. dgc_encode's out_bytes); max_bytes: host bounds on them."""
    W = len(max_bytes)
    ptrs = (ctypes.c_void_p * max(W, 1))(*[_ptr(s) for s in streams])
    bounds = (ctypes.c_uint64 * max(W, 1))(*[int(b) for b in max_bytes])
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    return _check(lib().dgc_decode_accumulate_dev(
        ctypes.cast(ptrs, ctypes.c_void_p), _ptr(stream_bytes), ctypes.cast(bounds, ctypes.c_void_p),
        W, _ptr(dense), int(n), 1 if accumulate else 0, _ptr(status), _ptr(ws), int(ws_bytes),
        _stream(stream)), "dgc_decode_accumulate_dev")


def dgc_decode_apply_dev(streams, stream_bytes, max_bytes, w, n: int, lr: float, status, ws,
                         ws_bytes: int | None = None, stream=None) -> int:
    """dgc_decode_apply with the message sizes in device memory (see dgc_decode_accumulate_dev)."""
    W = len(max_bytes)
    ptrs = (ctypes.c_void_p * max(W, 1))(*[_ptr(s) for s in streams])
    bounds = (ctypes.c_uint64 * max(W, 1))(*[int(b) for b in max_bytes])
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    return _check(lib().dgc_decode_apply_dev(
        ctypes.cast(ptrs, ctypes.c_void_p), _ptr(stream_bytes), ctypes.cast(bounds, ctypes.c_void_p),
        W, _ptr(w), int(n), float(lr), _ptr(status), _ptr(ws), int(ws_bytes), _stream(stream)),
        "dgc_decode_apply_dev")


def dgc_encode_quant(idx, val, count, n: int, alpha: float, bits: int, v, out, out_bytes, status,
                     ws, max_count: int | None = None, out_cap: int | None = None,
                     ws_bytes: int | None = None, stream=None) -> int:
    """Version-2 message of `bits`-bit integers; v (or None) takes back each remainder."""
    max_count = idx.numel() if max_count is None else max_count
    out_cap = out.numel() * out.element_size() if out_cap is None else out_cap
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    return _check(lib().dgc_encode_quant(_ptr(idx), _ptr(val), _ptr(count), int(max_count),
                                         int(n), float(alpha), int(bits),
                                         None if v is None else _ptr(v), _ptr(out), int(out_cap),
                                         _ptr(out_bytes), _ptr(status), _ptr(ws), int(ws_bytes),
                                         _stream(stream)), "dgc_encode_quant")


def dgc_decode_workspace_quant(stream_bytes, n: int, bits: int) -> int:
    W = len(stream_bytes)
    arr = (ctypes.c_uint64 * max(W, 1))(*[int(b) for b in stream_bytes])
    out = ctypes.c_size_t(0)
    _check(lib().dgc_decode_workspace_quant(W, ctypes.cast(arr, ctypes.c_void_p), int(n),
                                            int(bits), ctypes.byref(out)),
           "dgc_decode_workspace_quant")
    return out.value


def dgc_decode_accumulate_quant(streams, stream_bytes, bits: int, alpha: float, dense, n: int,
                                accumulate: bool, status, ws, ws_bytes: int | None = None,
                                stream=None) -> int:
    W = len(stream_bytes)
    ptrs = (ctypes.c_void_p * max(W, 1))(*[_ptr(s) for s in streams])
    sizes = (ctypes.c_uint64 * max(W, 1))(*[int(b) for b in stream_bytes])
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    return _check(lib().dgc_decode_accumulate_quant(
        ctypes.cast(ptrs, ctypes.c_void_p), ctypes.cast(sizes, ctypes.c_void_p), W, int(bits),
        float(alpha), _ptr(dense), int(n), int(bool(accumulate)), _ptr(status), _ptr(ws),
        int(ws_bytes), _stream(stream)), "dgc_decode_accumulate_quant")


def dgc_decode_apply_quant(streams, stream_bytes, bits: int, alpha: float, w, n: int, lr: float,
                           status, ws, ws_bytes: int | None = None, stream=None) -> int:
    W = len(stream_bytes)
    ptrs = (ctypes.c_void_p * max(W, 1))(*[_ptr(s) for s in streams])
    sizes = (ctypes.c_uint64 * max(W, 1))(*[int(b) for b in stream_bytes])
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    return _check(lib().dgc_decode_apply_quant(
        ctypes.cast(ptrs, ctypes.c_void_p), ctypes.cast(sizes, ctypes.c_void_p), W, int(bits),
        float(alpha), _ptr(w), int(n), float(lr), _ptr(status), _ptr(ws), int(ws_bytes),
        _stream(stream)), "dgc_decode_apply_quant")


def dgc_compress_shared(g, u, v, seg_off, params: dgc_params, idx, count, out_val, status, ws,
                        n: int | None = None, max_count: int | None = None,
                        ws_bytes: int | None = None, stream=None) -> int:
    """One learner's step at a shared index set idx (device, ascending), count device int64."""
    n = g.numel() if n is None else n
    nseg = seg_off.numel() - 1
    max_count = idx.numel() if max_count is None else max_count
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    return _check(lib().dgc_compress_shared(_ptr(g), _ptr(u), _ptr(v), int(n), _ptr(seg_off),
                                            int(nseg), ctypes.byref(params), _ptr(idx),
                                            _ptr(count), int(max_count), _ptr(out_val),
                                            _ptr(status), _ptr(ws), int(ws_bytes),
                                            _stream(stream)), "dgc_compress_shared")


def dgc_sum_shared_workspace(W: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().dgc_sum_shared_workspace(int(W), ctypes.byref(out)), "dgc_sum_shared_workspace")
    return out.value


def dgc_sum_shared(vals, count, max_count: int, out, status, ws, ws_bytes: int | None = None,
                   stream=None) -> int:
    """vals: list of device addresses or float32 CUDA tensors (the learners, in order)."""
    W = len(vals)
    ptrs = (ctypes.c_void_p * max(W, 1))(*[_ptr(x) for x in vals])
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    return _check(lib().dgc_sum_shared(ctypes.cast(ptrs, ctypes.c_void_p), W, _ptr(count),
                                       int(max_count), _ptr(out), _ptr(status), _ptr(ws),
                                       int(ws_bytes), _stream(stream)), "dgc_sum_shared")


# ----------------------------------------------------------------------------- utilities
def dgc_read_status(status, stream=None) -> int:
    return int(lib().dgc_read_status(_ptr(status), _stream(stream)))


def dgc_status_string(code: int) -> str:
    return lib().dgc_status_string(int(code)).decode()


def dgc_launch_count() -> int:
    return int(lib().dgc_launch_count())


def dgc_set_l2_fetch_granularity(nbytes: int) -> int:
    """Context limit cudaLimitMaxL2FetchGranularity for the current device (0..128 bytes)."""
    return _check(lib().dgc_set_l2_fetch_granularity(int(nbytes)), "dgc_set_l2_fetch_granularity")


def dgc_profile_stream_pass(begin, end) -> None:
    """begin/end: torch.cuda.Event objects (created with enable_timing=True), or None."""
    handles = []
    for ev in (begin, end):
        if ev is None:
            handles.append(None)
            continue
        if not ev.cuda_event:  # torch creates the CUDA event on its first record
            ev.record()
        handles.append(ev.cuda_event)
    lib().dgc_profile_stream_pass(*handles)


def dgc_selftest_wait_timeout(status, spin_limit: int, stream=None) -> int:
    return _check(lib().dgc_selftest_wait_timeout(_ptr(status), int(spin_limit), _stream(stream)),
                  "dgc_selftest_wait_timeout")
