"""The oracle: a plain single-threaded CPU restatement of the DGC compressor, codec and decoder.

TEST INFRASTRUCTURE ONLY. The test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` are its only users; the product library never imports it and shares no code
with it. This module compiles ``dgc_oracle.c`` with gcc (once, next to the source) and wraps
it with ctypes and numpy.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dgc_oracle.c")
_HDR = os.path.join(_HERE, "dgc_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

EXACT, SAMPLED, ADACOMP = 0, 1, 2
MASK_MOMENTUM = 1
OK, EINVAL, ECAPACITY, ECORRUPT, EUNSUPPORTED, ENOMEM = 0, -1, -2, -5, -6, -7


class Params(ctypes.Structure):
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


class SegStats(ctypes.Structure):
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


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no fast-math, no FMA contraction)."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or max(
            os.path.getmtime(_SRC), os.path.getmtime(_HDR)) > os.path.getmtime(_LIB)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call([
                "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-Wall",
                "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        path = os.environ.get("DGC_ORACLE_LIB")  # a mutated copy, for checking the pins
        if not path:
            path = build()
        L = ctypes.CDLL(path)
        u64, i64, i32, u32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
        vp = ctypes.c_void_p
        L.orc_ppb.restype = u64
        L.orc_ppb.argtypes = [ctypes.c_double]
        L.orc_count.restype = u64
        L.orc_count.argtypes = [u64, u64]
        L.orc_mix64.restype = u64
        L.orc_mix64.argtypes = [u64]
        L.orc_sample_position.restype = u64
        L.orc_sample_position.argtypes = [u64, u32, u64, u64]
        L.orc_sumsq.restype = ctypes.c_double
        L.orc_sumsq.argtypes = [vp, i64]
        L.orc_clip_scale.restype = ctypes.c_float
        L.orc_clip_scale.argtypes = [vp, i64, ctypes.c_float, ctypes.POINTER(ctypes.c_int)]
        L.orc_accumulate_one.restype = None
        L.orc_accumulate_one.argtypes = [ctypes.c_float] * 5 + [
            ctypes.c_int, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]
        L.orc_accumulate_leak.restype = None
        L.orc_accumulate_leak.argtypes = [ctypes.c_float] * 5 + [
            ctypes.c_int, ctypes.c_float, ctypes.POINTER(ctypes.c_float),
            ctypes.POINTER(ctypes.c_float)]
        L.orc_compress_shared.restype = ctypes.c_int
        L.orc_compress_shared.argtypes = [vp, vp, vp, i64, vp, i32, ctypes.POINTER(Params), vp,
                                          i64, vp]
        L.orc_sum_shared.restype = ctypes.c_int
        L.orc_sum_shared.argtypes = [vp, i32, i64, vp]
        L.orc_topk.restype = ctypes.c_int
        L.orc_topk.argtypes = [vp, vp, i64, i64, vp]
        L.orc_bin_select.restype = None
        L.orc_bin_select.argtypes = [vp, i64, u32, vp]
        L.orc_compress.restype = ctypes.c_int
        L.orc_compress.argtypes = [vp, vp, vp, i64, vp, i32, ctypes.POINTER(Params),
                                   vp, vp, i64, ctypes.POINTER(i64), vp]
        L.orc_encoded_size.restype = u64
        L.orc_encoded_size.argtypes = [vp, i64]
        L.orc_encode.restype = ctypes.c_int
        L.orc_encode.argtypes = [vp, vp, i64, i64, vp, u64, ctypes.POINTER(u64)]
        L.orc_decode_accumulate.restype = ctypes.c_int
        L.orc_decode_accumulate.argtypes = [vp, vp, i32, vp, i64, ctypes.c_int]
        L.orc_decode_apply.restype = ctypes.c_int
        L.orc_decode_apply.argtypes = [vp, vp, i32, vp, i64, ctypes.c_float]
        f32 = ctypes.c_float
        L.orc_encode_quant.restype = ctypes.c_int
        L.orc_encode_quant.argtypes = [vp, vp, i64, i64, f32, ctypes.c_int, vp, vp,
                                       ctypes.c_uint64, vp]
        L.orc_decode_accumulate_quant.restype = ctypes.c_int
        L.orc_decode_accumulate_quant.argtypes = [vp, vp, i32, ctypes.c_int, f32, vp, i64,
                                                  ctypes.c_int]
        L.orc_decode_apply_quant.restype = ctypes.c_int
        L.orc_decode_apply_quant.argtypes = [vp, vp, i32, ctypes.c_int, f32, vp, i64, f32]
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def make_params(mode=EXACT, sparsity=0.999, momentum=0.9, clip_norm=0.0, mask_momentum=True,
                sample_ratio=0.01, reselect_factor=1.3, seed=0, bin_size=1000,
                leak=0.0) -> Params:
    return Params(mode, MASK_MOMENTUM if mask_momentum else 0, float(sparsity),
                  float(momentum), float(clip_norm), float(sample_ratio),
                  float(reselect_factor), int(seed) & (2**64 - 1), int(bin_size), float(leak))


def ppb(fraction: float) -> int:
    return int(lib().orc_ppb(float(fraction)))


def count(n: int, ppb_: int) -> int:
    return int(lib().orc_count(int(n), int(ppb_)))


def mix64(z: int) -> int:
    return int(lib().orc_mix64(int(z) & (2**64 - 1)))


def sample_position(seed: int, segment: int, j: int, n_s: int) -> int:
    return int(lib().orc_sample_position(int(seed) & (2**64 - 1), int(segment), int(j), int(n_s)))


def sumsq(g: np.ndarray) -> float:
    g = np.ascontiguousarray(g, dtype=np.float32)
    return float(lib().orc_sumsq(_ptr(g), g.size))


def clip_scale(g: np.ndarray, clip_norm: float):
    g = np.ascontiguousarray(g, dtype=np.float32)
    clipped = ctypes.c_int(0)
    s = lib().orc_clip_scale(_ptr(g), g.size, float(clip_norm), ctypes.byref(clipped))
    return np.float32(s), bool(clipped.value)


def accumulate_one(g, u, v, momentum, scale=1.0, clipped=False):
    uo, vo = ctypes.c_float(), ctypes.c_float()
    lib().orc_accumulate_one(float(g), float(u), float(v), float(momentum), float(scale),
                             int(bool(clipped)), ctypes.byref(uo), ctypes.byref(vo))
    return np.float32(uo.value), np.float32(vo.value)


def accumulate_leak(g, u, v, momentum, leak, scale=1.0, clipped=False):
    uo, vo = ctypes.c_float(), ctypes.c_float()
    lib().orc_accumulate_leak(float(g), float(u), float(v), float(momentum), float(scale),
                              int(bool(clipped)), float(leak), ctypes.byref(uo), ctypes.byref(vo))
    return np.float32(uo.value), np.float32(vo.value)


def topk(v: np.ndarray, cand: np.ndarray, k: int) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    cand = np.ascontiguousarray(cand, dtype=np.uint32)
    sel = np.zeros(v.size, dtype=np.uint8)
    rc = lib().orc_topk(_ptr(v), _ptr(cand), cand.size, int(k), _ptr(sel))
    if rc != OK:
        raise RuntimeError(f"orc_topk failed: {rc}")
    return sel


def bin_select(v: np.ndarray, bin_size: int) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    sel = np.zeros(max(v.size, 1), dtype=np.uint8)
    lib().orc_bin_select(_ptr(v), v.size, int(bin_size), _ptr(sel))
    return sel[: v.size]


def max_out(n: int) -> int:
    return max(int(n), 1)


def compress(g, u, v, seg_off, params: Params):
    """One compressor step. u and v (float32 numpy arrays) are updated in place.

    Returns (idx uint32[count], val float32[count], stats list of dicts)."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    assert u.dtype == np.float32 and v.dtype == np.float32
    assert u.flags.c_contiguous and v.flags.c_contiguous
    seg_off = np.ascontiguousarray(seg_off, dtype=np.int64)
    nseg = seg_off.size - 1
    n = g.size
    cap = max_out(n)
    out_idx = np.empty(cap, np.uint32)
    out_val = np.empty(cap, np.float32)
    cnt = ctypes.c_int64(0)
    stats = (SegStats * nseg)()
    rc = lib().orc_compress(_ptr(g), _ptr(u), _ptr(v), n, _ptr(seg_off), nseg,
                            ctypes.byref(params), _ptr(out_idx), _ptr(out_val), cap,
                            ctypes.byref(cnt), ctypes.cast(stats, ctypes.c_void_p))
    if rc != OK:
        raise RuntimeError(f"orc_compress failed: {rc}")
    c = cnt.value
    st = [dict(k=s.k, candidates=s.candidates, sent=s.sent, thresh_key=s.thresh_key,
               sample_key=s.sample_key, reselected=s.reselected,
               clip_scale=np.float32(s.clip_scale), clip_sumsq=float(s.clip_sumsq))
          for s in stats]
    return out_idx[:c].copy(), out_val[:c].copy(), st


def encode(idx, val, n: int) -> bytes:
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    val = np.ascontiguousarray(val, dtype=np.float32)
    size = int(lib().orc_encoded_size(_ptr(idx), idx.size))
    out = np.zeros(max(size, 1), np.uint8)
    nb = ctypes.c_uint64(0)
    rc = lib().orc_encode(_ptr(idx), _ptr(val), idx.size, int(n), _ptr(out), out.size,
                          ctypes.byref(nb))
    if rc != OK:
        raise RuntimeError(f"orc_encode failed: {rc}")
    return out[: nb.value].tobytes()


def decode_accumulate(streams, n: int, dense=None, accumulate=False):
    """Decode and sum the messages in order. Returns (rc, dense)."""
    bufs = [np.frombuffer(s, dtype=np.uint8) if len(s) else np.zeros(1, np.uint8)
            for s in streams]
    W = len(bufs)
    ptrs = (ctypes.c_void_p * max(W, 1))(*[b.ctypes.data for b in bufs])
    sizes = (ctypes.c_uint64 * max(W, 1))(*[len(s) for s in streams])
    if dense is None:
        dense = np.zeros(n, np.float32)
    else:
        dense = np.ascontiguousarray(dense, dtype=np.float32).copy()
    rc = lib().orc_decode_accumulate(ctypes.cast(ptrs, ctypes.c_void_p),
                                     ctypes.cast(sizes, ctypes.c_void_p), W,
                                     _ptr(dense) if n else None, int(n), int(bool(accumulate)))
    return rc, dense


def decode_apply(streams, n: int, w, lr: float):
    """Decode and sum the messages in order, then w <- fmaf(-lr, sum, w). Returns (rc, w)."""
    bufs = [np.frombuffer(s, dtype=np.uint8) if len(s) else np.zeros(1, np.uint8)
            for s in streams]
    W = len(bufs)
    ptrs = (ctypes.c_void_p * max(W, 1))(*[b.ctypes.data for b in bufs])
    sizes = (ctypes.c_uint64 * max(W, 1))(*[len(s) for s in streams])
    w = np.ascontiguousarray(w, dtype=np.float32).copy()
    rc = lib().orc_decode_apply(ctypes.cast(ptrs, ctypes.c_void_p),
                                ctypes.cast(sizes, ctypes.c_void_p), W,
                                _ptr(w) if n else None, int(n), float(lr))
    return rc, w


def encode_quant(idx, val, n: int, alpha: float, bits: int, v=None):
    """Integer-valued message (version 2). Returns (rc, message bytes, residual v after the
    quantizer put each sent entry's remainder back), v being a copy of the given array."""
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    val = np.ascontiguousarray(val, dtype=np.float32)
    vv = None if v is None else np.ascontiguousarray(v, dtype=np.float32).copy()
    cap = 40 + 6 * (idx.size + int(n) // 65535 + 1)
    out = np.zeros(cap, np.uint8)
    nb = ctypes.c_uint64(0)
    rc = lib().orc_encode_quant(_ptr(idx), _ptr(val), idx.size, int(n), float(alpha), int(bits),
                                None if vv is None else _ptr(vv), _ptr(out), out.size,
                                ctypes.byref(nb))
    return rc, (out[: nb.value].tobytes() if rc == OK else b""), vv


def _streams(streams):
    bufs = [np.frombuffer(s, dtype=np.uint8) if len(s) else np.zeros(1, np.uint8)
            for s in streams]
    W = len(bufs)
    ptrs = (ctypes.c_void_p * max(W, 1))(*[b.ctypes.data for b in bufs])
    sizes = (ctypes.c_uint64 * max(W, 1))(*[len(s) for s in streams])
    return bufs, W, ctypes.cast(ptrs, ctypes.c_void_p), ctypes.cast(sizes, ctypes.c_void_p)


def decode_accumulate_quant(streams, n: int, bits: int, alpha: float, dense=None,
                            accumulate=False):
    """Sum version-2 messages of `bits`-bit values exactly in integers, divide by alpha once.
    Returns (rc, dense)."""
    bufs, W, ptrs, sizes = _streams(streams)
    dense = (np.zeros(n, np.float32) if dense is None
             else np.ascontiguousarray(dense, dtype=np.float32).copy())
    rc = lib().orc_decode_accumulate_quant(ptrs, sizes, W, int(bits), float(alpha),
                                           _ptr(dense) if n else None, int(n),
                                           int(bool(accumulate)))
    return rc, dense


def decode_apply_quant(streams, n: int, bits: int, alpha: float, w, lr: float):
    """w <- fmaf(-lr, (float)S / alpha, w) for version-2 messages. Returns (rc, w)."""
    bufs, W, ptrs, sizes = _streams(streams)
    w = np.ascontiguousarray(w, dtype=np.float32).copy()
    rc = lib().orc_decode_apply_quant(ptrs, sizes, W, int(bits), float(alpha),
                                      _ptr(w) if n else None,
                                      int(n), float(lr))
    return rc, w


def compress_shared(g, u, v, seg_off, params: Params, idx):
    """One step at the shared index set idx; u and v are updated in place. Returns (rc, values)."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    assert u.dtype == np.float32 and v.dtype == np.float32
    seg_off = np.ascontiguousarray(seg_off, dtype=np.int64)
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    out = np.zeros(max(idx.size, 1), np.float32)
    rc = lib().orc_compress_shared(_ptr(g), _ptr(u), _ptr(v), g.size, _ptr(seg_off),
                                   seg_off.size - 1, ctypes.byref(params), _ptr(idx), idx.size,
                                   _ptr(out))
    return rc, out[: idx.size].copy()


def sum_shared(vals):
    """Learner-ordered binary32 sum of equal-length value vectors. Returns (rc, sum)."""
    arrs = [np.ascontiguousarray(a, dtype=np.float32) for a in vals]
    count = arrs[0].size if arrs else 0
    ptrs = (ctypes.c_void_p * max(len(arrs), 1))(*[a.ctypes.data for a in arrs])
    out = np.zeros(max(count, 1), np.float32)
    rc = lib().orc_sum_shared(ctypes.cast(ptrs, ctypes.c_void_p), len(arrs), count, _ptr(out))
    return rc, out[:count].copy()
