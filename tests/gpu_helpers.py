"""Buffers and calls for driving libdgc from the tests (torch only allocates and copies)."""
from __future__ import annotations

import numpy as np
import torch

import sparsified_gradient_compression_gb300 as dgc

STATS_DTYPE = np.dtype([("k", "<u8"), ("candidates", "<u8"), ("sent", "<u8"),
                        ("thresh_key", "<u4"), ("sample_key", "<u4"), ("reselected", "<u4"),
                        ("clip_scale", "<f4"), ("clip_sumsq", "<f8")])
assert STATS_DTYPE.itemsize == dgc.STATS_BYTES


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.float32, copy=False)


class Compressor:
    """Owns the workspace and outputs of dgc_compress for one (n, segments, params) shape."""

    def __init__(self, n: int, seg_off, params: dgc.dgc_params):
        self.n = int(n)
        seg = np.asarray(seg_off, dtype=np.int64)
        self.nseg = seg.size - 1
        self.params = params
        self.seg_off = torch.from_numpy(seg).cuda()
        self.ws_bytes = dgc.dgc_compress_workspace(self.n, self.nseg, params)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device="cuda")
        self.cap = dgc.dgc_compress_max_out(self.n, self.nseg, params)
        self.out_idx = torch.empty(max(self.cap, 1), dtype=torch.int32, device="cuda")
        self.out_val = torch.empty(max(self.cap, 1), dtype=torch.float32, device="cuda")
        self.out_count = torch.zeros(1, dtype=torch.int64, device="cuda")
        self.stats = torch.zeros(self.nseg * dgc.STATS_BYTES, dtype=torch.uint8, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def __call__(self, g: torch.Tensor, u: torch.Tensor, v: torch.Tensor):
        dgc.dgc_compress(g, u, v, self.seg_off, self.params, self.out_idx, self.out_val,
                         self.out_count, self.stats, self.status, self.ws, n=self.n,
                         out_cap=self.cap, ws_bytes=self.ws_bytes)

    def status_code(self) -> int:
        return dgc.dgc_read_status(self.status)

    def results(self):
        torch.cuda.synchronize()
        c = int(self.out_count.item())
        idx = self.out_idx[:c].cpu().numpy().view(np.uint32).copy()
        val = self.out_val[:c].cpu().numpy().copy()
        st = np.frombuffer(self.stats.cpu().numpy().tobytes(), dtype=STATS_DTYPE)
        return idx, val, st


class Encoder:
    def __init__(self, max_count: int, n: int):
        self.max_count, self.n = int(max_count), int(n)
        self.cap = dgc.dgc_encode_max_bytes(self.max_count, self.n)
        self.out = torch.zeros(self.cap + 16, dtype=torch.uint8, device="cuda")
        self.out_bytes = torch.zeros(1, dtype=torch.int64, device="cuda")
        self.ws_bytes = dgc.dgc_encode_workspace(self.max_count)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def __call__(self, idx: torch.Tensor, val: torch.Tensor, count: torch.Tensor):
        dgc.dgc_encode(idx, val, count, self.n, self.out, self.out_bytes, self.status, self.ws,
                       max_count=self.max_count, out_cap=self.cap, ws_bytes=self.ws_bytes)

    def message(self) -> bytes:
        torch.cuda.synchronize()
        nb = int(self.out_bytes.item())
        return self.out[:nb].cpu().numpy().tobytes()


def decode(messages, n: int, dense: torch.Tensor | None = None, accumulate=False):
    """Decode host byte strings on the GPU; returns (status, dense tensor)."""
    bufs = []
    for m in messages:
        t = torch.zeros(max(len(m), 16) + 16, dtype=torch.uint8, device="cuda")
        if len(m):
            t[: len(m)] = torch.frombuffer(bytearray(m), dtype=torch.uint8).cuda()
        bufs.append(t)
    sizes = [len(m) for m in messages]
    ws_bytes = dgc.dgc_decode_workspace(sizes, n)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    if dense is None:
        dense = torch.full((max(n, 1),), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dgc.dgc_decode_accumulate(bufs, sizes, dense, n, accumulate, status, ws, ws_bytes=ws_bytes)
    return dgc.dgc_read_status(status), dense


def decode_apply(messages, n: int, w: np.ndarray, lr: float):
    """w <- fma(-lr, ordered sum of the messages, w) on the GPU; returns (status, w on host)."""
    bufs = []
    for m in messages:
        t = torch.zeros(max(len(m), 16) + 16, dtype=torch.uint8, device="cuda")
        if len(m):
            t[: len(m)] = torch.frombuffer(bytearray(m), dtype=torch.uint8).cuda()
        bufs.append(t)
    sizes = [len(m) for m in messages]
    ws_bytes = dgc.dgc_decode_workspace(sizes, n)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    wd = dev_f32(w) if n else torch.zeros(1, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dgc.dgc_decode_apply(bufs, sizes, wd, n, lr, status, ws, ws_bytes=ws_bytes)
    return dgc.dgc_read_status(status), host_f32(wd)[:n]


def encode_quant(idx: np.ndarray, val: np.ndarray, n: int, alpha: float, bits: int,
                 v: np.ndarray | None = None):
    """Version-2 message on the GPU; returns (status, message bytes, residual v on host or None)."""
    k = idx.size
    enc = Encoder(max(k, 1), n)
    d_idx = torch.from_numpy(np.append(idx, np.uint32(0)).astype(np.uint32).view(np.int32)).cuda()
    d_val = dev_f32(np.append(val, np.float32(0)))
    d_v = None if v is None else dev_f32(v)
    dgc.dgc_encode_quant(d_idx, d_val, torch.tensor([k], dtype=torch.int64, device="cuda"), n,
                         alpha, bits, d_v, enc.out, enc.out_bytes, enc.status, enc.ws,
                         max_count=enc.max_count, out_cap=enc.cap, ws_bytes=enc.ws_bytes)
    rc = dgc.dgc_read_status(enc.status)
    return rc, (enc.message() if rc == 0 else b""), (None if d_v is None else host_f32(d_v))


def _device_messages(messages):
    bufs = []
    for m in messages:
        t = torch.zeros(max(len(m), 16) + 16, dtype=torch.uint8, device="cuda")
        if len(m):
            t[: len(m)] = torch.frombuffer(bytearray(m), dtype=torch.uint8).cuda()
        bufs.append(t)
    return bufs, [len(m) for m in messages]


def decode_quant(messages, n: int, bits: int, alpha: float, dense: np.ndarray | None = None,
                 accumulate=False):
    """Version-2 decode on the GPU; returns (status, dense on host)."""
    bufs, sizes = _device_messages(messages)
    ws_bytes = dgc.dgc_decode_workspace_quant(sizes, n, bits)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    d = (torch.full((max(n, 1),), float("nan"), dtype=torch.float32, device="cuda")
         if dense is None else dev_f32(dense))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dgc.dgc_decode_accumulate_quant(bufs, sizes, bits, alpha, d, n, accumulate, status, ws,
                                    ws_bytes=ws_bytes)
    return dgc.dgc_read_status(status), host_f32(d)[:n]


def decode_apply_quant(messages, n: int, bits: int, alpha: float, w: np.ndarray, lr: float):
    bufs, sizes = _device_messages(messages)
    ws_bytes = dgc.dgc_decode_workspace_quant(sizes, n, bits)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    wd = dev_f32(w) if n else torch.zeros(1, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dgc.dgc_decode_apply_quant(bufs, sizes, bits, alpha, wd, n, lr, status, ws, ws_bytes=ws_bytes)
    return dgc.dgc_read_status(status), host_f32(wd)[:n]
