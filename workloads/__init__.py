"""Seeded synthetic inputs shaped like the DGC review's workloads.

Both the CUDA path (tests, bench) and the oracle take their inputs from here; this module holds
none of the compressor's arithmetic, only random gradients and the segment layouts they come in.
Every array is a deterministic function of (workload, step, tensor/learner, chunk): a chunk of
2^22 entries is drawn from its own numpy PCG64 stream, so the values do not depend on how many
threads draw them.

Workloads (stand-ins for the ImageNet/ResNet-50 and LibriSpeech/DeepSpeech models of the DGC
review, whose datasets and weights are not used):
  single     -- one tensor of 1,048,576 entries, g ~ N(0, 0.01^2)
  resnet50   -- 161 tensors with ResNet-50's parameter shapes (25,557,032 entries, ~97 MB),
                tensor t drawn from N(0, s_t^2) with s_t = 10^(-4 + 3U) fixed per tensor
  deepspeech -- flat bucket of 122,000,000 entries (~488 MB): 5 segments of 24,000,000 and one
                of 2,000,000; g = 1e-3 * Student-t(3)
  bucket1g   -- flat bucket of 2^30 entries (4 GiB): g ~ N(0, 1e-4) (variance) with
                round(1e-4 * n) fixed positions multiplied by 100
  learners   -- W independent learners of 25,557,032 entries each, g ~ N(0, 0.01^2)
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 22
_IDS = {"single": 1, "resnet50": 2, "deepspeech": 3, "bucket1g": 4, "learners": 5, "misc": 9}


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _fill(out: np.ndarray, words, draw) -> np.ndarray:
    n = out.size
    nchunks = (n + CHUNK - 1) // CHUNK

    def work(c):
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(words) + [c])))
        draw(rng, out[lo:hi])

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(min(_threads(), nchunks)) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def normal(words, n: int, sigma: float, out: np.ndarray | None = None) -> np.ndarray:
    """n float32 draws of sigma * N(0, 1) (the product rounded to float32)."""
    out = np.empty(n, np.float32) if out is None else out
    s = np.float32(sigma)

    def draw(rng, o):
        rng.standard_normal(out=o, dtype=np.float32)
        o *= s

    return _fill(out, words, draw)


def student_t(words, n: int, df: float, scale: float, out=None) -> np.ndarray:
    out = np.empty(n, np.float32) if out is None else out

    def draw(rng, o):
        o[:] = (rng.standard_t(df, size=o.size) * scale).astype(np.float32)

    return _fill(out, words, draw)


# ---------------------------------------------------------------- ResNet-50 parameter shapes
def resnet50_shapes():
    """(name, shape) of ResNet-50's 161 parameter tensors in definition order: stem conv + BN,
    bottleneck stages of [3, 4, 6, 3] blocks with widths 64/128/256/512 (x4 expansion, a
    1x1 conv + BN downsample on each stage's first block), then the 1000-way classifier."""
    shapes = [("conv1.weight", (64, 3, 7, 7)), ("bn1.weight", (64,)), ("bn1.bias", (64,))]
    inplanes = 64
    for li, (blocks, width) in enumerate(zip([3, 4, 6, 3], [64, 128, 256, 512]), start=1):
        for b in range(blocks):
            p = f"layer{li}.{b}."
            out = width * 4
            shapes += [(p + "conv1.weight", (width, inplanes, 1, 1)),
                       (p + "bn1.weight", (width,)), (p + "bn1.bias", (width,)),
                       (p + "conv2.weight", (width, width, 3, 3)),
                       (p + "bn2.weight", (width,)), (p + "bn2.bias", (width,)),
                       (p + "conv3.weight", (out, width, 1, 1)),
                       (p + "bn3.weight", (out,)), (p + "bn3.bias", (out,))]
            if b == 0:
                shapes += [(p + "downsample.0.weight", (out, inplanes, 1, 1)),
                           (p + "downsample.1.weight", (out,)),
                           (p + "downsample.1.bias", (out,))]
            inplanes = out
    shapes += [("fc.weight", (1000, 2048)), ("fc.bias", (1000,))]
    return shapes


def segments_from_sizes(sizes) -> np.ndarray:
    off = np.zeros(len(sizes) + 1, np.int64)
    off[1:] = np.cumsum(np.asarray(sizes, dtype=np.int64))
    return off


def resnet50_segments() -> np.ndarray:
    return segments_from_sizes([math.prod(s) for _, s in resnet50_shapes()])


def resnet50_sigmas(seed: int = 0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([_IDS["resnet50"], seed,
                                                                      0xA11CE])))
    return (10.0 ** (-4.0 + 3.0 * rng.random(161))).astype(np.float64)


def deepspeech_segments() -> np.ndarray:
    return segments_from_sizes([24_000_000] * 5 + [2_000_000])


# ------------------------------------------------------------------------- per-step gradients
def gradient(workload: str, step: int, seed: int = 0, learner: int = 0, n: int | None = None,
             out: np.ndarray | None = None) -> np.ndarray:
    """The fresh float32 gradient of `workload` at `step` (and `learner`)."""
    wid = _IDS[workload]
    if workload == "single":
        return normal([wid, seed, step, 0], n or 1_048_576, 0.01, out)
    if workload == "learners":
        return normal([wid, seed, step, learner], n or 25_557_032, 0.01, out)
    if workload == "resnet50":
        off = resnet50_segments()
        sig = resnet50_sigmas(seed)
        g = np.empty(int(off[-1]), np.float32) if out is None else out
        for t in range(161):
            normal([wid, seed, step, t], int(off[t + 1] - off[t]), float(sig[t]),
                   out=g[off[t]:off[t + 1]])
        return g
    if workload == "deepspeech":
        return student_t([wid, seed, step], n or 122_000_000, 3.0, 1e-3, out)
    if workload == "bucket1g":
        n = n or (1 << 30)
        g = normal([wid, seed, step], n, 0.01, out)
        pos = outlier_positions(n, seed)
        g[pos] *= np.float32(100.0)
        return g
    raise KeyError(workload)


def outlier_positions(n: int, seed: int = 0) -> np.ndarray:
    """round(1e-4 * n) distinct positions, fixed for a seed (the same every step)."""
    m = int(round(1e-4 * n))
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([_IDS["bucket1g"], seed,
                                                                      7])))
    return np.sort(rng.choice(n, size=m, replace=False)).astype(np.int64)


def misc(words, n: int, sigma: float = 1.0) -> np.ndarray:
    """Small seeded arrays for edge-case tests."""
    return normal([_IDS["misc"]] + list(words), n, sigma)


WARMUP_SPARSITY = (0.75, 0.9375, 0.984375, 0.99609375, 0.999)
