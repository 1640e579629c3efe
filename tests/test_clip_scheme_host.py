"""A host model of the GPU clipping sum's integer steps (CPU only).

The kernels `k_clip_tiles` and `k_clip_round` sum the squares of a segment exactly. The
segment is cut into 4096-entry tiles; each block of the grid takes a contiguous range of the
tiles. In a tile, warp w holds entries [512 w, 512 w + 512), 16 per thread, and each thread sums
its squares in two 64-bit bands below its own largest entry: an entry with e' = e_band + d
(d <= 6) adds the 64-bit product of its significand shifted left by d with itself,
(m 2^d)^2 = m^2 4^d, which needs m 2^d to fit 32 bits. The thread's largest e' is read off its
largest |x| bits (a thread that holds inf or NaN counts as 254). Each thread adds its band sums
into its own 128-bit window, anchored 68 bits below the square of the largest e' its warp has
seen since the window opened. A warp keeps its window over up to 16 tiles of a segment and
flushes it (the threads' windows summed, then added to the block's digits) when a tile brings a
larger e', after 16 tiles, and when the block leaves the segment. Anything below the window goes
to the block's 32-bit digits held in 64-bit words (shared memory) at once. When a block is done
with the segment, its digits, carries propagated, are added to the segment's words in global
memory. One thread per segment then propagates the carries and rounds once to binary64.

This model takes the same steps with Python integers and asserts the bounds the kernels rely
on: a shifted significand below 2^30, a band sum below 2^64, a window term below 2^118 and a
warp window below 2^128, a block word below 2^56 and a global word below 2^42. Its S must equal
the oracle's, the exact sum rounded once (the DGC review's local gradient clipping; the pages
fix no order of summation). It checks the scheme; the GPU parity tests check the kernels
themselves against the oracle, S included.
"""
import math
import struct

import numpy as np
import pytest

TILE, THREADS, PER, WARP = 4096, 256, 16, 32
GRID = 608  # blocks of the kernel's grid (4 per SM on 152 SMs)
DIGITS = 20  # 32-bit digits of X = sum M 2^(2e'-2) < 2^586
WIN_TILES = 16  # tiles a warp window holds before it is flushed


def _digits_add(words, i, sh, x):
    """words[i..i+2] += x 2^(32 i + sh) in three pieces below 2^32, 2^33 and 2^31."""
    assert 0 <= x < 2**64 and 0 <= sh < 32
    lo, hi = (x & 0xFFFFFFFF) << sh, (x >> 32) << sh
    words[i] += lo & 0xFFFFFFFF
    words[i + 1] += (lo >> 32) + (hi & 0xFFFFFFFF)
    words[i + 2] += hi >> 32


class _Warp:
    """A warp's window: its anchor E, lowest bit lo, tiles held, one part per thread."""

    def __init__(self):
        self.E, self.lo, self.ntw, self.win = 0, 0, 0, [0] * WARP

    def flush(self, block_words):
        if self.ntw == 0:
            return
        W = sum(self.win)
        assert W < 2**128
        _digits_add(block_words, self.lo >> 5, self.lo & 31, W & (2**64 - 1))
        _digits_add(block_words, (self.lo >> 5) + 2, self.lo & 31, W >> 64)
        self.ntw, self.win = 0, [0] * WARP


def _tile(block_words, bits, warps):
    """One tile (|x| bits, zero-padded to 4096) into its warps' windows and the block's digits;
    returns inf/NaN flags."""
    bits = list(bits) + [0] * (TILE - len(bits))
    threads = [bits[PER * t:PER * t + PER] for t in range(THREADS)]
    # the thread's largest e' from its largest |x| bits; inf or NaN counts as 254
    et = [max(min(max(th) >> 23, 254), 1) for th in threads]
    flags = 0
    for wi, w0 in enumerate(range(0, THREADS, WARP)):
        wp = warps[wi]
        em = max(et[w0:w0 + WARP])
        if wp.ntw == WIN_TILES or (wp.ntw and em > wp.E):
            wp.flush(block_words)
        if wp.ntw == 0:
            wp.E, wp.lo = em, max(2 * em - 68, 0)  # the window's lowest bit of X
        wp.ntw += 1
        lo = wp.lo

        for t in range(w0, w0 + WARP):
            lane = t - w0

            def place(v, bit):
                if v == 0:
                    return
                if bit >= lo:
                    assert v << (bit - lo) < 2**118
                    wp.win[lane] += v << (bit - lo)
                else:
                    _digits_add(block_words, bit >> 5, bit & 31, v)

            th = threads[t]
            if any((a >> 23) == 255 for a in th):  # a thread holding inf or NaN: entry by entry
                for a in th:
                    e = a >> 23
                    if e == 255:
                        flags |= 4 if a & 0x7FFFFF else 2
                        continue
                    m = (a & 0x7FFFFF) | 0x800000 if e else a
                    place(m * m, 2 * max(e, 1) - 2)
                continue
            ea = max(et[t], 7) - 6  # band 1: e' in [ea, ea + 6]
            eb = max(ea, 8) - 7     # band 2: e' in [eb, ea - 1]
            A1 = A2 = 0
            # the kernel's A2 in 64-bit words: every entry outside band 1 adds the square of its
            # significand shifted by (e - eb) mod 32, truncated to 32 bits; the entries below
            # band 2 then take their terms back out, so A2 ends exact modulo 2^64
            A2w = 0
            for a in th:
                e = a >> 23
                if e < ea:
                    w = (((a & 0x7FFFFF) | 0x800000) << ((e - eb) % 32)) % 2**32
                    A2w = (A2w + w * w) % 2**64
                    if e < eb:
                        A2w = (A2w - w * w) % 2**64
            for a in th:
                e = a >> 23  # band membership by the raw exponent: zeros and subnormals below
                if e >= eb:
                    assert e >= 1
                    m = (a & 0x7FFFFF) | 0x800000  # a normal entry's significand
                    sh = e - (ea if e >= ea else eb)
                    assert 0 <= sh <= 6
                    mm = m << sh
                    assert mm < 2**30
                    if e >= ea:
                        A1 += mm * mm
                    else:
                        A2 += mm * mm
                elif a:
                    ep = max(e, 1)
                    m = (a & 0x7FFFFF) | 0x800000 if e else a
                    _digits_add(block_words, (2 * ep - 2) >> 5, (2 * ep - 2) & 31, m * m)
            assert A1 < 2**64 and A2 < 2**64 and A2w == A2
            place(A1, 2 * ea - 2)
            place(A2, 2 * eb - 2)
        assert max(wp.win) < 2**128
    return flags


def _flush(seg_words, block_words):
    """A block's digits, carries propagated, into the segment's words (one add per digit)."""
    assert max(block_words) < 2**56
    carry = 0
    for j in range(DIGITS):
        s = block_words[j] + carry
        seg_words[j] += s & 0xFFFFFFFF
        carry = s >> 32
        block_words[j] = 0
    assert carry == 0


def _round(words):
    """Carries into 32-bit digits, then X 2^-298 rounded once to binary64 (ties to even)."""
    X, carry = 0, 0
    for j in range(DIGITS):
        s = words[j] + carry
        X |= (s & 0xFFFFFFFF) << (32 * j)
        carry = s >> 32
    assert carry == 0 and X < 2**586
    if X == 0:
        return 0.0
    t = X.bit_length() - 1
    if t <= 52:
        mant, low = X, 0
    else:
        low = t - 52
        mant, rest = X >> low, X & ((1 << low) - 1)
        half = 1 << (low - 1)
        if rest > half or (rest == half and mant & 1):
            mant += 1
            if mant == 1 << 53:
                mant, low = mant >> 1, low + 1
    return math.ldexp(mant, low - 298)


def model_sumsq(g, grid=GRID):
    """One segment through the kernels' steps: its tiles shared out as contiguous ranges over
    the blocks of a grid (as many as tiles, at most `grid`)."""
    bits = (np.asarray(g, np.float32).view(np.uint32) & 0x7FFFFFFF).tolist()
    tiles = [bits[t0:t0 + TILE] for t0 in range(0, len(bits), TILE)]
    words, flags = [0] * DIGITS, 0
    G = max(1, min(len(tiles), grid))
    for b in range(G):
        block, warps = [0] * DIGITS, [_Warp() for _ in range(THREADS // WARP)]
        for c in range(len(tiles) * b // G, len(tiles) * (b + 1) // G):
            flags |= _tile(block, tiles[c], warps)
        for wp in warps:
            wp.flush(block)
        _flush(words, block)
    assert max(words) < 2**42
    if flags & 4:
        return math.nan
    if flags & 2:
        return math.inf
    return _round(words)


def _cases():
    rng = np.random.default_rng(31)
    out = []
    for n in (1, 17, 4096, 5000, 40_003):  # the last spans ten tiles over several blocks
        out.append(("normal", (rng.standard_normal(n) * 1e-3).astype(np.float32)))
        out.append(("60 binades", (rng.standard_normal(n) * 2.0 ** rng.integers(-30, 30, n))
                    .astype(np.float32)))
        bits = rng.integers(0, 0x7F7FFFFF, n, endpoint=True).astype(np.uint32)
        out.append(("every exponent", bits.view(np.float32)))
        c = rng.standard_normal(n).astype(np.float32)
        c[::7] = np.float32(1e-44)
        out.append(("subnormals among normals", c))
        c = (rng.standard_normal(n) * 1e-39).astype(np.float32)  # tiny normals and subnormals
        c[::5] = np.float32(0.0)
        out.append(("near the subnormal range, with zeros", c))
        out.append(("largest binary32", np.full(n, np.finfo(np.float32).max, np.float32)))
        out.append(("least subnormal", np.full(n, np.float32(2.0**-149))))
        c = rng.standard_normal(n).astype(np.float32)
        c[::5] = np.inf
        c[1::9] = np.nan
        out.append(("inf and NaN", c))
        c = rng.standard_normal(n).astype(np.float32)
        c[::3] = -np.inf
        out.append(("inf", c))
    # 22 tiles: one block's warps hold a window over 16 tiles, then flush and reopen it; the
    # scale rises tile by tile (each tile reopens the window), falls, or jumps once
    n = 22 * TILE + 77
    ramp = np.arange(n) // TILE
    base = rng.standard_normal(n)
    out.append(("22 tiles", (base * 1e-2).astype(np.float32)))
    out.append(("22 tiles, rising", (base * 2.0 ** (3 * ramp - 30)).astype(np.float32)))
    out.append(("22 tiles, falling", (base * 2.0 ** (30 - 3 * ramp)).astype(np.float32)))
    out.append(("22 tiles, one jump", (base * np.where(ramp < 9, 1e-6, 1e6)).astype(np.float32)))
    return out


@pytest.mark.parametrize("name,g", _cases(), ids=lambda x: x if isinstance(x, str) else "")
def test_kernel_scheme_reaches_the_oracle(orc, name, g):
    want = orc.sumsq(g)
    for grid in (GRID, 1, 2):  # one block per tile, one block for all tiles, two blocks
        got = model_sumsq(g, grid)
        assert (math.isnan(want) and math.isnan(got)) or \
            struct.pack("<d", want) == struct.pack("<d", got), (name, grid, want, got)


def test_block_words_bound_at_the_largest_share():
    # the most tiles a block of the 608-block grid sums for one segment (n < 2^32 entries, so
    # fewer than 2^20 tiles), each adding at most 8 x 2 + 4096 shared adds of under 2^33 to a word
    # (two per warp flush, at most one flush per warp and tile; one per entry below the bands or
    # the window), and the warps' last flushes
    tiles_per_block = -(-(2**20) // GRID) + 1
    assert (tiles_per_block * (8 * 2 + 4096) + 8 * 2) * 2**33 < 2**56
    # a warp window: 32 threads x WIN_TILES tiles x (two terms below 2^118, or 16 single
    # squares below 2^114 for a thread holding inf or NaN)
    assert WARP * WIN_TILES * max(2 * 2**118, 16 * 2**114) <= 2**128
    assert GRID * 2**32 < 2**42  # one add of a 32-bit digit per block
