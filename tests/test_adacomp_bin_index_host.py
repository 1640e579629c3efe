"""The AdaComp streaming pass's bin index by reciprocal, checked exhaustively on the host.

The AdaComp citation snippet (fixed-size bins of each layer's residual, a bin's largest |residual|
as its threshold) needs the bin of every entry. The streaming pass finds the local bin of tile
offset x, for bins of L entries shorter than a tile, as

    q = floor( fl32( fl32(x + 0.5) * fl32(1/L) ) )

with fl32 binary32 round-to-nearest-even (the kernel's __fadd_rn, __fmul_rn and __float2uint_rd,
and the host's 1.0f / (float)L). x is the tile start's offset within its bin plus the offset in
the tile, so x < L + tile. This test takes the same binary32 steps with numpy and checks q == x // L
for every L in [4, 4095] and every x < L + 4096, which covers every tile length up to 4096 the
kernel may be built with (the default tile is 2048 entries). No GPU is needed: binary32 addition,
multiplication and division are correctly rounded on both sides.
"""
import numpy as np

TILE_MAX = 4096  # the largest streaming tile the kernel's static_assert admits


def _bin_by_reciprocal(x: np.ndarray, L: int) -> np.ndarray:
    inv = np.float32(1.0) / np.float32(L)                      # the host's 1.0f / (float)L
    xf = x.astype(np.float32)                                  # exact: x < 2^24
    s = xf + np.float32(0.5)                                   # __fadd_rn (exact here)
    prod = s * inv                                             # __fmul_rn
    assert prod.dtype == np.float32
    return np.floor(prod).astype(np.int64)                     # __float2uint_rd


def test_bin_index_by_reciprocal_equals_integer_division():
    bad = []
    for L in range(4, TILE_MAX):
        x = np.arange(L + TILE_MAX, dtype=np.int64)
        q = _bin_by_reciprocal(x, L)
        wrong = np.nonzero(q != x // L)[0]
        if wrong.size:
            bad.append((L, int(x[wrong[0]])))
    assert not bad, f"reciprocal bin index differs from x // L at (L, x) = {bad[:5]}"


def test_the_check_catches_a_wrong_shortcut():
    # without the half-entry offset the product lands just under an integer for some x = j L
    # (fl32(1/L) below 1/L), so a plain floor(x * fl32(1/L)) is not a valid bin index
    def plain(x, L):
        inv = np.float32(1.0) / np.float32(L)
        return np.floor(x.astype(np.float32) * inv).astype(np.int64)

    found = False
    for L in range(4, 200):
        x = np.arange(L + TILE_MAX, dtype=np.int64)
        if np.any(plain(x, L) != x // L):
            found = True
            break
    assert found
