"""Property checks of the oracle over generated inputs (CPU only; skipped where hypothesis is
not installed).

The clipping norm's square is the exact sum of the entries' squares rounded once to binary64
(the DGC review, Proposed method, local gradient clipping; the pages fix no order of summation).
Python's math.fsum rounds the exact sum of binary64 values correctly, and every square of a
binary32 value is exact in binary64, so the two must agree on every finite input. Neither side
orders the entries, so any permutation gives the same S.
"""
import math

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

# any finite binary32, subnormals and both signs included, and zeros
finite_bits = st.integers(min_value=0, max_value=0x7F7FFFFF).flatmap(
    lambda b: st.sampled_from([b, b | 0x80000000]))
# magnitudes near one binade mixed with far smaller ones: rounding ties and sticky bits
clustered_bits = st.tuples(st.integers(0x3F000000, 0x3F800000), st.integers(0, 0x3F800000)) \
    .map(lambda t: t[0] if t[1] & 1 else t[1])


def _as_f32(bits):
    return np.array(bits, dtype=np.uint32).view(np.float32)


@settings(max_examples=300, deadline=None)
@given(st.lists(finite_bits, max_size=200))
def test_sumsq_equals_fsum_of_exact_squares(orc, bits):
    g = _as_f32(bits)
    assert orc.sumsq(g) == math.fsum(float(x) * float(x) for x in g)


@settings(max_examples=200, deadline=None)
@given(st.lists(clustered_bits, min_size=1, max_size=300), st.randoms(use_true_random=False))
def test_sumsq_ignores_the_order_of_entries(orc, bits, rnd):
    g = _as_f32(bits)
    h = g.copy()
    rnd.shuffle(h)
    S = orc.sumsq(g)
    assert S == orc.sumsq(h) == math.fsum(float(x) * float(x) for x in g)


@settings(max_examples=100, deadline=None)
@given(st.lists(finite_bits, min_size=1, max_size=50),
       st.sampled_from([np.inf, -np.inf, np.nan]), st.integers(0, 49))
def test_sumsq_non_finite_entry(orc, bits, bad, at):
    g = _as_f32(bits)
    g[at % g.size] = bad
    S = orc.sumsq(g)
    if math.isnan(bad):
        assert math.isnan(S)
    else:
        assert S == math.inf
