"""Property checks of the oracle over generated inputs (CPU only; skipped where hypothesis is
not installed).

The clipping norm's square is the exact sum of the entries' squares rounded once to binary64
(the DGC review, Proposed method, local gradient clipping; the pages fix no order of summation).
Python's math.fsum rounds the exact sum of binary64 values correctly, and every square of a
binary32 value is exact in binary64, so the two must agree on every finite input. Neither side
orders the entries, so any permutation gives the same S. The message format's size rule and
its round trip are checked on index sets whose gaps sit at the 16-bit escape boundary.
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


# Message format of the DGC review (Proposed method: 32-bit values with 16-bit zero-run
# lengths): a gap of r skipped entries before a value takes r // 65535 escape tokens and one
# value token, so T = |S| + sum(r // 65535) and the message is 32 + 6T bytes, padded to a
# multiple of 4. Gaps around the escape boundary are drawn on purpose.
boundary_gaps = st.one_of(
    st.sampled_from([0, 1, 65533, 65534, 65535, 65536, 131069, 131070, 131071, 196605]),
    st.integers(0, 300_000))


@settings(max_examples=150, deadline=None)
@given(st.lists(boundary_gaps, max_size=12), st.integers(0, 70_000), st.data())
def test_codec_roundtrip_at_escape_boundaries(orc, gaps, tail, data):
    idx = np.cumsum(np.array(gaps, dtype=np.int64) + 1) - 1
    n = int(idx[-1] + 1 + tail) if idx.size else tail
    vals = data.draw(st.lists(finite_bits, min_size=idx.size, max_size=idx.size))
    val = _as_f32(vals)
    msg = orc.encode(idx.astype(np.uint32), val, n)
    T = idx.size + sum(g // 65535 for g in gaps)
    assert len(msg) == 32 + 6 * T + (2 if T % 2 else 0)
    rc, dense = orc.decode_accumulate([msg], n)
    assert rc == 0
    exp = np.zeros(n, np.float32)
    exp[idx] = np.float32(0.0) + val  # the decoded sum starts at +0, so -0 arrives as +0
    assert np.array_equal(dense.view(np.uint32), exp.view(np.uint32))
