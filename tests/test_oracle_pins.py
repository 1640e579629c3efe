"""Pins of the oracle against what the DGC pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: published SplitMix64
outputs, exact rational arithmetic (the definition of a correctly rounded fma/add), brute-force
sorting on tiny inputs, hand-built codec streams, and sizes printed in the DGC review.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest

import exact_fp32 as X
import workloads
from conftest import read_golden

GOLD = 0x9E3779B97F4A7C15
M64 = 2**64 - 1


def _sm_mix(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def sm_outputs(seed, count):
    """SplitMix64 outputs; pinned to published values in test_python_splitmix_published."""
    out, s = [], seed
    for _ in range(count):
        s = (s + GOLD) & M64
        out.append(_sm_mix(s))
    return out


# ---------------------------------------------------------------------------------- SplitMix64
def test_oracle_splitmix64_published_outputs(orc):
    for _, vals in read_golden("splitmix64.txt"):
        seed, outs = vals[0], vals[1:]
        s = seed
        for o in outs:
            s = (s + GOLD) & M64
            assert orc.mix64(s) == o


def test_python_splitmix_published():
    for _, vals in read_golden("splitmix64.txt"):
        assert sm_outputs(vals[0], len(vals) - 1) == vals[1:]


@pytest.mark.parametrize("seed", [0, 1234567, M64, 42])
def test_sample_positions_follow_definition(orc, seed):
    for s in [0, 1, 5, 160]:
        seg_seed = sm_outputs(seed, s + 1)[-1]
        xs = sm_outputs(seg_seed, 16)
        for n_s in [1, 2, 999, 24_000_000, 2**32 - 1]:
            for j in range(16):
                p = orc.sample_position(seed, s, j, n_s)
                assert p == (xs[j] * n_s) >> 64
                assert 0 <= p < n_s


# ---------------------------------------------------------------------------------- k rule
@pytest.mark.parametrize("n,sparsity", [
    (1_048_576, "0.999"), (1 << 30, "0.75"), (1 << 30, "0.9375"), (1 << 30, "0.984375"),
    (1 << 30, "0.99609375"), (1 << 30, "0.999"), (24_000_000, "0.999"), (2_000_000, "0.999"),
    (2_359_296, "0.999"), (64, "0.999"), (999, "0.999"), (1001, "0.999"), (1, "0.999"),
    (0, "0.999"), (1000, "0"), (1000, "1"), (4096, "0.5"), (10_737_419, "0.999"),
    (2**32 - 1, "0.999"), (123_457, "0.99"), (7, "0.3")])
def test_count_is_ceiling_of_exact_fraction(orc, n, sparsity):
    expect = math.ceil(n * (1 - Fraction(sparsity)))
    assert orc.count(n, orc.ppb(1.0 - float(sparsity))) == expect


def test_single_tensor_k_is_1049(orc):
    # 0.1% of 1,048,576 is 1048.576: the rounded-up count is 1049.
    assert orc.count(1_048_576, orc.ppb(1 - 0.999)) == 1049


def test_warmup_schedule_is_powers_of_four():
    # DGC review, Proposed method, bullet 6 (warm-up raises sparsity gradually); the schedule's
    # first four densities are 4^-1..4^-4 exactly, then 0.1%.
    for i, s in enumerate(workloads.WARMUP_SPARSITY[:4], start=1):
        assert Fraction(s) == 1 - Fraction(1, 4**i)
    assert workloads.WARMUP_SPARSITY[4] == 0.999


def test_deepspeech_message_size_matches_dgc_review(orc):
    # DGC review, Abstract: DeepSpeech's 488 MB gradient becomes 0.74 MB. 488 MB of binary32 is
    # 122,000,000 entries; at 99.9% the six segments send 5 * 24,000 + 2,000 = 122,000 values,
    # 6 bytes each in this format, i.e. 0.732 MB: within 2% of the printed figure.
    off = workloads.deepspeech_segments()
    assert off[-1] * 4 == 488_000_000
    d = orc.ppb(1 - 0.999)
    k = sum(orc.count(int(b - a), d) for a, b in zip(off[:-1], off[1:]))
    assert k == 122_000
    idx = np.arange(k, dtype=np.uint32) * 1000 + 7  # gaps of 999 < 65535: no escapes
    msg = orc.encode(idx, np.ones(k, np.float32), int(off[-1]))
    assert len(msg) == 32 + 6 * k
    assert abs(len(msg) / 1e6 - 0.74) / 0.74 < 0.02


# ---------------------------------------------------------------------------------- selection
def brute_topk(v, k, among=None):
    keys = [X.key(x) for x in v]
    cand = range(len(v)) if among is None else among
    order = sorted(cand, key=lambda i: (-keys[i], i))
    return sorted(order[:k])


def _tricky(rng, n, kind):
    if kind == 0:
        return rng.standard_normal(n).astype(np.float32)
    if kind == 1:
        return rng.integers(-3, 4, n).astype(np.float32)
    if kind == 2:
        return np.where(rng.random(n) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
    if kind == 3:
        mags = np.array([0.5, 1.0, 2.0, 1e-30, 3.0e30], np.float32)
    else:  # keys at the top of the range; only for tests that do no arithmetic
        mags = np.array([0.5, 3.0e38, np.inf, 1e-45, 0.0], np.float32)
    return (mags[rng.integers(0, mags.size, n)] * rng.choice([-1, 1], n)).astype(np.float32)


@pytest.mark.parametrize("seed", range(120))
def test_topk_matches_bruteforce(orc, seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 300))
    v = _tricky(rng, n, seed % 5)
    k = int(rng.integers(0, n + 1))
    sel = orc.topk(v, np.arange(n, dtype=np.uint32), k)
    assert np.nonzero(sel)[0].tolist() == brute_topk(v, k)


def _exact_accumulate(g, u, v, m, scale=None):
    """u' = fma(m, u, g'), v' = v + u' with g' = g * scale when scale is given; exact rational
    arithmetic rounded once per operation."""
    un = np.empty_like(u)
    vn = np.empty_like(v)
    for i in range(g.size):
        gp = g[i] if scale is None else X.mul_f32(g[i], scale)
        un[i] = X.fma_f32(m, u[i], gp)
        vn[i] = X.add_f32(v[i], un[i])
    return un, vn


def _random_segments(rng, n, max_seg=4):
    nseg = int(rng.integers(1, max_seg + 1))
    cuts = np.sort(rng.integers(0, n + 1, nseg - 1))
    return np.concatenate([[0], cuts, [n]]).astype(np.int64)


@pytest.mark.parametrize("seed", range(40))
def test_exact_compress_matches_definition(orc, seed):
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 400))
    off = _random_segments(rng, n)
    kind = seed % 4
    g = _tricky(rng, n, kind)
    u = (_tricky(rng, n, kind) * np.float32(0.5)).astype(np.float32)
    v = _tricky(rng, n, (kind + 1) % 4)
    m = np.float32(rng.choice([0.0, 0.5, 0.9, 1.0]))
    sparsity = float(rng.choice([0.0, 0.5, 0.9, 0.99, 0.999, 1.0]))
    mask = bool(seed % 2)
    un, vn = _exact_accumulate(g, u, v, m)
    exp_idx = []
    for a, b in zip(off[:-1], off[1:]):
        k = math.ceil((b - a) * (1 - Fraction(str(sparsity))))
        exp_idx += [int(a) + i for i in brute_topk(vn[a:b], k)]
    p = orc.make_params(orc.EXACT, sparsity, float(m), mask_momentum=mask)
    uu, vv = u.copy(), v.copy()
    idx, val, st = orc.compress(g, uu, vv, off, p)
    assert idx.tolist() == exp_idx
    assert [X.bits(x) for x in val] == [X.bits(vn[i]) for i in exp_idx]
    v_exp, u_exp = vn.copy(), un.copy()
    v_exp[exp_idx] = 0.0
    if mask:
        u_exp[exp_idx] = 0.0
    assert vv.view(np.uint32).tolist() == v_exp.view(np.uint32).tolist()
    assert uu.view(np.uint32).tolist() == u_exp.view(np.uint32).tolist()
    assert sum(s["sent"] for s in st) == len(exp_idx)


def _nonzero_normal(rng, n, scale=1.0):
    x = (rng.standard_normal(n) * scale).astype(np.float32)
    x[x == 0] = np.float32(0.25)
    return x


def test_sparsity0_masking_off_is_dense_momentum_sgd(orc):
    # DGC review, Proposed method, bullet 3: momentum correction makes the sparse update follow
    # dense momentum SGD. With nothing held back (sparsity 0) and no masking, every step sends
    # exactly the momentum velocity u_t = m * u_{t-1} + g_t.
    rng = np.random.default_rng(7)
    n, m = 257, np.float32(0.9)
    u = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    vel = np.zeros(n, np.float32)
    p = orc.make_params(orc.EXACT, 0.0, 0.9, mask_momentum=False)
    for _ in range(5):
        g = _nonzero_normal(rng, n, 0.01)
        vel = np.array([X.fma_f32(m, vel[i], g[i]) for i in range(n)], np.float32)
        idx, val, _ = orc.compress(g, u, v, np.array([0, n]), p)
        assert idx.tolist() == list(range(n))
        assert val.view(np.uint32).tolist() == vel.view(np.uint32).tolist()
        assert not v.any()


def test_sparsity0_masking_on_is_plain_sgd(orc):
    # DGC review, Proposed method, bullet 5: with momentum factor masking the momentum of a sent
    # entry is cleared, so with sparsity 0 each step sends the fresh gradient itself.
    rng = np.random.default_rng(8)
    n = 300
    u = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    p = orc.make_params(orc.EXACT, 0.0, 0.9, mask_momentum=True)
    for _ in range(4):
        g = _nonzero_normal(rng, n)
        idx, val, _ = orc.compress(g, u, v, np.array([0, n]), p)
        assert val.view(np.uint32).tolist() == g.view(np.uint32).tolist()
        assert not u.any() and not v.any()


def test_momentum0_sparsity0_sends_gradient(orc):
    rng = np.random.default_rng(9)
    n = 100
    g = _nonzero_normal(rng, n)
    u = _nonzero_normal(rng, n)
    v = np.zeros(n, np.float32)
    idx, val, _ = orc.compress(g, u, v, np.array([0, n]),
                               orc.make_params(orc.EXACT, 0.0, 0.0, mask_momentum=False))
    assert val.view(np.uint32).tolist() == g.view(np.uint32).tolist()


@pytest.mark.parametrize("mode", [0, 1])
def test_conservation_sent_plus_residual(orc, mode):
    # DGC review, Proposed method, bullet 1: what is not sent stays in the local accumulator.
    # Sent value + residual equals what an all-held-back step (sparsity 1) accumulates, bitwise.
    rng = np.random.default_rng(11 + mode)
    n = 5000
    off = np.array([0, 1234, 1234, 4000, n])
    g, u0, v0 = (_nonzero_normal(rng, n) for _ in range(3))
    ua, va, ub, vb = u0.copy(), v0.copy(), u0.copy(), v0.copy()
    pa = orc.make_params(mode, 0.99, 0.9, mask_momentum=True, sample_ratio=0.05, seed=3)
    pb = orc.make_params(mode, 1.0, 0.9, mask_momentum=True, sample_ratio=0.05, seed=3)
    idx, val, _ = orc.compress(g, ua, va, off, pa)
    idx_b, _, _ = orc.compress(g, ub, vb, off, pb)
    assert idx_b.size == 0 and idx.size > 0
    sent = np.zeros(n, bool)
    sent[idx] = True
    assert val.view(np.uint32).tolist() == vb[idx].view(np.uint32).tolist()
    assert not va[sent].any() and not ua[sent].any()
    assert va[~sent].view(np.uint32).tolist() == vb[~sent].view(np.uint32).tolist()
    assert ua[~sent].view(np.uint32).tolist() == ub[~sent].view(np.uint32).tolist()


@pytest.mark.parametrize("seed", range(12))
def test_accumulate_one_is_single_rounding_fma(orc, seed):
    rng = np.random.default_rng(50 + seed)
    for _ in range(200):
        g, u, v = (np.float32(x) for x in rng.standard_normal(3) * 10.0 ** rng.integers(-6, 6, 3))
        m = np.float32(rng.choice([0.9, 0.99, 0.5, 1.0, 0.0]))
        uo, vo = orc.accumulate_one(g, u, v, m)
        ue = X.fma_f32(m, u, g)
        assert X.bits(uo) == X.bits(ue)
        assert X.bits(vo) == X.bits(X.add_f32(v, ue))


@pytest.mark.parametrize("seed", range(2))
def test_accumulate_one_clipped_scales_g_first(orc, seed):
    # a clipped gradient enters as the binary32 product g * scale (one rounding), then the fma;
    # an unclipped one enters bitwise, whatever scale is passed
    rng = np.random.default_rng(70 + seed)
    for _ in range(200):
        g, u, v = (np.float32(x) for x in rng.standard_normal(3) * 10.0 ** rng.integers(-6, 6, 3))
        scale = np.float32(rng.uniform(0.01, 0.99))
        m = np.float32(rng.choice([0.9, 0.5, 0.0]))
        uo, vo = orc.accumulate_one(g, u, v, m, scale=scale, clipped=True)
        ue = X.fma_f32(m, u, X.mul_f32(g, scale))
        assert X.bits(uo) == X.bits(ue)
        assert X.bits(vo) == X.bits(X.add_f32(v, ue))
        uo, _ = orc.accumulate_one(g, u, v, m, scale=scale, clipped=False)
        assert X.bits(uo) == X.bits(X.fma_f32(m, u, g))


# ---------------------------------------------------------------------------------- clipping
def test_clip_scale_closed_form(orc):
    # DGC review, Proposed method, bullet 4: norm of (3, 4) is 5; bound 1 gives 1/5 in binary32.
    s, clipped = orc.clip_scale(np.array([3.0, 4.0], np.float32), 1.0)
    assert clipped and X.bits(s) == X.bits(X.round_f32(Fraction(1, 5)))
    s, clipped = orc.clip_scale(np.array([3.0, 4.0], np.float32), 5.0)
    assert not clipped and s == 1.0


def _is_nearest_binary64(S: float, exact: Fraction) -> bool:
    """S is a binary64 nearest to `exact`; on a tie, the one whose significand is even."""
    here = abs(Fraction(S) - exact)
    for nb in (np.nextafter(S, -np.inf), np.nextafter(S, np.inf)):
        there = abs(Fraction(float(nb)) - exact)
        if there < here:
            return False
        if there == here and (struct.unpack("<Q", struct.pack("<d", S))[0] & 1):
            return False
    return True


@pytest.mark.parametrize("n", [1, 2, 4095, 4096, 4097, 12289, 50_000])
def test_sumsq_is_the_exact_sum_rounded_once(orc, n):
    # Entries over ~60 binades, subnormals included: S must be the binary64 nearest to the exact
    # rational sum of squares (ties to even), and equal to Python's correctly rounded math.fsum
    # of the (exact) binary64 squares.
    rng = np.random.default_rng(n)
    g = (rng.standard_normal(n) * 2.0 ** rng.integers(-30, 30, n)).astype(np.float32)
    g[rng.integers(0, n, max(1, n // 100))] = np.float32(1e-44)
    exact = sum(Fraction(float(x)) ** 2 for x in g)
    S = orc.sumsq(g)
    assert _is_nearest_binary64(S, exact)
    assert S == math.fsum(float(x) * float(x) for x in g)


def test_sumsq_exact_on_integers(orc):
    g = np.ones(4096 * 3 + 5, np.float32)
    assert orc.sumsq(g) == g.size
    g = np.arange(-2000, 2001, dtype=np.float32)
    assert orc.sumsq(g) == sum(int(x) ** 2 for x in range(-2000, 2001))


def test_compress_reports_the_squared_norm(orc):
    # the per-segment stat is S itself (math.fsum of the exact binary64 squares), 0 when
    # clipping is off
    rng = np.random.default_rng(23)
    n = 9000
    off = np.array([0, 0, 4097, 5000, n])
    g = (rng.standard_normal(n) * 2.0 ** rng.integers(-20, 20, n)).astype(np.float32)
    for c in (0.0, 1.0):
        u = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        _, _, st = orc.compress(g, u, v, off, orc.make_params(orc.EXACT, 0.99, 0.9, clip_norm=c))
        for s, (a, b) in enumerate(zip(off[:-1], off[1:])):
            want = math.fsum(float(x) * float(x) for x in g[a:b]) if c else 0.0
            assert st[s]["clip_sumsq"] == want


def test_clip_within_bound_is_bitwise_noop(orc):
    rng = np.random.default_rng(21)
    n = 9000
    off = np.array([0, 100, 5000, n])
    g, u, v = (_nonzero_normal(rng, n, 1e-3) for _ in range(3))
    outs = []
    for c in (0.0, 1e6):
        uu, vv = u.copy(), v.copy()
        idx, val, _ = orc.compress(g, uu, vv, off, orc.make_params(orc.EXACT, 0.99, 0.9,
                                                                    clip_norm=c))
        outs.append((idx.tolist(), val.tobytes(), uu.tobytes(), vv.tobytes()))
    assert outs[0] == outs[1]


def test_clipped_gradient_has_norm_c(orc):
    # With momentum 0, sparsity 0 and masking, the sent values are the clipped gradient itself.
    rng = np.random.default_rng(22)
    n = 20_000
    off = np.array([0, 7000, n])
    g = _nonzero_normal(rng, n)
    u = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    idx, val, st = orc.compress(g, u, v, off, orc.make_params(orc.EXACT, 0.0, 0.0, clip_norm=2.5))
    for s, (a, b) in enumerate(zip(off[:-1], off[1:])):
        norm = math.sqrt(sum(float(x) ** 2 for x in val[a:b]))
        assert abs(norm - 2.5) / 2.5 < 1e-6
        assert X.bits(val[a]) == X.bits(X.mul_f32(g[a], st[s]["clip_scale"]))


# ---------------------------------------------------------------------------------- sampled
def _expected_sampled(vn, off, sparsity, ratio, factor, seed):
    d = 1 - Fraction(str(sparsity))
    out, info = [], []
    for s, (a, b) in enumerate(zip(off[:-1], off[1:])):
        ns = int(b - a)
        k = math.ceil(ns * d)
        if k == 0:
            info.append((0, 0, 0))
            continue
        ms = math.ceil(ns * Fraction(str(ratio)))
        ks = math.ceil(ms * d)
        seg_seed = sm_outputs(seed, s + 1)[-1]
        pos = [(x * ns) >> 64 for x in sm_outputs(seg_seed, ms)]
        keys = sorted((X.key(vn[a + p]) for p in pos), reverse=True)
        t = keys[ks - 1]
        C = [i for i in range(ns) if X.key(vn[a + i]) >= t]
        resel = len(C) * 10**9 > round(factor * 10**9) * k
        S = brute_topk(vn[a:b], k, among=C) if resel else C
        out += [int(a) + i for i in S]
        info.append((t, len(C), int(resel)))
    return out, info


@pytest.mark.parametrize("seed", range(30))
def test_sampled_compress_matches_definition(orc, seed):
    rng = np.random.default_rng(3000 + seed)
    n = int(rng.integers(200, 3000))
    off = _random_segments(rng, n, 3)
    kind = [0, 1, 3][seed % 3]  # kind 1 and 3: many ties -> |C| >> k -> re-selection
    g, u, v = (_tricky(rng, n, kind) for _ in range(3))
    m = np.float32(0.9)
    sparsity = float(rng.choice([0.5, 0.9, 0.99, 0.999]))
    ratio = float(rng.choice([0.01, 0.05, 0.2]))
    rseed = int(rng.integers(0, 2**63))
    un, vn = _exact_accumulate(g, u, v, m)
    exp_idx, info = _expected_sampled(vn, off, sparsity, ratio, 1.3, rseed)
    p = orc.make_params(orc.SAMPLED, sparsity, 0.9, sample_ratio=ratio, reselect_factor=1.3,
                        seed=rseed)
    uu, vv = u.copy(), v.copy()
    idx, val, st = orc.compress(g, uu, vv, off, p)
    assert idx.tolist() == exp_idx
    for s, (t, nc, resel) in enumerate(info):
        if st[s]["k"]:
            assert (st[s]["sample_key"], st[s]["candidates"], st[s]["reselected"]) == (t, nc, resel)


def test_sampled_reselect_equals_exact_selection(orc):
    # When re-selection runs, C holds every entry with |v| >= t and more than k of them, so the
    # exact top-k over C is the exact top-k of the whole segment.
    rng = np.random.default_rng(5)
    n = 20_000
    g = rng.integers(-2, 3, n).astype(np.float32)  # heavy ties -> |C| >> k
    u = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    off = np.array([0, n])
    ps = orc.make_params(orc.SAMPLED, 0.999, 0.9, sample_ratio=0.01, seed=1)
    pe = orc.make_params(orc.EXACT, 0.999, 0.9)
    i1, v1, st = orc.compress(g, u.copy(), v.copy(), off, ps)
    i2, v2, _ = orc.compress(g, u.copy(), v.copy(), off, pe)
    assert st[0]["reselected"] == 1
    assert i1.tolist() == i2.tolist() and v1.tobytes() == v2.tobytes()


# ---------------------------------------------------------------------------------- codec
def golden_message(name):
    n, entries, tokens, size = None, [], [], None
    for tag, vals in read_golden(name):
        if tag == "n":
            n = vals[0]
        elif tag == "entry":
            entries.append(vals)
        elif tag == "token":
            tokens.append(vals)
        elif tag == "size":
            size = vals[0]
    T = len(tokens)
    msg = struct.pack("<4sHHQQQ", b"DGC1", 1, 0, n, T, len(entries))
    msg += b"".join(struct.pack("<I", t[1]) for t in tokens)
    msg += b"".join(struct.pack("<H", t[0]) for t in tokens)
    msg += b"\0" * ((-len(msg)) % 4)
    idx = np.array([e[0] for e in entries], np.uint32)
    val = np.array([e[1] for e in entries], np.uint32).view(np.float32)
    return n, idx, val, msg, size


@pytest.mark.parametrize("name", ["codec_gaps.txt", "codec_single.txt", "codec_odd.txt",
                                  "codec_empty.txt"])
def test_codec_golden(orc, name):
    n, idx, val, msg, size = golden_message(name)
    assert len(msg) == size
    assert orc.encode(idx, val, n) == msg
    rc, dense = orc.decode_accumulate([msg], n)
    assert rc == 0
    exp = np.zeros(n, np.float32)
    exp[idx] = exp[idx] + val  # +0 + x: a sent -0.0 lands as +0.0
    assert dense.view(np.uint32).tolist() == exp.view(np.uint32).tolist()


def test_decode_order_golden(orc):
    rows = read_golden("decode_order.txt")
    n = rows[0][1][0]
    msgs = [orc.encode(np.array([r[1][0]], np.uint32),
                       np.array([r[1][1]], np.uint32).view(np.float32), n)
            for r in rows if r[0] == "learner"]
    rc, dense = orc.decode_accumulate(msgs, n)
    assert rc == 0
    for tag, (pos, b) in ((t, v) for t, v in rows if t == "expect"):
        assert X.bits(dense[pos]) == b


def _walk_positions(msg):
    n, T, nnz = struct.unpack_from("<QQQ", msg, 8)
    runs = struct.unpack_from(f"<{T}H", msg, 32 + 4 * T)
    pos, out = -1, []
    for r in runs:
        if r == 0xFFFF:
            pos += 0xFFFF
        else:
            pos += r + 1
            out.append(pos)
    return out


@pytest.mark.parametrize("seed", range(25))
def test_codec_roundtrip_random(orc, seed):
    rng = np.random.default_rng(700 + seed)
    n = int(rng.integers(1, 2_000_000))
    k = int(rng.integers(0, min(n, 3000) + 1))
    idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
    val = _tricky(rng, k, seed % 4)
    msg = orc.encode(idx, val, n)
    assert _walk_positions(msg) == idx.tolist()  # the format is a bijection on (idx, val)
    gaps = np.diff(np.concatenate([[-1], idx.astype(np.int64)])) - 1
    T = k + int((gaps // 65535).sum())
    assert len(msg) == 32 + 6 * T + (2 if T % 2 else 0)
    rc, dense = orc.decode_accumulate([msg], n)
    assert rc == 0
    exp = np.zeros(n, np.float32)
    exp[idx] += val
    assert np.array_equal(dense.view(np.uint32), exp.view(np.uint32))


def test_decode_sums_learners_in_order(orc):
    rng = np.random.default_rng(31)
    n, W = 5000, 7
    msgs, parts = [], []
    for _ in range(W):
        idx = np.sort(rng.choice(n, size=400, replace=False)).astype(np.uint32)
        val = (rng.standard_normal(400) * 10.0 ** rng.integers(-4, 4, 400)).astype(np.float32)
        msgs.append(orc.encode(idx, val, n))
        parts.append((idx, val))
    base = rng.standard_normal(n).astype(np.float32)
    for acc in (False, True):
        exp = base.copy() if acc else np.zeros(n, np.float32)
        for idx, val in parts:
            exp[idx] = exp[idx] + val  # numpy binary32 addition, one rounding each
        rc, dense = orc.decode_accumulate(msgs, n, dense=base, accumulate=acc)
        assert rc == 0
        assert np.array_equal(dense.view(np.uint32), exp.view(np.uint32))


def test_decode_rejects_malformed(orc):
    n = 1000
    good = orc.encode(np.array([5, 999], np.uint32), np.array([1.0, 2.0], np.float32), n)
    bad = [b"XGC1" + good[4:], good[:4] + struct.pack("<H", 2) + good[6:],
           good[:8] + struct.pack("<Q", n + 1) + good[16:], good + b"\0\0\0\0", good[:31],
           good[:32 + 8] + struct.pack("<H", 999) + good[32 + 10:]]  # second run past n
    for b in bad:
        base = np.full(n, 7.0, np.float32)
        rc, dense = orc.decode_accumulate([good, b], n, dense=base, accumulate=True)
        assert rc == orc.ECORRUPT
        assert np.all(dense == 7.0)


# ------------------------------------------------------------- the clipping sum, rounded once
# The reading makes the sum of squares exact and rounds it once to binary64 (ties to even), so no
# order of summation shows. The inputs are powers of two worked out by hand: 2^54 has spacing 4
# between binary64 neighbours, so 2^54 + 1 rounds down, 2^54 + 2 is a tie that goes to the even
# 2^54, and 2^54 + 3 rounds up to 2^54 + 4.
def _sparse(n, items):
    g = np.zeros(n, np.float32)
    for i, x in items:
        g[i] = x
    return g


@pytest.mark.parametrize("ones,expected", [(1, 2.0**54), (2, 2.0**54), (3, 2.0**54 + 4),
                                           (4, 2.0**54 + 4), (6, 2.0**54 + 8)])
def test_sumsq_rounds_once_to_nearest_even(orc, ones, expected):
    g = _sparse(16384, [(0, 2.0**27)] + [(4096 * (i % 4) + i, 1.0) for i in range(1, ones + 1)])
    assert orc.sumsq(g) == expected
    # the same entries in any order give the same S: a running binary64 sum from the left
    # would drop each 1 against 2^54 and return 2^54 for every count above
    rng = np.random.default_rng(ones)
    for _ in range(3):
        assert orc.sumsq(g[rng.permutation(g.size)]) == expected


def test_sumsq_keeps_what_partial_sums_would_drop(orc):
    # 2^-298 (the square of the least binary32 subnormal) is far below the spacing of 1.0, but
    # 2^53 of them would add up to 2^-245; here 3 of them next to 1 vanish, alone they stay
    tiny = np.float32(2.0**-149)
    assert orc.sumsq(np.array([tiny], np.float32)) == 2.0**-298
    assert orc.sumsq(np.array([tiny, tiny, tiny], np.float32)) == 3 * 2.0**-298
    assert orc.sumsq(np.array([1.0, tiny, tiny, tiny], np.float32)) == 1.0
    # the largest binary32 squared four times: exact, far from binary64 overflow
    big = np.float32(np.finfo(np.float32).max)
    assert orc.sumsq(np.full(4, big, np.float32)) == 4 * float(big) ** 2
    # above 1 the spacing is 2^-52: two squares of 2^-27 (2^-54 each) make exactly half of it,
    # a tie that stays at the even 1.0; a trace more (2^-298) tips it to 1 + 2^-52
    h = 2.0**-27
    assert orc.sumsq(np.array([1.0, h], np.float32)) == 1.0
    assert orc.sumsq(np.array([1.0, h, h], np.float32)) == 1.0
    assert orc.sumsq(np.array([h, 1.0, tiny, h], np.float32)) == 1.0 + 2.0**-52


def test_sumsq_non_finite(orc):
    assert math.isnan(orc.sumsq(np.array([1.0, np.nan, np.inf], np.float32)))
    assert orc.sumsq(np.array([1.0, -np.inf, 2.0], np.float32)) == math.inf
    assert orc.sumsq(np.zeros(0, np.float32)) == 0.0


def test_reselect_not_taken_at_exactly_factor_times_k(orc):
    # |C| = 13 = 1.3 * 10 is not more than 1.3k: C is sent as it is (13 entries, no re-selection).
    n, big = 100, np.float32(5.0)
    g = np.ones(n, np.float32)
    g[np.arange(13) * 7] = big
    off = np.array([0, n])
    for seed in range(200):
        exp_idx, info = _expected_sampled(g, off, 0.9, 1.0, 1.3, seed)
        if info[0][1] == 13:
            break
    else:
        pytest.fail("no seed gives |C| = 13")
    assert info[0][2] == 0 and len(exp_idx) == 13
    u = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    idx, _, st = orc.compress(g, u, v, off, orc.make_params(orc.SAMPLED, 0.9, 0.0,
                                                             sample_ratio=1.0, seed=seed))
    assert idx.tolist() == exp_idx
    assert st[0]["candidates"] == 13 and st[0]["reselected"] == 0


# ---------------------------------------------------------------------- AdaComp bins
def brute_bins(v, L):
    """Per run of L entries: the indices whose |v| equals the run's largest |v|, if above 0."""
    keys = [X.key(x) for x in v]
    out = []
    for b in range(0, len(v), L):
        mx = max(keys[b:b + L])
        if mx > 0:
            out += [i for i in range(b, min(b + L, len(v))) if keys[i] == mx]
    return out


@pytest.mark.parametrize("seed", range(60))
def test_bin_select_matches_bruteforce(orc, seed):
    rng = np.random.default_rng(4000 + seed)
    n = int(rng.integers(1, 400))
    v = _tricky(rng, n, seed % 5)
    L = int(rng.choice([1, 2, 3, 7, 16, 50, 1000]))
    sel = orc.bin_select(v, L)
    assert np.nonzero(sel)[0].tolist() == brute_bins(v, L)


def test_bin_select_closed_forms(orc):
    rng = np.random.default_rng(1)
    v = rng.standard_normal(1000).astype(np.float32)
    v[::10] = 0.0
    # one entry per bin: every nonzero entry is its own bin's largest
    assert np.nonzero(orc.bin_select(v, 1))[0].tolist() == np.nonzero(v)[0].tolist()
    # one bin larger than everything: the entries at the largest |v|
    assert np.nonzero(orc.bin_select(v, 5000))[0].tolist() == [int(np.argmax(np.abs(v)))]
    assert not orc.bin_select(np.zeros(100, np.float32), 10).any()
    w = np.array([1, -3, 3, 2, -3, 0, 0, 0, 5, -5], np.float32)
    assert np.nonzero(orc.bin_select(w, 5))[0].tolist() == [1, 2, 4, 8, 9]


@pytest.mark.parametrize("seed", range(20))
def test_adacomp_compress_matches_definition(orc, seed):
    rng = np.random.default_rng(5000 + seed)
    n = int(rng.integers(1, 500))
    off = _random_segments(rng, n)
    kind = seed % 4
    g, u, v = (_tricky(rng, n, kind) for _ in range(3))
    m = np.float32(rng.choice([0.0, 0.9]))
    L = int(rng.choice([1, 4, 10, 64]))
    mask = bool(seed % 2)
    un, vn = _exact_accumulate(g, u, v, m)
    exp_idx = []
    for a, b in zip(off[:-1], off[1:]):
        exp_idx += [int(a) + i for i in brute_bins(vn[a:b], L)]
    p = orc.make_params(orc.ADACOMP, 0.999, float(m), mask_momentum=mask, bin_size=L)
    uu, vv = u.copy(), v.copy()
    idx, val, st = orc.compress(g, uu, vv, off, p)
    assert idx.tolist() == exp_idx
    assert [X.bits(x) for x in val] == [X.bits(vn[i]) for i in exp_idx]
    v_exp = vn.copy()
    v_exp[exp_idx] = 0.0
    assert vv.view(np.uint32).tolist() == v_exp.view(np.uint32).tolist()
    for s_, (a, b) in zip(st, zip(off[:-1], off[1:])):
        assert s_["k"] == -(-(int(b) - int(a)) // L)


# ------------------------------------------------------------------ decode -> plain SGD step
# Reading of "[Paper Review] Deep Gradient Compression ...", Abstract (distributed SGD) and
# "Proposed method" (momentum correction keeps the velocity on the learner): the receiver adds
# the messages in learner order from +0 and takes w <- fmaf(-lr, sum, w), one rounding. The
# expected values below come from exact rational arithmetic, not from the oracle.
def _apply_expected(w, parts, lr):
    s = {}
    for idx, val in parts:
        for i, x in zip(idx.tolist(), val):
            s[i] = X.add_f32(s.get(i, np.float32(0.0)), x)
    exp = w.copy()
    for i, t in s.items():
        exp[i] = X.fma_f32(np.float32(-lr), t, w[i])
    return exp, s


@pytest.mark.parametrize("name", ["codec_gaps.txt", "codec_single.txt", "codec_odd.txt",
                                  "codec_empty.txt"])
def test_decode_apply_golden_streams(orc, name):
    n, idx, val, msg, _ = golden_message(name)
    rng = np.random.default_rng(17)
    w = _tricky(rng, n, 0)
    exp, _ = _apply_expected(w, [(idx, val)], 0.75)
    rc, out = orc.decode_apply([msg], n, w, 0.75)
    assert rc == 0
    assert out.view(np.uint32).tolist() == exp.view(np.uint32).tolist()


def test_decode_apply_learner_order_golden(orc):
    # the ordered sum at index 2 is exactly 0 (see decode_order.txt), so w[2] keeps its bits;
    # any other order would leave 1 or -1e8 + ... and move w[2]
    rows = read_golden("decode_order.txt")
    n = rows[0][1][0]
    msgs = [orc.encode(np.array([r[1][0]], np.uint32),
                       np.array([r[1][1]], np.uint32).view(np.float32), n)
            for r in rows if r[0] == "learner"]
    w = np.array([1.5, -2.5, 3.25, -0.0], np.float32)
    rc, out = orc.decode_apply(msgs, n, w, 0.5)
    assert rc == 0 and out.view(np.uint32).tolist() == w.view(np.uint32).tolist()


@pytest.mark.parametrize("seed", range(6))
def test_decode_apply_random_learners(orc, seed):
    rng = np.random.default_rng(900 + seed)
    n, W = int(rng.integers(1, 3000)), int(rng.integers(1, 6))
    lr = float(np.float32(rng.choice([0.1, 0.37, 1.0, 3.0]))) if seed else float(np.float32(0.37))
    msgs, parts = [], []
    for _ in range(W):
        k = int(rng.integers(0, min(n, 300) + 1))
        idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
        val = (rng.standard_normal(k) * 10.0 ** rng.integers(-3, 3, k)).astype(np.float32)
        msgs.append(orc.encode(idx, val, n))
        parts.append((idx, val))
    w = (rng.standard_normal(n) * 10.0 ** rng.integers(-3, 3, n)).astype(np.float32)
    w[rng.random(n) < 0.05] = -0.0
    exp, s = _apply_expected(w, parts, lr)
    rc, out = orc.decode_apply(msgs, n, w, lr)
    assert rc == 0
    assert out.view(np.uint32).tolist() == exp.view(np.uint32).tolist()
    # the single rounding matters on these inputs: a separate multiply and subtract differs
    if seed == 0:
        two = [X.add_f32(w[i], -X.mul_f32(lr, t)) for i, t in s.items()]
        assert any(X.bits(a) != X.bits(exp[i]) for a, i in zip(two, s.keys()))


def test_decode_apply_closed_forms(orc):
    rng = np.random.default_rng(5)
    n = 2000
    idx = np.sort(rng.choice(n, 100, replace=False)).astype(np.uint32)
    val = rng.standard_normal(100).astype(np.float32)
    msg = orc.encode(idx, val, n)
    w = rng.standard_normal(n).astype(np.float32)
    w[::7] = -0.0
    untouched = np.setdiff1d(np.arange(n), idx)
    rc, out = orc.decode_apply([msg], n, w, 0.0)  # lr = +0: no value moves (a touched -0 may
    assert rc == 0 and np.array_equal(out, w)     # become +0: -0*t + -0 is +0 for t < 0)
    assert out[untouched].view(np.uint32).tolist() == w[untouched].view(np.uint32).tolist()
    rc, out = orc.decode_apply([msg], n, np.zeros(n, np.float32), 1.0)  # from 0, lr 1: -sum
    exp = np.zeros(n, np.float32)
    exp[idx] = -val
    assert rc == 0 and out.view(np.uint32).tolist() == exp.view(np.uint32).tolist()
    rc, out = orc.decode_apply([msg], n, w, 2.0)  # untouched entries keep their bits, -0 too
    assert out[untouched].view(np.uint32).tolist() == w[untouched].view(np.uint32).tolist()


def test_decode_apply_rejects(orc):
    n = 100
    msg = orc.encode(np.array([3], np.uint32), np.array([1.0], np.float32), n)
    w = np.full(n, 2.0, np.float32)
    for lr in (-0.0, -1.0, math.inf, math.nan):
        rc, out = orc.decode_apply([msg], n, w, lr)
        assert rc == orc.EINVAL and np.all(out == 2.0)
    rc, out = orc.decode_apply([msg, b"XGC1" + msg[4:]], n, w, 1.0)
    assert rc == orc.ECORRUPT and np.all(out == 2.0)


# --------------------------------------------------------------- integer-valued messages
# Reading of "AdaComp ..." (abstract: sparse and quantized residues) and of the IntSGD page
# (abstract: scale by a shared number, round to integers): see tests/golden/codec_quant8.txt.
def golden_quant(name):
    rows = read_golden(name)
    kv = {t: v for t, v in rows if t in ("n", "alpha", "bits", "size")}
    n, bits, size = kv["n"][0], kv["bits"][0], kv["size"][0]
    alpha = X.from_bits(kv["alpha"][0])
    ent = [v for t, v in rows if t == "entry"]
    tok = [v for t, v in rows if t == "token"]
    T = len(tok)
    msg = struct.pack("<4sHHQQII", b"DGC1", 2, bits, n, T, kv["alpha"][0], len(ent))
    fmt = "<b" if bits == 8 else "<h"
    msg += b"".join(struct.pack(fmt, t[1]) for t in tok)
    msg += b"\0" * (len(msg) % 2)
    msg += b"".join(struct.pack("<H", t[0]) for t in tok)
    return n, bits, alpha, ent, msg, size


@pytest.mark.parametrize("name", ["codec_quant8.txt", "codec_quant16.txt"])
def test_quant_golden(orc, name):
    n, bits, alpha, ent, msg, size = golden_quant(name)
    assert len(msg) == size
    idx = np.array([e[0] for e in ent], np.uint32)
    val = np.array([e[1] for e in ent], np.uint32).view(np.float32)
    v = np.full(n, 9.0, np.float32)
    rc, out, v2 = orc.encode_quant(idx, val, n, alpha, bits, v)
    assert rc == 0 and out == msg
    assert [X.bits(v2[e[0]]) for e in ent] == [e[3] for e in ent]
    rest = np.setdiff1d(np.arange(n), idx)
    assert np.all(v2[rest] == 9.0)  # only sent entries take their remainder back
    rc, dense = orc.decode_accumulate_quant([msg], n, bits, alpha)
    assert rc == 0
    exp = np.zeros(n, np.float32)
    exp[idx] = np.array([e[4] for e in ent], np.uint32).view(np.float32)
    assert dense.view(np.uint32).tolist() == exp.view(np.uint32).tolist()


def _quant_expected(val, alpha, bits):
    """q and residual from the definition, in exact rational arithmetic."""
    Q = 2 ** (bits - 1) - 1
    p = X.mul_f32(alpha, val)
    if math.isnan(float(p)):
        q = 0
    else:
        q = int(np.rint(np.float64(p)))  # p is a binary32 value: rint in binary64 is exact
        q = max(-Q, min(Q, q))
    deq = X.round_f32(Fraction(q) / Fraction(float(alpha))) if q else np.float32(0.0)
    return q, X.add_f32(val, -deq)


@pytest.mark.parametrize("seed", range(8))
def test_quant_random_against_definition(orc, seed):
    rng = np.random.default_rng(1200 + seed)
    n = int(rng.integers(1, 200_000))
    k = int(rng.integers(0, min(n, 400) + 1))
    bits = 8 if seed % 2 else 16
    alpha = np.float32(rng.choice([1.0, 3.0, 1000.0, 0.37, 2.0 ** 20]))
    idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
    val = (rng.standard_normal(k) * 10.0 ** rng.integers(-6, 3, k)).astype(np.float32)
    val[rng.random(k) < 0.05] = np.float32(-0.0)
    rc, msg, v = orc.encode_quant(idx, val, n, alpha, bits, np.zeros(n, np.float32))
    assert rc == 0
    T = struct.unpack_from("<Q", msg, 16)[0]  # the size follows from T and b
    assert len(msg) == 32 + T * bits // 8 + (T * bits // 8) % 2 + 2 * T
    Q = 2 ** (bits - 1) - 1
    qs = []
    for j, x in enumerate(val):
        q, r = _quant_expected(x, alpha, bits)
        qs.append(q)
        assert X.bits(v[idx[j]]) == X.bits(r)
        if abs(q) < Q:  # not clamped: the remainder is exact, q/alpha + r == v
            deq = Fraction(float(X.round_f32(Fraction(q) / Fraction(float(alpha))))) if q else 0
            assert deq + Fraction(float(r)) == Fraction(float(x))
    # the message's integers, read back by walking the layout
    T = struct.unpack_from("<Q", msg, 16)[0]
    vals = struct.unpack_from(f"<{T}{'b' if bits == 8 else 'h'}", msg, 32)
    at = 32 + T * bits // 8
    at += at % 2
    runs = struct.unpack_from(f"<{T}H", msg, at)
    got = [q for q, r in zip(vals, runs) if r != 0xFFFF]
    assert got == qs


def test_quant_nan_and_infinities(orc):
    n = 10
    idx = np.array([1, 2, 3], np.uint32)
    val = np.array([np.nan, np.inf, -np.inf], np.float32)
    rc, msg, v = orc.encode_quant(idx, val, n, 2.0, 8, np.zeros(n, np.float32))
    assert rc == 0
    assert struct.unpack_from("<3b", msg, 32) == (0, 127, -127)


@pytest.mark.parametrize("seed", range(4))
def test_quant_decode_sums_integers_in_any_order(orc, seed):
    rng = np.random.default_rng(1300 + seed)
    n, W, bits = 5000, int(rng.integers(2, 700)), 16
    alpha = np.float32(rng.choice([0.5, 3.0, 1000.0]))
    msgs, S, touched = [], {}, set()
    for _ in range(W):
        k = int(rng.integers(0, 50))
        idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
        val = (rng.choice([-1, 1], k) * rng.integers(0, 40000, k) / float(alpha)).astype(np.float32)
        rc, m, _ = orc.encode_quant(idx, val, n, alpha, bits)
        assert rc == 0
        msgs.append(m)
        for j, x in enumerate(val):
            q, _ = _quant_expected(x, alpha, bits)
            S[int(idx[j])] = S.get(int(idx[j]), 0) + q
            touched.add(int(idx[j]))
    base = rng.standard_normal(n).astype(np.float32)
    base[::5] = np.float32(-0.0)
    for acc in (False, True):
        exp = base.copy() if acc else np.zeros(n, np.float32)
        for i in touched:
            x = X.round_f32(Fraction(float(X.round_f32(Fraction(S[i])))) / Fraction(float(alpha)))
            exp[i] = X.add_f32(exp[i], x) if acc else x
        rc, dense = orc.decode_accumulate_quant(msgs, n, bits, alpha, dense=base, accumulate=acc)
        assert rc == 0 and dense.view(np.uint32).tolist() == exp.view(np.uint32).tolist()
        perm = [msgs[i] for i in rng.permutation(W)]  # integer sums: the order cannot matter
        rc, dense2 = orc.decode_accumulate_quant(perm, n, bits, alpha, dense=base, accumulate=acc)
        assert rc == 0 and dense2.view(np.uint32).tolist() == exp.view(np.uint32).tolist()
    lr = 0.37
    rc, w = orc.decode_apply_quant(msgs, n, bits, alpha, base, lr)
    exp = base.copy()
    for i in touched:
        t = X.round_f32(Fraction(float(X.round_f32(Fraction(S[i])))) / Fraction(float(alpha)))
        exp[i] = X.fma_f32(np.float32(-lr), t, base[i])
    assert rc == 0 and w.view(np.uint32).tolist() == exp.view(np.uint32).tolist()


def test_quant_rejects(orc):
    n = 100
    idx, val = np.array([3, 7], np.uint32), np.array([1.0, -2.0], np.float32)
    for alpha, bits in ((0.0, 8), (-1.0, 8), (math.inf, 8), (math.nan, 16), (1.0, 4), (1.0, 32)):
        assert orc.encode_quant(idx, val, n, alpha, bits)[0] == orc.EINVAL
    rc, m, _ = orc.encode_quant(idx, val, n, 2.0, 8)
    assert orc.decode_accumulate_quant([m], n, 8, 2.0)[0] == 0
    assert orc.decode_accumulate_quant([m], n, 8, 4.0)[0] == orc.ECORRUPT   # another alpha
    assert orc.decode_accumulate_quant([m], n, 16, 2.0)[0] == orc.ECORRUPT  # another width
    v1 = orc.encode(idx, val, n)
    assert orc.decode_accumulate_quant([m, v1], n, 8, 2.0)[0] == orc.ECORRUPT  # a float message
    assert orc.decode_accumulate([m], n)[0] == orc.ECORRUPT                     # and the reverse
    assert orc.decode_accumulate_quant([m + b"\0\0\0\0"], n, 8, 2.0)[0] == orc.ECORRUPT
    assert orc.decode_accumulate_quant([m], n, 8, -2.0)[0] == orc.EINVAL
    assert orc.decode_accumulate_quant([m], n, 12, 2.0)[0] == orc.EINVAL
    assert orc.decode_apply_quant([m], n, 8, 2.0, np.zeros(n, np.float32), -1.0)[0] == orc.EINVAL
    base = np.full(n, 5.0, np.float32)
    rc, d = orc.decode_accumulate_quant([m, m[:-4]], n, 8, 2.0, dense=base, accumulate=True)
    assert rc == orc.ECORRUPT and np.all(d == 5.0)
    assert orc.decode_accumulate_quant([m] * 65537, n, 8, 2.0)[0] == orc.EUNSUPPORTED


# ------------------------------------------------------------- ScaleComp: leak and shared set
# Readings of the ScaleComp abstract (first page): the low-pass filter in the local accumulation
# is a leaky accumulator v <- fma(leak, v, u); the commutative compressor sends every learner's
# accumulator at one shared index set, so the messages add up position by position.
def _exact_accumulate_leak(g, u, v, m, leak):
    un = np.empty_like(u)
    vn = np.empty_like(v)
    for i in range(g.size):
        un[i] = X.fma_f32(m, u[i], g[i])
        vn[i] = X.fma_f32(leak, v[i], un[i])
    return un, vn


@pytest.mark.parametrize("seed", range(6))
def test_accumulate_leak_is_single_rounding_fma(orc, seed):
    rng = np.random.default_rng(3000 + seed)
    for _ in range(200):
        g, u, v = (np.float32(x) for x in rng.standard_normal(3) * 10.0 ** rng.integers(-6, 6, 3))
        m = np.float32(rng.choice([0.9, 0.0]))
        leak = np.float32(rng.choice([0.5, 0.9, 0.999, 1.0, 0.1]))
        uo, vo = orc.accumulate_leak(g, u, v, m, leak)
        ue = X.fma_f32(m, u, g)
        assert X.bits(uo) == X.bits(ue) and X.bits(vo) == X.bits(X.fma_f32(leak, v, ue))
        if leak == 1.0:  # fma(1, v, u) is the plain sum: DGC's accumulation
            assert X.bits(vo) == X.bits(orc.accumulate_one(g, u, v, m)[1])


@pytest.mark.parametrize("seed", range(8))
def test_leak_in_compress(orc, seed):
    rng = np.random.default_rng(3100 + seed)
    n = int(rng.integers(1, 3000))
    off = _random_segments(rng, n)
    g, u, v = (rng.standard_normal(n).astype(np.float32) for _ in range(3))
    mode = [orc.EXACT, orc.SAMPLED, orc.ADACOMP][seed % 3]
    # leak 0 (off) and leak 1 give the same step, bit for bit
    outs = []
    for leak in (0.0, 1.0):
        uu, vv = u.copy(), v.copy()
        idx, val, _ = orc.compress(g, uu, vv, off, orc.make_params(mode, 0.99, 0.9, seed=3,
                                                                   bin_size=16, leak=leak))
        outs.append((idx, val, uu, vv))
    assert all(np.array_equal(a.view(np.uint32), b.view(np.uint32))
               for a, b in zip(outs[0][1:], outs[1][1:])) and np.array_equal(outs[0][0], outs[1][0])
    # a real leak: the accumulator follows the definition, the selection runs on it
    leak = np.float32(0.75)
    un, vn = _exact_accumulate_leak(g, u, v, np.float32(0.9), leak)
    uu, vv = u.copy(), v.copy()
    idx, val, _ = orc.compress(g, uu, vv, off, orc.make_params(orc.EXACT, 0.99, 0.9,
                                                               mask_momentum=False, leak=leak))
    exp_idx = []
    for a, b in zip(off[:-1], off[1:]):
        k = orc.count(int(b - a), orc.ppb(1 - 0.99))
        exp_idx += [int(a) + i for i in brute_topk(vn[a:b], k)]
    assert sorted(exp_idx) == idx.tolist()
    assert [X.bits(x) for x in val] == [X.bits(vn[i]) for i in idx]
    vn[idx] = 0.0
    assert vv.view(np.uint32).tolist() == vn.view(np.uint32).tolist()
    assert uu.view(np.uint32).tolist() == un.view(np.uint32).tolist()


@pytest.mark.parametrize("seed", range(10))
def test_compress_shared_matches_definition(orc, seed):
    rng = np.random.default_rng(3200 + seed)
    n = int(rng.integers(1, 2000))
    off = _random_segments(rng, n)
    g, u, v = (_tricky(rng, n, seed % 4) for _ in range(3))
    k = int(rng.integers(0, n + 1))
    idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
    leak = np.float32(rng.choice([1.0, 0.9]))
    mask = bool(seed % 2)
    p = orc.make_params(orc.SAMPLED, 0.999, 0.9, mask_momentum=mask, leak=leak)
    un, vn = _exact_accumulate_leak(g, u, v, np.float32(0.9), leak)
    uu, vv = u.copy(), v.copy()
    rc, val = orc.compress_shared(g, uu, vv, off, p, idx)
    assert rc == 0
    assert [X.bits(x) for x in val] == [X.bits(vn[i]) for i in idx]
    vn[idx] = 0.0
    if mask:
        un[idx] = 0.0
    assert vv.view(np.uint32).tolist() == vn.view(np.uint32).tolist()
    assert uu.view(np.uint32).tolist() == un.view(np.uint32).tolist()


@pytest.mark.parametrize("seed", range(6))
def test_compress_shared_at_own_selection_is_compress(orc, seed):
    # the learner that chose S, sending at S, takes exactly the step dgc_compress takes
    rng = np.random.default_rng(3300 + seed)
    n = int(rng.integers(100, 5000))
    off = _random_segments(rng, n)
    p = orc.make_params([orc.EXACT, orc.SAMPLED, orc.ADACOMP][seed % 3], 0.99, 0.9, clip_norm=1.0,
                        seed=seed, bin_size=50, leak=0.9)
    g, u, v = (rng.standard_normal(n).astype(np.float32) for _ in range(3))
    ua, va, ub, vb = u.copy(), v.copy(), u.copy(), v.copy()
    idx, val, _ = orc.compress(g, ua, va, off, p)
    rc, val2 = orc.compress_shared(g, ub, vb, off, p, idx)
    assert rc == 0 and val.view(np.uint32).tolist() == val2.view(np.uint32).tolist()
    assert np.array_equal(ua.view(np.uint32), ub.view(np.uint32))
    assert np.array_equal(va.view(np.uint32), vb.view(np.uint32))


def test_sum_shared_order_and_definition(orc):
    rows = read_golden("decode_order.txt")  # 1e8, 1, -1e8 at one position: ordered sum 0
    vals = [np.array([np.uint32(r[1][1])], np.uint32).view(np.float32) for r in rows
            if r[0] == "learner"]
    rc, out = orc.sum_shared(vals)
    assert rc == 0 and X.bits(out[0]) == 0
    rng = np.random.default_rng(7)
    vals = [(rng.standard_normal(500) * 10.0 ** rng.integers(-3, 3, 500)).astype(np.float32)
            for _ in range(9)]
    exp = np.zeros(500, np.float32)
    for a in vals:
        exp = np.array([X.add_f32(x, y) for x, y in zip(exp, a)], np.float32)
    rc, out = orc.sum_shared(vals)
    assert rc == 0 and out.view(np.uint32).tolist() == exp.view(np.uint32).tolist()


def test_shared_rejects(orc):
    n = 50
    g = np.ones(n, np.float32)
    off = np.array([0, n])
    for leak in (-0.5, 1.5, math.nan):
        p = orc.make_params(orc.EXACT, 0.9, 0.9, leak=leak)
        assert orc.compress_shared(g, np.zeros(n, np.float32), np.zeros(n, np.float32), off, p,
                                   np.array([1], np.uint32))[0] == orc.EINVAL
    p = orc.make_params(orc.EXACT, 0.9, 0.9)
    for bad in ([3, 3], [4, 2], [n]):
        u, v = np.zeros(n, np.float32), np.ones(n, np.float32)
        assert orc.compress_shared(g, u, v, off, p, np.array(bad, np.uint32))[0] == orc.EINVAL
        assert np.all(v == 1.0)  # nothing changes on a rejected call
    with pytest.raises(RuntimeError):
        orc.compress(g, np.zeros(n, np.float32), np.zeros(n, np.float32), off,
                     orc.make_params(orc.EXACT, 0.9, 0.9, leak=1.5))
