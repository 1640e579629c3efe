"""Parity of the CUDA path (through the C ABI) with the oracle, element by element.

Integer and index results (selected sets, encoded bytes, counts, keys) must be bit-identical.
The floating-point results are too: the kernels perform the same binary32/binary64 operations
in the same order as the oracle (fma for u, one rounding per add, the fixed clipping sum), so
u, v, the sent values and the decoded sums are compared bitwise -- tighter than the 1e-6 /
1-ulp / 1e-5 tolerances the workloads allow.
"""
import math

import numpy as np
import pytest
import torch

import gpu_helpers
import oracle
import sparsified_gradient_compression_gb300 as dgc
import workloads
from conftest import read_golden
from gpu_helpers import (Compressor, Encoder, decode, decode_apply, decode_apply_quant,
                         decode_quant, dev_f32, encode_quant, host_f32)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    dgc.build()
    dgc.lib()
    oracle.lib()


def dev_idx(idx):
    """uint32 indices plus one spare entry, as a device int32 tensor."""
    a = np.zeros(idx.size + 1, np.uint32)
    a[: idx.size] = idx
    return torch.from_numpy(a.view(np.int32)).cuda()


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def same_bits(a, b):
    return np.array_equal(bits(a), bits(b))


def params_pair(**kw):
    return dgc.make_params(**kw), oracle.make_params(**kw)


def run_steps(grads, seg_off, steps, check_state=True, u0=None, v0=None, **kw):
    """Run `steps` compressor steps on both sides; compare outputs, state and stats each step."""
    n = int(seg_off[-1])
    pd, po = params_pair(**kw)
    comp = Compressor(n, seg_off, pd)
    u_h = np.zeros(n, np.float32) if u0 is None else u0.copy()
    v_h = np.zeros(n, np.float32) if v0 is None else v0.copy()
    u_d, v_d = dev_f32(u_h), dev_f32(v_h)
    outs = []
    for t in range(steps):
        g = grads(t)
        comp(dev_f32(g), u_d, v_d)
        assert comp.status_code() == 0
        idx, val, st = comp.results()
        oidx, oval, ost = oracle.compress(g, u_h, v_h, seg_off, po)
        assert idx.size == oidx.size, f"step {t}: |S| {idx.size} vs {oidx.size}"
        assert np.array_equal(idx, oidx), f"step {t}: index sets differ"
        assert same_bits(val, oval), f"step {t}: sent values differ"
        if check_state:
            assert same_bits(host_f32(v_d), v_h), f"step {t}: residual v differs"
            assert same_bits(host_f32(u_d), u_h), f"step {t}: momentum u differs"
        for s, o in enumerate(ost):
            got = st[s]
            assert got["k"] == o["k"] and got["sent"] == o["sent"], (t, s)
            assert got["candidates"] == o["candidates"], (t, s)
            assert got["thresh_key"] == o["thresh_key"], (t, s)
            assert got["sample_key"] == o["sample_key"], (t, s)
            assert got["reselected"] == o["reselected"], (t, s)
            assert bits(np.float32(got["clip_scale"])) == bits(o["clip_scale"]), (t, s)
            # the squared norm itself, bitwise (the binary32 scale hides most ulps of S)
            gs, os_ = float(got["clip_sumsq"]), o["clip_sumsq"]
            assert (gs == os_ or (math.isnan(gs) and math.isnan(os_))), (t, s, gs, os_)
        outs.append((idx, val))
    return outs, u_d, v_d


# ------------------------------------------------------------------- the five workloads
def test_single_tensor_1m_exact_three_steps_and_codec():
    n = 1_048_576
    off = np.array([0, n])
    outs, _, _ = run_steps(lambda t: workloads.gradient("single", t), off, 3,
                           mode=dgc.SELECT_EXACT, sparsity=0.999, momentum=0.9)
    for idx, val in outs:
        assert idx.size == 1049
        enc = Encoder(idx.size, n)
        cnt = torch.tensor([idx.size], dtype=torch.int64, device="cuda")
        enc(torch.from_numpy(idx.view(np.int32)).cuda(), dev_f32(val), cnt)
        msg = enc.message()
        assert msg == oracle.encode(idx, val, n)
        rc, dense = decode([msg], n)
        orc_rc, odense = oracle.decode_accumulate([msg], n)
        assert rc == 0 and orc_rc == 0
        assert same_bits(host_f32(dense), odense)


@pytest.mark.slow
def test_resnet50_161_tensors_clip_exact_ten_steps():
    off = workloads.resnet50_segments()
    run_steps(lambda t: workloads.gradient("resnet50", t), off, 10, mode=dgc.SELECT_EXACT,
              sparsity=0.999, momentum=0.9, clip_norm=1.0)


@pytest.mark.slow
def test_deepspeech_sampled_six_segments():
    off = workloads.deepspeech_segments()
    # the workload's 10 steps, every step's selection, values, u, v and statistics bitwise
    outs, _, _ = run_steps(lambda t: workloads.gradient("deepspeech", t), off, 10,
                           mode=dgc.SELECT_SAMPLED, sparsity=0.999, momentum=0.9,
                           sample_ratio=0.01, reselect_factor=1.3, seed=1234)
    # the message size the DGC review prints for DeepSpeech: 0.74 MB
    idx, val = outs[-1]
    assert abs(len(oracle.encode(idx, val, int(off[-1]))) / 1e6 - 0.74) / 0.74 < 0.1


@pytest.mark.slow
def test_bucket_1g_sampled_warmup_schedule():
    n = 1 << 30
    off = np.array([0, n])
    pd, po = params_pair(mode=dgc.SELECT_SAMPLED, sparsity=0.75, momentum=0.9, sample_ratio=0.01,
                         reselect_factor=1.3, seed=99)
    u_h = np.zeros(n, np.float32)
    v_h = np.zeros(n, np.float32)
    u_d = torch.zeros(n, dtype=torch.float32, device="cuda")
    v_d = torch.zeros(n, dtype=torch.float32, device="cuda")
    for t, s in enumerate(workloads.WARMUP_SPARSITY):
        pd.sparsity = po.sparsity = s
        comp = Compressor(n, off, pd)
        g = workloads.gradient("bucket1g", t)
        comp(dev_f32(g), u_d, v_d)
        assert comp.status_code() == 0
        idx, val, st = comp.results()
        oidx, oval, ost = oracle.compress(g, u_h, v_h, off, po)
        assert np.array_equal(idx, oidx) and same_bits(val, oval), f"step {t}"
        assert st[0]["sample_key"] == ost[0]["sample_key"]
        assert st[0]["candidates"] == ost[0]["candidates"]
        assert same_bits(host_f32(v_d), v_h) and same_bits(host_f32(u_d), u_h), f"step {t}"
        del comp
        torch.cuda.empty_cache()


@pytest.mark.slow
def test_bucket_1g_adacomp_bins_of_1000():
    # the AdaComp bench configuration at full size: 2^30 entries, bins of 1000, two steps
    n = 1 << 30
    off = np.array([0, n])
    pd, po = params_pair(mode=dgc.SELECT_ADACOMP, momentum=0.9, bin_size=1000)
    u_h = np.zeros(n, np.float32)
    v_h = np.zeros(n, np.float32)
    u_d = torch.zeros(n, dtype=torch.float32, device="cuda")
    v_d = torch.zeros(n, dtype=torch.float32, device="cuda")
    comp = Compressor(n, off, pd)
    for t in range(2):
        g = workloads.gradient("bucket1g", t)
        comp(dev_f32(g), u_d, v_d)
        assert comp.status_code() == 0
        idx, val, st = comp.results()
        oidx, oval, ost = oracle.compress(g, u_h, v_h, off, po)
        assert np.array_equal(idx, oidx) and same_bits(val, oval), f"step {t}"
        assert st[0]["sent"] == ost[0]["sent"]
        assert same_bits(host_f32(v_d), v_h) and same_bits(host_f32(u_d), u_h), f"step {t}"
    del comp
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_bench_pipeline_1g_in_cuda_graphs():
    # the bench's own step on the 1B bucket in the configuration it times: the warm-up schedule
    # call by call, then compress and encode as CUDA graph replays at 99.9% on gradient buffers
    # resident in HBM; every step's selection, state, message and decoded dense array against
    # the oracle
    import bench

    n = 1 << 30
    off = np.array([0, n])
    sched = list(workloads.WARMUP_SPARSITY[:4]) + [0.999]
    kw = dict(mode=dgc.SELECT_SAMPLED, momentum=0.9, sample_ratio=0.01, reselect_factor=1.3,
              seed=bench.SEED)
    pd = [dgc.make_params(sparsity=s, **kw) for s in sched]
    po = [oracle.make_params(sparsity=s, **kw) for s in sched]
    pipe = bench.Pipeline(n, pd, torch.device("cuda", 0))
    hosts = [workloads.gradient("bucket1g", step=i, seed=0, n=n) for i in range(2)]
    pool = [torch.from_numpy(h).cuda() for h in hosts]
    u_h = np.zeros(n, np.float32)
    v_h = np.zeros(n, np.float32)

    def check(t, g_h, p_o):
        oidx, oval, _ = oracle.compress(g_h, u_h, v_h, off, p_o)
        assert dgc.dgc_read_status(pipe.status) == 0
        c = int(pipe.out_count.item())
        assert np.array_equal(pipe.out_idx[:c].cpu().numpy().view(np.uint32), oidx), t
        assert same_bits(pipe.out_val[:c].cpu().numpy(), oval), t
        assert same_bits(host_f32(pipe.v), v_h) and same_bits(host_f32(pipe.u), u_h), t
        msg = pipe.msg[: int(pipe.msg_bytes.item())].cpu().numpy().tobytes()
        assert msg == oracle.encode(oidx, oval, n), t
        _, odense = oracle.decode_accumulate([msg], n)
        assert same_bits(host_f32(pipe.dense), odense), t

    for i in range(4):  # the warm-up schedule, call by call
        pipe.step(pool[i % 2], pd[i])
        torch.cuda.synchronize()
        check(i, hosts[i % 2], po[i])
    graphs = [pipe.capture(g, pd[-1]) for g in pool]
    torch.cuda.synchronize()
    for i in range(4, 7):  # 99.9%, replayed
        pipe.step(pool[i % 2], pd[-1], None, graphs[i % 2])
        torch.cuda.synchronize()
        check(i, hosts[i % 2], po[-1])
    del pipe, pool, graphs
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_aggregation_64_learners():
    n, W, k = 25_557_032, 64, 25_558
    for step in range(5):
        msgs_gpu, msgs_orc = [], []
        for w in range(W):
            rng = np.random.Generator(np.random.PCG64([5, step, w]))
            idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
            val = (rng.standard_normal(k) * 0.01).astype(np.float32)
            enc = Encoder(k, n)
            enc(torch.from_numpy(idx.view(np.int32)).cuda(), dev_f32(val),
                torch.tensor([k], dtype=torch.int64, device="cuda"))
            msgs_gpu.append(enc.message())
            msgs_orc.append(oracle.encode(idx, val, n))
            assert msgs_gpu[-1] == msgs_orc[-1]
        rc, dense = decode(msgs_gpu, n)
        orc_rc, odense = oracle.decode_accumulate(msgs_orc, n)
        assert rc == 0 and orc_rc == 0
        assert same_bits(host_f32(dense), odense)
        # the same messages as one SGD step on weights (1/W folded into lr)
        w0 = np.random.Generator(np.random.PCG64([6, step])).standard_normal(n).astype(np.float32)
        rc, w_gpu = decode_apply(msgs_gpu, n, w0, 0.1 / W)
        orc_rc, w_orc = oracle.decode_apply(msgs_orc, n, w0, np.float32(0.1 / W))
        assert rc == 0 and orc_rc == 0
        assert same_bits(w_gpu, w_orc)
        if step < 2:  # the same learners' entries as 16-bit integer messages
            qmsgs = []
            for w in range(W):
                rng = np.random.Generator(np.random.PCG64([5, step, w]))
                idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
                val = (rng.standard_normal(k) * 0.01).astype(np.float32)
                rc, m, _ = oracle.encode_quant(idx, val, n, 1e5, 16)
                assert rc == 0
                qmsgs.append(m)
            rc, dq = decode_quant(qmsgs, n, 16, 1e5)
            orc_rc, odq = oracle.decode_accumulate_quant(qmsgs, n, 16, 1e5)
            assert rc == 0 and orc_rc == 0 and same_bits(dq, odq)
            rc, wq = decode_apply_quant(qmsgs, n, 16, 1e5, w0, 0.1 / W)
            orc_rc, owq = oracle.decode_apply_quant(qmsgs, n, 16, 1e5, w0, np.float32(0.1 / W))
            assert rc == 0 and orc_rc == 0 and same_bits(wq, owq)


@pytest.mark.slow
def test_aggregation_64_learners_end_to_end():
    # The aggregation workload as its recipe states it, 5 steps: each of the 64 learners runs
    # the compressor (momentum 0.9, exact top-k at 99.9%, k = 25,558) and the encoder on its own
    # seeded gradients; every step's 64 messages are decoded and summed in learner order
    # (dgc_decode_accumulate) and applied as one SGD step (dgc_decode_apply). The oracle runs
    # the same chain, its learners spread over a spawned process pool (its exact top-k sorts all
    # 25.6M entries, ~5 s per learner and step on one core). Compared bitwise: every message,
    # each learner's u and v after the last step (SHA-256 digests), every step's dense sum and
    # updated weights.
    import concurrent.futures as cf
    import hashlib
    import multiprocessing as mp
    import os

    import aggregation_oracle as agg

    n, W, steps = agg.N_LEARNER, 64, 5
    workers = max(1, min(16, os.cpu_count() or 1))
    pool = cf.ProcessPoolExecutor(workers, mp_context=mp.get_context("spawn"))
    try:
        futs = [pool.submit(agg.learner_messages, w, steps, n) for w in range(W)]
        off = np.array([0, n])
        pd = dgc.make_params(mode=dgc.SELECT_EXACT, sparsity=0.999, momentum=0.9)
        comp = Compressor(n, off, pd)
        enc = Encoder(comp.cap, n)
        gpu_msgs = [[None] * W for _ in range(steps)]  # device copies, [step][learner]
        gpu_host = [[None] * W for _ in range(steps)]
        digests = []
        for w in range(W):
            u_d = torch.zeros(n, dtype=torch.float32, device="cuda")
            v_d = torch.zeros(n, dtype=torch.float32, device="cuda")
            for t in range(steps):
                comp(dev_f32(workloads.gradient("learners", t, learner=w, n=n)), u_d, v_d)
                enc(comp.out_idx, comp.out_val, comp.out_count)
                assert comp.status_code() == 0 and dgc.dgc_read_status(enc.status) == 0
                nb = int(enc.out_bytes.item())
                gpu_msgs[t][w] = enc.out[:nb].clone()
                gpu_host[t][w] = gpu_msgs[t][w].cpu().numpy().tobytes()
            digests.append((hashlib.sha256(host_f32(u_d).tobytes()).hexdigest(),
                            hashlib.sha256(host_f32(v_d).tobytes()).hexdigest()))
            del u_d, v_d
        orc = [f.result() for f in futs]
    finally:
        pool.shutdown(cancel_futures=True)
    for w in range(W):
        omsgs, ou, ov = orc[w]
        for t in range(steps):
            assert gpu_host[t][w] == omsgs[t], f"learner {w}, step {t}: messages differ"
        assert digests[w] == (ou, ov), f"learner {w}: u or v differs after {steps} steps"
    ws_bytes = max(dgc.dgc_decode_workspace([len(m) for m in gpu_host[t]], n)
                   for t in range(steps))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dense = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    for t in range(steps):
        sizes = [len(m) for m in gpu_host[t]]
        dgc.dgc_decode_accumulate(gpu_msgs[t], sizes, dense, n, False, status, ws,
                                  ws_bytes=ws_bytes)
        assert dgc.dgc_read_status(status) == 0
        orc_rc, odense = oracle.decode_accumulate([orc[w][0][t] for w in range(W)], n)
        assert orc_rc == 0 and same_bits(host_f32(dense), odense), f"step {t}: dense sum"
        w0 = np.random.Generator(np.random.PCG64([7, t])).standard_normal(n).astype(np.float32)
        w_d = dev_f32(w0)
        dgc.dgc_decode_apply(gpu_msgs[t], sizes, w_d, n, 0.1 / W, status, ws, ws_bytes=ws_bytes)
        assert dgc.dgc_read_status(status) == 0
        orc_rc, w_orc = oracle.decode_apply([orc[w][0][t] for w in range(W)], n, w0,
                                            np.float32(0.1 / W))
        assert orc_rc == 0 and same_bits(host_f32(w_d), w_orc), f"step {t}: SGD step"
        del w_d
    del comp, enc, gpu_msgs, dense, ws
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_learner_compress_full_size():
    # two of the aggregation workload's learners through the whole compressor at full size
    n = 25_557_032
    off = np.array([0, n])
    for learner in (0, 63):
        run_steps(lambda t: workloads.gradient("learners", t, learner=learner), off, 2,
                  mode=dgc.SELECT_EXACT, sparsity=0.999, momentum=0.9)


@pytest.mark.parametrize("mode", [dgc.SELECT_EXACT, dgc.SELECT_SAMPLED])
@pytest.mark.parametrize("mask", [True, False])
def test_candidate_clusters_around_the_speculative_send_limit(mode, mask):
    # Streaming tiles with at most 64 candidates store them as sent and keep their values aside;
    # the emit step puts back the ones the selection leaves out, and other tiles are masked as
    # before. Clusters of 55..75 large entries in 21 tiles put tiles on both sides of that limit
    # (and exact mode's re-selection leaves some candidates out), next to tiles with a few.
    n = 1 << 20
    off = np.array([0, n])
    rng = np.random.default_rng(77 + 2 * mode + mask)

    def grads(t):
        g = workloads.misc([90, mode, int(mask), t], n, 0.01)
        for c, size in enumerate(range(55, 76)):
            tile = 3 + 23 * c
            at = tile * 2048 + np.sort(rng.choice(2048, size=size, replace=False))
            g[at] = np.float32(50.0) * (1 + rng.random(size)).astype(np.float32)
        return g

    run_steps(grads, off, 3, mode=mode, sparsity=0.998, momentum=0.9, mask_momentum=mask,
              sample_ratio=0.01, reselect_factor=1.3, seed=5)


# --------------------------------------------------------------------- shapes and edges
EDGE_N = [1, 3, 15, 17, 4095, 8191, 8192, 8193, 40_000, 100_003]


def _segments(rng, n):
    kind = rng.integers(0, 4)
    if kind == 0:
        return np.array([0, n])
    cuts = np.sort(rng.integers(0, n + 1, int(rng.integers(1, 12))))
    off = np.concatenate([[0], cuts, [n]])
    if kind == 2:  # force empty and length-1 segments
        off = np.concatenate([[0, 0, min(1, n)], cuts, [n, n]])
        off.sort()
    return off.astype(np.int64)


@pytest.mark.parametrize("case", range(40))
def test_exact_edges(case):
    rng = np.random.default_rng(9000 + case)
    n = EDGE_N[case % len(EDGE_N)]
    off = _segments(rng, n)
    sparsity = float(rng.choice([0.0, 0.5, 0.9, 0.99, 0.999, 1.0]))
    kind = case % 3
    scale = float(10.0 ** rng.integers(-4, 1))

    def grads(t):
        r = np.random.default_rng([case, t])
        if kind == 1:  # many ties and zeros
            return r.integers(-2, 3, n).astype(np.float32)
        return (r.standard_normal(n) * scale).astype(np.float32)

    run_steps(grads, off, 3, mode=dgc.SELECT_EXACT, sparsity=sparsity,
              momentum=float(rng.choice([0.0, 0.9])), clip_norm=float(rng.choice([0.0, 0.5])),
              mask_momentum=bool(case % 2))


def _extreme_segment(r, kind, size):
    """Finite binary32 values at the ends of the range, for the clipping sum of squares."""
    if kind == 0:  # subnormals: |x| < 2^-126
        bits_ = r.integers(1, 1 << 23, size).astype(np.uint32)
    elif kind == 1:  # huge: squares far beyond binary32, well inside binary64
        bits_ = r.integers(0x71000000, 0x7F7FFFFF, size, endpoint=True).astype(np.uint32)
    elif kind == 2:  # every exponent, subnormal to the largest finite
        bits_ = r.integers(1, 0x7F7FFFFF, size, endpoint=True).astype(np.uint32)
    else:  # mostly zeros
        bits_ = np.where(r.random(size) < 0.01, r.integers(0x30000000, 0x40000000, size),
                         0).astype(np.uint32)
    bits_ |= (r.integers(0, 2, size).astype(np.uint32) << 31)
    return bits_.view(np.float32)


@pytest.mark.parametrize("case", range(6))
def test_clip_extreme_magnitudes(case):
    # the clip norm's binary64 squares and sums at the edges of the binary32 range: subnormal
    # gradients (no clipping), gradients whose norm overflows binary32, every exponent mixed
    rng = np.random.default_rng(12000 + case)
    sizes = [int(rng.integers(1, 20_000)) for _ in range(5)] + [4096, 12289]
    kinds = [int(rng.integers(0, 4)) for _ in sizes]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    n = int(off[-1])

    def grads(t):
        r = np.random.default_rng([case, t, 3])
        return np.concatenate([_extreme_segment(r, k, z) for k, z in zip(kinds, sizes)])

    run_steps(grads, off, 2, mode=[dgc.SELECT_EXACT, dgc.SELECT_SAMPLED][case % 2],
              sparsity=0.99, momentum=0.9, clip_norm=float([1.0, 1e-3, 3.0][case % 3]),
              sample_ratio=0.1, seed=case)


@pytest.mark.slow
def test_clip_long_tile_ranges():
    # more 4096-entry clipping tiles than 17 per block of the 608-block grid: a warp keeps its
    # window over 16 tiles, then flushes it; the scale changes from tile to tile (rising ramps
    # reopen the window every tile, falling ones keep it), and the segments end mid-range
    n = 45_000_000
    off = np.array([0, 13_000_001, 31_000_000, n], dtype=np.int64)
    tile = np.arange(n, dtype=np.int64) // 4096
    ramp = np.where(tile % 60 < 30, tile % 30, 30 - tile % 30) - 15

    def grads(t):
        r = np.random.default_rng([4242, t])
        return (r.standard_normal(n) * np.exp2(ramp - 8.0)).astype(np.float32)

    run_steps(grads, off, 2, mode=dgc.SELECT_SAMPLED, sparsity=0.999, momentum=0.9,
              clip_norm=1.0, sample_ratio=0.01, seed=3)


@pytest.mark.parametrize("mode", ["exact", "sampled", "adacomp"])
def test_many_segments(mode):
    # ~6000 segments of 1-300 entries around a few large ones: more segments than one wave of
    # on-chip selects, than the staged candidate ranges, and than the plan's 1024-segment passes;
    # streaming, emit and clip tiles that cross dozens of segments
    rng = np.random.default_rng({"exact": 1, "sampled": 2, "adacomp": 3}[mode])
    sizes = list(rng.integers(1, 300, 6000))
    for at, big in ((1000, 40_000), (3000, 120_000), (5999, 70_000)):
        sizes[at] = big
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    n = int(off[-1])
    m = {"exact": dgc.SELECT_EXACT, "sampled": dgc.SELECT_SAMPLED, "adacomp": dgc.SELECT_ADACOMP}
    run_steps(lambda t: workloads.misc([t, 77], n, 0.01), off, 2, mode=m[mode], sparsity=0.99,
              momentum=0.9, clip_norm=0.05, sample_ratio=0.1, seed=5, bin_size=64,
              mask_momentum=True)


@pytest.mark.parametrize("case", range(40))
def test_sampled_edges(case):
    rng = np.random.default_rng(7000 + case)
    n = EDGE_N[case % len(EDGE_N)] * (1 + case % 3)
    off = _segments(rng, n)
    sparsity = float(rng.choice([0.0, 0.5, 0.9, 0.99, 0.999, 1.0]))
    kind = case % 3

    def grads(t):
        r = np.random.default_rng([case, t, 1])
        if kind == 1:  # ties: C much larger than k, so the exact re-selection runs
            return r.integers(-2, 3, n).astype(np.float32)
        return (r.standard_t(3, n) * 1e-3).astype(np.float32)

    run_steps(grads, off, 3, mode=dgc.SELECT_SAMPLED, sparsity=sparsity, momentum=0.9,
              sample_ratio=float(rng.choice([0.01, 0.1, 1.0])), reselect_factor=1.3,
              seed=int(rng.integers(0, 2**63)), mask_momentum=bool(case % 2),
              clip_norm=float(rng.choice([0.0, 1.0])))


@pytest.mark.parametrize("case", range(30))
def test_adacomp_edges(case):
    # AdaComp bin-local selection against the oracle: bins of bin_size entries per segment, the
    # entries at each bin's largest |v| sent (ties included, all-zero bins send nothing)
    rng = np.random.default_rng(11000 + case)
    n = EDGE_N[case % len(EDGE_N)] * (1 + case % 2)
    off = _segments(rng, n)
    L = int(rng.choice([1, 3, 17, 50, 1000, 2048, 5000]))
    kind = case % 3

    def grads(t):
        r = np.random.default_rng([case, t, 2])
        if kind == 1:
            return r.integers(-2, 3, n).astype(np.float32)
        if kind == 2:
            x = (r.standard_normal(n) * 0.01).astype(np.float32)
            x[r.random(n) < 0.5] = 0.0
            return x
        return (r.standard_normal(n) * 0.01).astype(np.float32)

    run_steps(grads, off, 3, mode=dgc.SELECT_ADACOMP, bin_size=L,
              momentum=float(rng.choice([0.0, 0.9])), mask_momentum=bool(case % 2),
              clip_norm=float(rng.choice([0.0, 1.0])))


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 7, 127, 128, 129, 1000, 2047, 2048, 2049, 4096])
def test_adacomp_bin_sizes_one_segment(L):
    # one segment, so every tile but the ragged last one takes the per-lane bin arithmetic; the
    # sizes straddle its branches (under 4, under 128, under the 2048-entry tile)
    n = 3 * 2048 * 5 + 1234
    off = np.array([0, n])
    run_steps(lambda t: (np.random.default_rng([L, t]).standard_normal(n) * 0.01)
              .astype(np.float32), off, 2, mode=dgc.SELECT_ADACOMP, bin_size=L, momentum=0.9)


@pytest.mark.slow
def test_adacomp_resnet50_layout():
    off = workloads.resnet50_segments()
    run_steps(lambda t: workloads.gradient("resnet50", t), off, 3, mode=dgc.SELECT_ADACOMP,
              bin_size=1000, momentum=0.9, clip_norm=1.0)


def test_exact_tight_sample_bound_falls_back():
    # White-box: exact mode bounds the threshold from below with a 1% sample drawn from the same
    # SplitMix64 positions (seed from the params). Putting the only large values exactly at the
    # sampled positions makes that bound admit fewer than k candidates (the draws repeat a few
    # positions), which forces the re-compaction from v. The result must still be exact.
    n, seed = 400_000, 77
    ms = -(-n // 100)
    pos = np.unique([oracle.sample_position(seed, 0, j, n) for j in range(ms)])
    k = -(-n // 100)  # sparsity 0.99
    assert pos.size < k
    g = np.full(n, 1e-6, np.float32)
    g[pos] = 1.0
    run_steps(lambda t: g * np.float32(1 + t), np.array([0, n]), 2, mode=dgc.SELECT_EXACT,
              sparsity=0.99, momentum=0.9, seed=seed)


def test_all_equal_magnitudes_ties_to_lower_index():
    n = 50_000
    g = np.where(np.arange(n) % 2 == 0, np.float32(0.5), np.float32(-0.5)).astype(np.float32)
    for mode in (dgc.SELECT_EXACT, dgc.SELECT_SAMPLED):
        outs, _, _ = run_steps(lambda t: g, np.array([0, n]), 2, mode=mode, sparsity=0.999,
                               momentum=0.0)
        assert outs[0][0].tolist() == list(range(50))


def test_empty_gradient():
    outs, _, _ = run_steps(lambda t: np.zeros(0, np.float32), np.array([0, 0, 0]), 1,
                           mode=dgc.SELECT_EXACT)
    assert outs[0][0].size == 0


# ------------------------------------------------------------------------------- codec
def golden_message(name):
    import struct

    n, entries, tokens = None, [], []
    for tag, vals in read_golden(name):
        if tag == "n":
            n = vals[0]
        elif tag == "entry":
            entries.append(vals)
        elif tag == "token":
            tokens.append(vals)
    T = len(tokens)
    msg = struct.pack("<4sHHQQQ", b"DGC1", 1, 0, n, T, len(entries))
    msg += b"".join(struct.pack("<I", t[1]) for t in tokens)
    msg += b"".join(struct.pack("<H", t[0]) for t in tokens)
    msg += b"\0" * ((-len(msg)) % 4)
    idx = np.array([e[0] for e in entries], np.uint32)
    val = np.array([e[1] for e in entries], np.uint32).view(np.float32)
    return n, idx, val, msg


@pytest.mark.parametrize("name", ["codec_gaps.txt", "codec_single.txt", "codec_odd.txt",
                                  "codec_empty.txt"])
def test_codec_golden_on_gpu(name):
    n, idx, val, msg = golden_message(name)
    enc = Encoder(max(idx.size, 1), n)
    enc(dev_idx(idx), dev_f32(np.append(val, np.float32(0))),
        torch.tensor([idx.size], dtype=torch.int64, device="cuda"))
    assert dgc.dgc_read_status(enc.status) == 0
    assert enc.message() == msg
    rc, dense = decode([msg], n)
    assert rc == 0
    exp = np.zeros(n, np.float32)
    exp[idx] = exp[idx] + val
    assert same_bits(host_f32(dense)[:n], exp)


def test_decode_order_golden_on_gpu():
    rows = read_golden("decode_order.txt")
    n = rows[0][1][0]
    msgs = [oracle.encode(np.array([v[0]], np.uint32), np.array([v[1]], np.uint32).view(np.float32), n)
            for t, v in rows if t == "learner"]
    rc, dense = decode(msgs, n)
    assert rc == 0
    d = host_f32(dense)
    for t, (pos, b) in ((t, v) for t, v in rows if t == "expect"):
        assert int(bits(d[pos:pos + 1])[0]) == b


@pytest.mark.parametrize("seed", range(8))
def test_decode_many_learners_and_accumulate(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 3_000_000))
    W = int(rng.integers(1, 300))
    msgs = []
    for w in range(W):
        k = int(rng.integers(0, min(n, 20_000) + 1))
        idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
        msgs.append(oracle.encode(idx, (rng.standard_normal(k) * 10.0 ** rng.integers(-3, 3, k))
                                  .astype(np.float32), n))
    base = rng.standard_normal(n).astype(np.float32)
    for acc in (False, True):
        rc, dense = decode(msgs, n, dense=dev_f32(base), accumulate=acc)
        orc_rc, odense = oracle.decode_accumulate(msgs, n, dense=base, accumulate=acc)
        assert rc == 0 and orc_rc == 0
        assert same_bits(host_f32(dense), odense)


@pytest.mark.parametrize("case", ["same set, 300 learners", "dense messages, 40 learners",
                                  "half shared, 70 learners", "shared positions, 8 learners",
                                  "crowded and sparse tiles, 12 learners"])
def test_decode_collisions_and_crowded_tiles(case):
    # The worst cases of the ordered multi-message sum: every learner at the same positions (as
    # many values meet at one position as there are learners, across the 256-message groups),
    # messages that send every entry (tens of thousands of tokens per dense tile), and learners
    # that share half of their positions. Dense sums, accumulation and the SGD step, bitwise.
    rng = np.random.default_rng(len(case))
    msgs = []
    if case.startswith("same set"):
        n, W = 20_003, 300
        idx = np.sort(rng.choice(n, size=3000, replace=False)).astype(np.uint32)
        for _ in range(W):
            val = (rng.standard_normal(idx.size) * 10.0 ** rng.integers(-4, 4, idx.size))
            msgs.append(oracle.encode(idx, val.astype(np.float32), n))
    elif case.startswith("dense"):
        n, W = 9_000, 40
        idx = np.arange(n, dtype=np.uint32)
        for _ in range(W):
            val = (rng.standard_normal(n) * 10.0 ** rng.integers(-3, 3, n)).astype(np.float32)
            val[rng.random(n) < 0.05] = np.float32(-0.0)
            msgs.append(oracle.encode(idx, val, n))
    elif case.startswith("shared positions"):
        # few tokens per tile, but in odd tiles 8 learners meet at 12 positions (96 tokens at
        # shared positions) and in even tiles at 4 (32): a warp orders the second kind itself
        # and leaves the first kind to the block decoder
        n, W = 40_000, 8
        common = np.concatenate([t * 4096 + 300 * np.arange(12 if t % 2 else 4)
                                 for t in range(n // 4096)])
        for _ in range(W):
            own = rng.choice(n, size=40, replace=False)
            idx = np.unique(np.concatenate([common, own])).astype(np.uint32)
            val = (rng.standard_normal(idx.size) * 10.0 ** rng.integers(-3, 3, idx.size))
            msgs.append(oracle.encode(idx, val.astype(np.float32), n))
    elif case.startswith("crowded and sparse"):
        # one crowded 16,384-entry tile (36,000 tokens) among sparse ones, shared positions in
        # both, and a ragged last tile: in the SGD step the sum kernel takes the sparse tiles and
        # leaves the crowded one to the round-based kernel
        n, W = 200_003, 12
        crowd = np.arange(3 * 16384, 3 * 16384 + 3000)
        common = rng.choice(n, size=50, replace=False)
        for _ in range(W):
            own = rng.choice(n, size=300, replace=False)
            idx = np.unique(np.concatenate([crowd, common, own])).astype(np.uint32)
            val = (rng.standard_normal(idx.size) * 10.0 ** rng.integers(-3, 3, idx.size))
            msgs.append(oracle.encode(idx, val.astype(np.float32), n))
    else:
        n, W = 100_000, 70
        common = rng.choice(n, size=4000, replace=False)
        for _ in range(W):
            own = rng.choice(n, size=4000, replace=False)
            idx = np.unique(np.concatenate([common, own])).astype(np.uint32)
            val = (rng.standard_normal(idx.size) * 0.01).astype(np.float32)
            msgs.append(oracle.encode(idx, val, n))
    base = rng.standard_normal(n).astype(np.float32)
    for acc in (False, True):
        rc, dense = decode(msgs, n, dense=dev_f32(base), accumulate=acc)
        orc_rc, odense = oracle.decode_accumulate(msgs, n, dense=base, accumulate=acc)
        assert rc == 0 and orc_rc == 0
        assert same_bits(host_f32(dense), odense), acc
    rc, got = decode_apply(msgs, n, base, 0.37)
    orc_rc, exp = oracle.decode_apply(msgs, n, base, np.float32(0.37))
    assert rc == 0 and orc_rc == 0
    assert same_bits(got, exp)


@pytest.mark.parametrize("W", [1, 7, 64, 100])
def test_decode_with_sizes_in_device_memory(W):
    # The _dev decoders read each message's size from device memory and lay their workspace
    # out for host bounds on the sizes; with up to 96 messages the table travels in kernel
    # parameters, with more it is copied. Results must equal the host-size calls bit for bit.
    rng = np.random.default_rng(500 + W)
    n = int(rng.integers(1, 2_000_000))
    msgs = []
    for w in range(W):
        k = 0 if (w % 5 == 3) else int(rng.integers(0, min(n, 30_000) + 1))  # some empty
        idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
        val = (rng.standard_normal(k) * 10.0 ** rng.integers(-3, 3, k)).astype(np.float32)
        msgs.append(oracle.encode(idx, val, n))
    bufs = []
    for m in msgs:
        t = torch.zeros(len(m) + 16, dtype=torch.uint8, device="cuda")
        t[: len(m)] = torch.frombuffer(bytearray(m), dtype=torch.uint8).cuda()
        bufs.append(t)
    sizes = [len(m) for m in msgs]
    bounds = [sz + int(rng.integers(0, 3)) * 6 + int(rng.integers(0, 5)) for sz in sizes]
    dsizes = torch.tensor(sizes, dtype=torch.int64, device="cuda")
    ws_bytes = dgc.dgc_decode_workspace_bound(bounds, n)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    base = rng.standard_normal(n).astype(np.float32)
    for acc in (False, True):
        dense = dev_f32(base)
        dgc.dgc_decode_accumulate_dev(bufs, dsizes, bounds, dense, n, acc, status, ws,
                                      ws_bytes=ws_bytes)
        assert dgc.dgc_read_status(status) == 0
        rc, ref = decode(msgs, n, dense=dev_f32(base), accumulate=acc)
        assert rc == 0 and same_bits(host_f32(dense), host_f32(ref)), acc
        _, odense = oracle.decode_accumulate(msgs, n, dense=base, accumulate=acc)
        assert same_bits(host_f32(dense), odense), acc
    w = dev_f32(base)
    dgc.dgc_decode_apply_dev(bufs, dsizes, bounds, w, n, 0.25, status, ws, ws_bytes=ws_bytes)
    assert dgc.dgc_read_status(status) == 0
    _, w_orc = oracle.decode_apply(msgs, n, base, np.float32(0.25))
    assert same_bits(host_f32(w), w_orc)


def test_decode_with_sizes_in_device_memory_rejects_bad_sizes():
    n = 10_000
    good = oracle.encode(np.array([5, 999, 4000], np.uint32),
                         np.array([1.0, -2.0, 3.5], np.float32), n)
    buf = torch.zeros(len(good) + 64, dtype=torch.uint8, device="cuda")
    buf[: len(good)] = torch.frombuffer(bytearray(good), dtype=torch.uint8).cuda()
    base = np.arange(n, dtype=np.float32)
    for size, bound in ((len(good) + 1, len(good) + 64),  # no message has that size
                        (len(good), len(good) - 6),       # above its bound
                        (len(good) + 4, len(good) + 64),  # 4 tokens by size, the header says 3
                        (31, 64)):                        # shorter than a header
        dsizes = torch.tensor([size], dtype=torch.int64, device="cuda")
        ws_bytes = dgc.dgc_decode_workspace_bound([bound], n)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        dense = dev_f32(base)
        dgc.dgc_decode_accumulate_dev([buf], dsizes, [bound], dense, n, False, status, ws,
                                      ws_bytes=ws_bytes)
        assert dgc.dgc_read_status(status) == dgc.ECORRUPT, (size, bound)
        assert same_bits(host_f32(dense), base), (size, bound)


def test_whole_step_in_one_cuda_graph():
    # compress, encode and a decode that reads the message size from device memory, captured as
    # one CUDA graph and replayed on fresh gradients: every step against the oracle
    n = 1_048_576
    off = np.array([0, n])
    pd, po = params_pair(mode=dgc.SELECT_SAMPLED, sparsity=0.999, momentum=0.9,
                         sample_ratio=0.01, reselect_factor=1.3, seed=21)
    comp = Compressor(n, off, pd)
    enc = Encoder(comp.cap, n)
    u_d = torch.zeros(n, device="cuda")
    v_d = torch.zeros(n, device="cuda")
    g_d = torch.zeros(n, device="cuda")
    dense = torch.zeros(n, device="cuda")
    bound = enc.cap
    ws_bytes = dgc.dgc_decode_workspace_bound([bound], n)
    dws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    dstatus = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        comp(g_d, u_d, v_d)
        enc(comp.out_idx, comp.out_val, comp.out_count)
        dgc.dgc_decode_accumulate_dev([enc.out], enc.out_bytes, [bound], dense, n, False, dstatus,
                                      dws, ws_bytes=ws_bytes)

    u_h = np.zeros(n, np.float32)
    v_h = np.zeros(n, np.float32)

    def check(t, g_h):
        oidx, oval, _ = oracle.compress(g_h, u_h, v_h, off, po)
        assert comp.status_code() == 0 and dgc.dgc_read_status(dstatus) == 0
        msg = enc.message()
        assert msg == oracle.encode(oidx, oval, n), t
        _, odense = oracle.decode_accumulate([msg], n)
        assert same_bits(host_f32(dense), odense), t
        assert same_bits(host_f32(v_d), v_h) and same_bits(host_f32(u_d), u_h), t

    g0 = workloads.gradient("single", 0)
    g_d.copy_(dev_f32(g0))
    step()  # one call outside capture: the sample cache and every lookup are set up
    torch.cuda.synchronize()
    check(0, g0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for t in range(1, 4):
        g = workloads.gradient("single", t)
        g_d.copy_(dev_f32(g))
        graph.replay()
        torch.cuda.synchronize()
        check(t, g)


@pytest.mark.parametrize("acc", [False, True])
def test_decode_single_message_both_modes(acc):
    # one message: the decoder clears dense (unless accumulating) and adds each value once
    rng = np.random.default_rng(77)
    n = 3_000_001
    idx = np.sort(rng.choice(n, size=5000, replace=False)).astype(np.uint32)
    idx[-1] = n - 1
    val = rng.standard_normal(5000).astype(np.float32)
    val[::7] = np.float32(-0.0)
    msg = oracle.encode(idx, val, n)
    base = rng.standard_normal(n).astype(np.float32)
    rc, dense = decode([msg], n, dense=dev_f32(base), accumulate=acc)
    orc_rc, odense = oracle.decode_accumulate([msg], n, dense=base, accumulate=acc)
    assert rc == 0 and orc_rc == 0
    assert same_bits(host_f32(dense), odense)


def test_decode_single_malformed_message_leaves_dense():
    import struct

    n = 1000
    good = oracle.encode(np.array([5, 999], np.uint32), np.array([1.0, 2.0], np.float32), n)
    for bad in (good[:32 + 8] + struct.pack("<H", 999) + good[32 + 10:], b"XGC1" + good[4:]):
        for acc in (False, True):
            rc, dense = decode([bad], n, dense=dev_f32(np.full(n, 7.0, np.float32)),
                               accumulate=acc)
            assert rc == dgc.ECORRUPT
            assert np.all(host_f32(dense) == 7.0)


def test_decode_zero_learners():
    rc, dense = decode([], 1000)
    assert rc == 0 and not host_f32(dense).any()


def test_encode_random_matches_oracle():
    rng = np.random.default_rng(4)
    for _ in range(10):
        n = int(rng.integers(1, 5_000_000))
        k = int(rng.integers(0, min(n, 300_000) + 1))
        idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
        val = rng.standard_normal(k).astype(np.float32)
        enc = Encoder(max(k, 1), n)
        enc(dev_idx(idx), dev_f32(np.append(val, np.float32(0))),
            torch.tensor([k], dtype=torch.int64, device="cuda"))
        assert enc.message() == oracle.encode(idx, val, n)


# ------------------------------------------------------------------ errors and recovery
def test_decode_rejects_malformed_and_leaves_dense():
    import struct

    n = 1000
    good = oracle.encode(np.array([5, 999], np.uint32), np.array([1.0, 2.0], np.float32), n)
    bad = [b"XGC1" + good[4:], good[:4] + struct.pack("<H", 2) + good[6:],
           good[:8] + struct.pack("<Q", n + 1) + good[16:],
           good[:32 + 8] + struct.pack("<H", 999) + good[32 + 10:]]
    for b in bad:
        base = dev_f32(np.full(n, 7.0, np.float32))
        rc, dense = decode([good, b], n, dense=base, accumulate=True)
        assert rc == dgc.ECORRUPT
        assert np.all(host_f32(dense) == 7.0)


def test_encode_rejects_unsorted_and_small_buffer():
    n = 100
    enc = Encoder(3, n)
    enc(torch.tensor([5, 3, 9], dtype=torch.int32, device="cuda"),
        dev_f32(np.ones(3, np.float32)), torch.tensor([3], dtype=torch.int64, device="cuda"))
    assert dgc.dgc_read_status(enc.status) == dgc.EINVAL
    enc = Encoder(3, n)
    enc.cap = 40  # 3 tokens need 32 + 18 + 2 = 52 bytes
    enc(torch.tensor([1, 2, 3], dtype=torch.int32, device="cuda"),
        dev_f32(np.ones(3, np.float32)), torch.tensor([3], dtype=torch.int64, device="cuda"))
    assert dgc.dgc_read_status(enc.status) == dgc.ECAPACITY
    assert int(enc.out_bytes.item()) == 52


def test_bad_segment_table_is_reported_and_state_untouched():
    n = 10_000
    pd = dgc.make_params(sparsity=0.99)
    comp = Compressor(n, np.array([0, 6000, n]), pd)
    comp.seg_off.copy_(torch.tensor([0, 7000, 5000], dtype=torch.int64))  # ends short of n
    u = dev_f32(np.ones(n, np.float32))
    v = dev_f32(np.ones(n, np.float32))
    comp(dev_f32(np.ones(n, np.float32)), u, v)
    assert comp.status_code() == dgc.EINVAL
    assert np.all(host_f32(u) == 1.0) and np.all(host_f32(v) == 1.0)
    assert int(comp.out_count.item()) == 0


def test_bounded_wait_times_out():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dgc.dgc_selftest_wait_timeout(status, 1000)
    assert dgc.dgc_read_status(status) == dgc.ETIMEOUT
    # the context is still usable afterwards
    x = torch.ones(10, device="cuda")
    assert float(x.sum()) == 10.0


def test_checkpoint_resume_is_bitwise():
    # The compressor state is exactly (u, v): restoring a copy reproduces the next step.
    n = 300_000
    off = np.array([0, 100_000, n])
    pd = dgc.make_params(mode=dgc.SELECT_SAMPLED, sparsity=0.99, seed=5)
    comp = Compressor(n, off, pd)
    u = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    gs = [dev_f32(workloads.misc([t], n, 0.01)) for t in range(4)]
    for t in range(3):
        comp(gs[t], u, v)
    ck = (u.clone(), v.clone())
    comp(gs[3], u, v)
    first = comp.results()
    u.copy_(ck[0])
    v.copy_(ck[1])
    comp(gs[3], u, v)
    second = comp.results()
    assert np.array_equal(first[0], second[0]) and same_bits(first[1], second[1])


@pytest.mark.parametrize("damage", ["whole", "past_header", "new_seed"])
def test_workspace_reuse_is_safe(damage):
    # The workspace carries the sample positions from one call to the next, validated by a tag
    # and a checksum. Whatever happens to the workspace between calls, results stay exact.
    n = 1_000_003
    off = np.array([0, 400_000, n])
    kw = dict(mode=dgc.SELECT_SAMPLED, sparsity=0.999, momentum=0.9, sample_ratio=0.05, seed=21)
    pd, po = params_pair(**kw)
    comp = Compressor(n, off, pd)
    u_h = np.zeros(n, np.float32)
    v_h = np.zeros(n, np.float32)
    u_d, v_d = dev_f32(u_h), dev_f32(v_h)
    gen = torch.Generator(device="cuda").manual_seed(5)
    for t in range(4):
        if t == 2:
            if damage == "whole":
                comp.ws.random_(0, 256, generator=gen)
            elif damage == "past_header":  # control words and cache header survive
                comp.ws[4096:].random_(0, 256, generator=gen)
            else:
                pd.seed = po.seed = 22
        g = workloads.misc([t, 3], n, 0.01)
        comp(dev_f32(g), u_d, v_d)
        assert comp.status_code() == 0
        idx, val, st = comp.results()
        oidx, oval, ost = oracle.compress(g, u_h, v_h, off, po)
        assert np.array_equal(idx, oidx) and same_bits(val, oval), f"step {t}"
        assert same_bits(host_f32(v_d), v_h) and same_bits(host_f32(u_d), u_h), f"step {t}"
        assert [s_["sample_key"] for s_ in st] == [o["sample_key"] for o in ost]


def test_runs_are_deterministic():
    n = 2_000_003
    off = np.array([0, 1_000_000, n])
    res = []
    for _ in range(2):
        for mode in (dgc.SELECT_EXACT, dgc.SELECT_SAMPLED):
            comp = Compressor(n, off, dgc.make_params(mode=mode, sparsity=0.999, seed=3))
            u = torch.zeros(n, device="cuda")
            v = torch.zeros(n, device="cuda")
            for t in range(3):
                comp(dev_f32(workloads.misc([t, 1], n, 0.01)), u, v)
            idx, val, _ = comp.results()
            res.append((idx.tobytes(), val.tobytes(), host_f32(u).tobytes(), host_f32(v).tobytes()))
    assert res[0] == res[2] and res[1] == res[3]


def test_launch_counter_counts_kernels():
    before = dgc.dgc_launch_count()
    run_steps(lambda t: workloads.misc([t], 10_000, 1.0), np.array([0, 10_000]), 1)
    assert dgc.dgc_launch_count() > before


@pytest.mark.parametrize("shift", [0, 1, 2, 3])
@pytest.mark.parametrize("n", [5, 4096, 4099, 3 * 4096 + 7, 100_003])
def test_decode_clear_any_alignment(shift, n):
    # one message decoded into a dense view that starts 0-3 floats past a 16-byte boundary: the
    # zeros and values (16-byte stores on a boundary, plain stores otherwise) cover exactly [0, n)
    rng = np.random.default_rng(n + shift)
    k = max(1, n // 100)
    idx = np.sort(rng.choice(n, k, replace=False)).astype(np.uint32)
    val = rng.standard_normal(k).astype(np.float32)
    msg = oracle.encode(idx, val, n)
    buf = torch.full((n + 8,), float("nan"), dtype=torch.float32, device="cuda")
    rc, _ = decode([msg], n, dense=buf[shift:shift + n])
    _, odense = oracle.decode_accumulate([msg], n)
    host = buf.cpu().numpy()
    assert rc == 0 and same_bits(host[shift:shift + n], odense)
    assert np.isnan(host[:shift]).all() and np.isnan(host[shift + n:]).all()


# --------------------------------------------------------------- decode -> plain SGD step
def _weights(rng, n):
    w = (rng.standard_normal(n) * 10.0 ** rng.integers(-3, 3, n)).astype(np.float32)
    w[rng.random(n) < 0.05] = np.float32(-0.0)
    return w


@pytest.mark.parametrize("name", ["codec_gaps.txt", "codec_single.txt", "codec_odd.txt",
                                  "codec_empty.txt", "decode_order.txt"])
def test_decode_apply_goldens(name):
    if name == "decode_order.txt":
        rows = read_golden(name)
        n = rows[0][1][0]
        msgs = [oracle.encode(np.array([v[0]], np.uint32),
                              np.array([v[1]], np.uint32).view(np.float32), n)
                for t, v in rows if t == "learner"]
    else:
        from test_oracle_pins import golden_message
        n, _, _, msg, _ = golden_message(name)
        msgs = [msg]
    w = _weights(np.random.default_rng(3), n)
    rc, got = decode_apply(msgs, n, w, 0.75)
    orc_rc, exp = oracle.decode_apply(msgs, n, w, 0.75)
    assert rc == 0 and orc_rc == 0
    assert same_bits(got, exp)


def test_decode_apply_single_message():
    # one message: no dense sum at all, one fma per received value
    rng = np.random.default_rng(78)
    n = 3_000_001
    idx = np.sort(rng.choice(n, size=5000, replace=False)).astype(np.uint32)
    idx[-1] = n - 1
    val = rng.standard_normal(5000).astype(np.float32)
    val[::7] = np.float32(-0.0)
    msg = oracle.encode(idx, val, n)
    w = _weights(rng, n)
    for lr in (0.37, 0.0, 1.0):
        rc, got = decode_apply([msg], n, w, lr)
        orc_rc, exp = oracle.decode_apply([msg], n, w, np.float32(lr))
        assert rc == 0 and orc_rc == 0
        assert same_bits(got, exp), lr


@pytest.mark.parametrize("seed", range(6))
def test_decode_apply_many_learners(seed):
    rng = np.random.default_rng(300 + seed)
    n = int(rng.integers(1, 3_000_000))
    W = int(rng.integers(2, 200))
    msgs = []
    for _ in range(W):
        k = int(rng.integers(0, min(n, 20_000) + 1))
        idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
        val = (rng.standard_normal(k) * 10.0 ** rng.integers(-3, 3, k)).astype(np.float32)
        val[rng.random(k) < 0.02] = np.float32(-0.0)
        msgs.append(oracle.encode(idx, val, n))
    w = _weights(rng, n)
    lr = float(np.float32(rng.choice([0.01, 0.37, 2.0])))
    rc, got = decode_apply(msgs, n, w, lr)
    orc_rc, exp = oracle.decode_apply(msgs, n, w, lr)
    assert rc == 0 and orc_rc == 0
    assert same_bits(got, exp)


def test_decode_apply_malformed_and_empty():
    import struct

    n = 1000
    good = oracle.encode(np.array([5, 999], np.uint32), np.array([1.0, 2.0], np.float32), n)
    bad = good[:32 + 8] + struct.pack("<H", 999) + good[32 + 10:]  # second position past n
    w = np.full(n, 7.0, np.float32)
    for msgs in ([bad], [good, bad], [bad, good]):
        rc, got = decode_apply(msgs, n, w, 0.5)
        assert rc == dgc.ECORRUPT
        assert np.all(got == 7.0)
    rc, got = decode_apply([], n, w, 0.5)  # no learners: the step is the identity
    assert rc == 0 and same_bits(got, w)
    with pytest.raises(dgc.DGCError) as e:
        decode_apply([good], n, w, -0.0)
    assert e.value.code == dgc.EINVAL


# ------------------------------------------------------------------- integer-valued messages


@pytest.mark.parametrize("name", ["codec_quant8.txt", "codec_quant16.txt"])
def test_quant_goldens_on_gpu(name):
    from test_oracle_pins import golden_quant
    n, bits, alpha, ent, msg, _ = golden_quant(name)
    idx = np.array([e[0] for e in ent], np.uint32)
    val = np.array([e[1] for e in ent], np.uint32).view(np.float32)
    rc, got, v = encode_quant(idx, val, n, float(alpha), bits, np.full(n, 9.0, np.float32))
    assert rc == 0 and got == msg
    assert [int(bits_of) for bits_of in v[idx].view(np.uint32)] == [e[3] for e in ent]
    assert np.all(np.delete(v, idx) == 9.0)
    rc, dense = decode_quant([msg], n, bits, float(alpha))
    orc_rc, odense = oracle.decode_accumulate_quant([msg], n, bits, alpha)
    assert rc == 0 and orc_rc == 0 and same_bits(dense, odense)


@pytest.mark.parametrize("seed", range(8))
def test_quant_encode_random(seed):
    rng = np.random.default_rng(2100 + seed)
    n = int(rng.integers(1, 5_000_000))
    k = int(rng.integers(0, min(n, 300_000) + 1))
    bits = 8 if seed % 2 else 16
    alpha = float(np.float32(rng.choice([1.0, 3.0, 1000.0, 0.37, 2.0 ** 20])))
    idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
    val = (rng.standard_normal(k) * 10.0 ** rng.integers(-6, 3, k)).astype(np.float32)
    val[rng.random(k) < 0.02] = np.float32(-0.0)
    val[rng.random(k) < 0.01] = np.float32(np.inf)
    v0 = rng.standard_normal(n).astype(np.float32)
    rc, msg, v = encode_quant(idx, val, n, alpha, bits, v0)
    orc_rc, omsg, ov = oracle.encode_quant(idx, val, n, alpha, bits, v0)
    assert rc == 0 and orc_rc == 0
    assert msg == omsg
    assert same_bits(v, ov)


@pytest.mark.parametrize("seed", range(6))
def test_quant_decode_learners(seed):
    rng = np.random.default_rng(2200 + seed)
    n = int(rng.integers(1, 3_000_000))
    W = int(rng.integers(1, 300))
    bits = 16 if seed % 2 else 8
    alpha = float(np.float32(rng.choice([0.5, 3.0, 1000.0])))
    msgs = []
    for _ in range(W):
        k = int(rng.integers(0, min(n, 20_000) + 1))
        idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
        val = (rng.standard_normal(k) * 10.0 ** rng.integers(-3, 2, k)).astype(np.float32)
        rc, m, _ = oracle.encode_quant(idx, val, n, alpha, bits)
        assert rc == 0
        msgs.append(m)
    base = rng.standard_normal(n).astype(np.float32)
    base[::9] = np.float32(-0.0)
    for acc in (False, True):
        rc, dense = decode_quant(msgs, n, bits, alpha, dense=base, accumulate=acc)
        orc_rc, odense = oracle.decode_accumulate_quant(msgs, n, bits, alpha, dense=base,
                                                        accumulate=acc)
        assert rc == 0 and orc_rc == 0 and same_bits(dense, odense), acc
    rc, w = decode_apply_quant(msgs, n, bits, alpha, base, 0.37)
    orc_rc, ow = oracle.decode_apply_quant(msgs, n, bits, alpha, base, np.float32(0.37))
    assert rc == 0 and orc_rc == 0 and same_bits(w, ow)


@pytest.mark.parametrize("bits", [8, 16])
@pytest.mark.parametrize("case", ["sparse, escapes", "crowded tiles", "ragged, shifted view"])
def test_quant_decode_one_message(bits, case):
    # one message of integers: each value dequantized once where it lands and +0 elsewhere, or
    # added onto dense when accumulating; gaps past 65535 entries (escape tokens), tiles holding
    # more tokens than one round stages, and a dense view 1-3 floats off a 16-byte boundary
    rng = np.random.default_rng(bits + len(case))
    if case.startswith("sparse"):
        n = 5_000_003
        idx = np.sort(rng.choice(n, 60, replace=False)).astype(np.uint32)
    elif case.startswith("crowded"):
        n = 70_001
        idx = np.sort(rng.choice(n, n // 2, replace=False)).astype(np.uint32)
    else:
        n = 3 * 16384 + 4101
        idx = np.sort(rng.choice(n, n // 40, replace=False)).astype(np.uint32)
    alpha = float(np.float32(rng.choice([0.5, 3.0, 1000.0])))
    val = (rng.standard_normal(idx.size) * 10.0 ** rng.integers(-3, 2, idx.size)).astype(np.float32)
    orc_rc, msg, _ = oracle.encode_quant(idx, val, n, alpha, bits)
    assert orc_rc == 0
    base = rng.standard_normal(n).astype(np.float32)
    base[::7] = np.float32(-0.0)
    shift = int(rng.integers(1, 4)) if case.startswith("ragged") else 0
    for acc in (False, True):
        buf = torch.full((n + 8,), float("nan"), dtype=torch.float32, device="cuda")
        buf[shift:shift + n] = torch.from_numpy(base).cuda()
        bufs, sizes = gpu_helpers._device_messages([msg])
        ws_bytes = dgc.dgc_decode_workspace_quant(sizes, n, bits)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        dgc.dgc_decode_accumulate_quant(bufs, sizes, bits, alpha, buf[shift:shift + n], n, acc,
                                        status, ws, ws_bytes=ws_bytes)
        orc_rc, odense = oracle.decode_accumulate_quant([msg], n, bits, alpha, dense=base,
                                                        accumulate=acc)
        host = buf.cpu().numpy()
        assert dgc.dgc_read_status(status) == 0 and orc_rc == 0
        assert same_bits(host[shift:shift + n], odense), (case, acc)
        assert np.isnan(host[:shift]).all() and np.isnan(host[shift + n:]).all()


def test_quant_nan_and_infinities_on_gpu():
    n = 10
    idx = np.array([1, 2, 3], np.uint32)
    val = np.array([np.nan, np.inf, -np.inf], np.float32)
    rc, msg, v = encode_quant(idx, val, n, 2.0, 8, np.zeros(n, np.float32))
    orc_rc, omsg, ov = oracle.encode_quant(idx, val, n, 2.0, 8, np.zeros(n, np.float32))
    assert rc == 0 and orc_rc == 0 and msg == omsg  # NaN -> 0, +-inf -> +-127
    assert np.isnan(v[1]) and np.isnan(ov[1])       # NaN - 0 is a NaN (payloads may differ)
    assert same_bits(v[2:4], ov[2:4])


def test_quant_decode_rejects_and_leaves_dense():
    n = 1000
    idx, val = np.array([5, 999], np.uint32), np.array([1.0, -2.0], np.float32)
    _, m8, _ = oracle.encode_quant(idx, val, n, 2.0, 8)
    _, m8b, _ = oracle.encode_quant(idx, val, n, 4.0, 8)   # another alpha
    v1 = oracle.encode(idx, val, n)                          # a binary32 message, 6 B per token
    base = np.full(n, 7.0, np.float32)
    for msgs in ([m8b], [m8, m8b], [m8b, m8]):
        rc, d = decode_quant(msgs, n, 8, 2.0, dense=base, accumulate=True)
        assert rc == dgc.ECORRUPT and np.all(d == 7.0)
        rc, w = decode_apply_quant(msgs, n, 8, 2.0, base, 0.5)
        assert rc == dgc.ECORRUPT and np.all(w == 7.0)
    # its 44 bytes fit both widths (8 bits: T = 4, 16 bits: T = 3): the header tells it apart
    for bits in (8, 16):
        rc, d = decode_quant([v1], n, bits, 2.0, dense=base, accumulate=True)
        assert rc == dgc.ECORRUPT and np.all(d == 7.0)
    with pytest.raises(dgc.DGCError) as e:  # 45 bytes: no message of this library
        decode_quant([v1 + b"\0"], n, 16, 2.0, dense=base)
    assert e.value.code == dgc.ECORRUPT
    with pytest.raises(dgc.DGCError) as e:  # 38 bytes: an 8-bit message, no 16-bit size
        decode_quant([m8], n, 16, 2.0, dense=base)
    assert e.value.code == dgc.ECORRUPT
    _, m16, _ = oracle.encode_quant(np.array([5, 6, 999], np.uint32), np.ones(3, np.float32), n,
                                    2.0, 16)  # 44 bytes, also an 8-bit size: the width differs
    rc, d = decode_quant([m16], n, 8, 2.0, dense=base, accumulate=True)
    assert rc == dgc.ECORRUPT and np.all(d == 7.0)


def test_quant_after_compress_matches_oracle():
    # the path a learner runs: compress (sampled, 99.9%), then 8-bit integers with the
    # remainders put back into the residual
    n = 4_000_003
    off = np.array([0, 1_000_000, n])
    pd, po = params_pair(mode=dgc.SELECT_SAMPLED, sparsity=0.999, momentum=0.9, seed=5)
    comp = Compressor(n, off, pd)
    u_h, v_h = np.zeros(n, np.float32), np.zeros(n, np.float32)
    u_d, v_d = dev_f32(u_h), dev_f32(v_h)
    for t in range(3):
        g = (np.random.default_rng([7, t]).standard_normal(n) * 0.01).astype(np.float32)
        comp(dev_f32(g), u_d, v_d)
        assert comp.status_code() == 0
        idx, val, _ = comp.results()
        oidx, oval, _ = oracle.compress(g, u_h, v_h, off, po)
        assert np.array_equal(idx, oidx) and same_bits(val, oval)
        alpha = 1000.0
        enc = Encoder(comp.cap, n)
        dgc.dgc_encode_quant(comp.out_idx, comp.out_val, comp.out_count, n, alpha, 8, v_d,
                             enc.out, enc.out_bytes, enc.status, enc.ws, max_count=comp.cap,
                             out_cap=enc.cap, ws_bytes=enc.ws_bytes)
        assert dgc.dgc_read_status(enc.status) == 0
        rc, omsg, v_h = oracle.encode_quant(oidx, oval, n, alpha, 8, v_h)
        assert rc == 0 and enc.message() == omsg
        assert same_bits(host_f32(v_d), v_h), f"step {t}"
        assert same_bits(host_f32(u_d), u_h)


# ---------------------------------------------------- ScaleComp: leak and one shared index set
@pytest.mark.parametrize("case", range(9))
def test_leak_all_modes(case):
    rng = np.random.default_rng(4000 + case)
    n = EDGE_N[case % len(EDGE_N)] * 3
    off = _segments(rng, n)
    mode = [dgc.SELECT_EXACT, dgc.SELECT_SAMPLED, dgc.SELECT_ADACOMP][case % 3]
    leak = float(np.float32(rng.choice([0.5, 0.9, 0.999])))
    run_steps(lambda t: (np.random.default_rng([case, t]).standard_normal(n) * 0.01)
              .astype(np.float32), off, 3, mode=mode, sparsity=0.99, momentum=0.9, bin_size=64,
              clip_norm=float(rng.choice([0.0, 1.0])), leak=leak)


class Shared:
    """dgc_compress_shared for one (n, segments, params) shape."""

    def __init__(self, n, seg_off, params, max_count):
        self.n, self.params, self.max_count = n, params, max(int(max_count), 1)
        self.seg = torch.from_numpy(np.asarray(seg_off, np.int64)).cuda()
        self.ws = torch.empty(max(dgc.dgc_compress_workspace(n, self.seg.numel() - 1, params), 256),
                              dtype=torch.uint8, device="cuda")
        self.out = torch.zeros(self.max_count, dtype=torch.float32, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def __call__(self, g, u, v, idx, count):
        dgc.dgc_compress_shared(g, u, v, self.seg, self.params, idx, count, self.out,
                                self.status, self.ws, n=self.n, max_count=self.max_count)
        return dgc.dgc_read_status(self.status)


@pytest.mark.parametrize("case", range(12))
def test_compress_shared_random_sets(case):
    rng = np.random.default_rng(4100 + case)
    n = EDGE_N[case % len(EDGE_N)] * (1 + case % 3)
    off = _segments(rng, n)
    kw = dict(mode=dgc.SELECT_SAMPLED, momentum=0.9, mask_momentum=bool(case % 2),
              clip_norm=float(rng.choice([0.0, 1.0])), leak=float(np.float32(rng.choice([0, 0.9]))))
    pd, po = params_pair(**kw)
    u_h, v_h = (rng.standard_normal(n).astype(np.float32) for _ in range(2))
    u_d, v_d = dev_f32(u_h), dev_f32(v_h)
    sh = Shared(n, off, pd, n)
    for t in range(3):
        g = (rng.standard_normal(n) * 0.01).astype(np.float32)
        k = int(rng.integers(0, n + 1))
        idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
        rc = sh(dev_f32(g), u_d, v_d, dev_idx(idx), torch.tensor([k], dtype=torch.int64,
                                                                device="cuda"))
        assert rc == 0
        orc_rc, oval = oracle.compress_shared(g, u_h, v_h, off, po, idx)
        assert orc_rc == 0
        assert same_bits(host_f32(sh.out)[:k], oval)
        assert same_bits(host_f32(v_d), v_h) and same_bits(host_f32(u_d), u_h), t


def test_compress_shared_rejects_bad_sets():
    n = 5000
    off = np.array([0, n])
    pd = dgc.make_params(mode=dgc.SELECT_EXACT)
    sh = Shared(n, off, pd, 8)
    for idx, count in (([3, 3, 9], 3), ([9, 3], 2), ([1, n], 2), ([1, 2], 9), ([1, 2], -1)):
        u = dev_f32(np.ones(n, np.float32))
        v = dev_f32(np.ones(n, np.float32))
        sh.out.fill_(7.0)
        rc = sh(dev_f32(np.ones(n, np.float32)), u, v, dev_idx(np.array(idx + [0] * 8, np.uint32)),
                torch.tensor([count], dtype=torch.int64, device="cuda"))
        assert rc == dgc.EINVAL
        assert torch.all(u == 1.0) and torch.all(v == 1.0) and torch.all(sh.out == 7.0)


def _sum_shared(vals, count=None, max_count=None):
    k = vals[0].size if vals else 0
    d = [dev_f32(np.append(x, np.float32(0))) for x in vals]
    out = torch.full((max(k, 1),), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(dgc.dgc_sum_shared_workspace(len(vals)), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = torch.tensor([k if count is None else count], dtype=torch.int64, device="cuda")
    dgc.dgc_sum_shared(d, c, k if max_count is None else max_count, out, status, ws)
    return dgc.dgc_read_status(status), host_f32(out)[:k]


def test_sum_shared_matches_oracle():
    rows = read_golden("decode_order.txt")  # 1e8 + 1 - 1e8 in learner order is exactly 0
    vals = [np.array([v[1]], np.uint32).view(np.float32) for t, v in rows if t == "learner"]
    rc, out = _sum_shared(vals)
    assert rc == 0 and int(out.view(np.uint32)[0]) == 0
    rng = np.random.default_rng(8)
    for W, k in ((1, 1000), (7, 123_457), (64, 25_558)):
        vals = [(rng.standard_normal(k) * 10.0 ** rng.integers(-3, 3, k)).astype(np.float32)
                for _ in range(W)]
        rc, out = _sum_shared(vals)
        orc_rc, oout = oracle.sum_shared(vals)
        assert rc == 0 and orc_rc == 0 and same_bits(out, oout)
    rc, out = _sum_shared([np.ones(10, np.float32)], count=11, max_count=10)
    assert rc == dgc.EINVAL and np.all(np.isnan(out))


def test_scalecomp_learners_rotating_chooser():
    _scalecomp_learners(4, 1_000_003, np.array([0, 300_000, 1_000_003]), 4)


@pytest.mark.slow
def test_scalecomp_learners_full_size():
    # eight learners of the aggregation workload's size (25,557,032 entries), two steps
    _scalecomp_learners(8, 25_557_032, np.array([0, 25_557_032]), 2)


def _scalecomp_learners(W, n, off, steps):
    # W learners, one shared set per step chosen by learner t mod W with the sampled compressor,
    # the others sending at that set, the value vectors summed: against the oracle run alike
    kw = dict(mode=dgc.SELECT_SAMPLED, sparsity=0.999, momentum=0.9, seed=11, leak=0.9)
    pd, po = params_pair(**kw)
    comp = Compressor(n, off, pd)
    sh = Shared(n, off, pd, comp.cap)
    state_h = [[np.zeros(n, np.float32), np.zeros(n, np.float32)] for _ in range(W)]
    state_d = [[dev_f32(a), dev_f32(b)] for a, b in state_h]
    for t in range(steps):
        grads = [(np.random.default_rng([9, t, w]).standard_normal(n) * 0.01).astype(np.float32)
                 for w in range(W)]
        lead = t % W
        comp(dev_f32(grads[lead]), *state_d[lead])
        assert comp.status_code() == 0
        idx, val, _ = comp.results()
        oidx, oval, _ = oracle.compress(grads[lead], *state_h[lead], off, po)
        assert np.array_equal(idx, oidx) and same_bits(val, oval)
        vals_d, vals_o = [None] * W, [None] * W
        vals_d[lead], vals_o[lead] = val, oval
        for w in range(W):
            if w == lead:
                continue
            assert sh(dev_f32(grads[w]), *state_d[w], comp.out_idx, comp.out_count) == 0
            vals_d[w] = host_f32(sh.out)[: idx.size].copy()
            rc, vals_o[w] = oracle.compress_shared(grads[w], *state_h[w], off, po, oidx)
            assert rc == 0 and same_bits(vals_d[w], vals_o[w])
        rc, total = _sum_shared(vals_d)
        orc_rc, ototal = oracle.sum_shared(vals_o)
        assert rc == 0 and orc_rc == 0 and same_bits(total, ototal)
        for w in range(W):
            assert same_bits(host_f32(state_d[w][1]), state_h[w][1]), (t, w)
            assert same_bits(host_f32(state_d[w][0]), state_h[w][0]), (t, w)


@pytest.mark.parametrize("seed", range(3))
def test_sampled_calls_with_changing_sparsity(seed):
    # one workspace across calls whose sparsity jumps both ways (the cached sample positions
    # stay valid, the threshold moves a long way), a zero-length segment, and one call with a
    # gradient ten times larger: every call bitwise equal to the oracle
    rng = np.random.default_rng(4700 + seed)
    n = 2_000_003
    off = np.array([0, 700_000, 700_000, 1_500_000, n])
    schedule = [0.999, 0.9, 0.999, 0.99, 0.5, 0.999, 0.999]
    u_h, v_h = np.zeros(n, np.float32), np.zeros(n, np.float32)
    u_d, v_d = dev_f32(u_h), dev_f32(v_h)
    comp = None
    for t, sp in enumerate(schedule):
        kw = dict(mode=dgc.SELECT_SAMPLED, sparsity=sp, momentum=0.9, seed=seed,
                  clip_norm=float(rng.choice([0.0, 1.0])))
        pd, po = params_pair(**kw)
        if comp is None:  # outputs sized for the densest call
            comp = Compressor(n, off, dgc.make_params(**dict(kw, sparsity=min(schedule))))
        comp.params = pd  # the same workspace across calls, as a training loop keeps it
        g = (rng.standard_normal(n) * 0.01 * (10.0 if t == 4 else 1.0)).astype(np.float32)
        comp(dev_f32(g), u_d, v_d)
        assert comp.status_code() == 0
        idx, val, st = comp.results()
        oidx, oval, ost = oracle.compress(g, u_h, v_h, off, po)
        assert np.array_equal(idx, oidx), f"call {t}"
        assert same_bits(val, oval)
        assert same_bits(host_f32(v_d), v_h) and same_bits(host_f32(u_d), u_h)
        for s, o in enumerate(ost):
            assert st[s]["candidates"] == o["candidates"] and st[s]["reselected"] == o["reselected"]
            assert st[s]["sample_key"] == o["sample_key"], (t, s)


def test_l2_fetch_granularity_hint_keeps_results():
    # the context limit is a fetch-size hint: the sampled step stays bitwise equal to the oracle
    assert dgc.dgc_set_l2_fetch_granularity(64) == 0
    n = 1_000_003
    off = np.array([0, 400_000, n])
    run_steps(lambda t: (np.random.default_rng([31, t]).standard_normal(n) * 0.01)
              .astype(np.float32), off, 3, mode=dgc.SELECT_SAMPLED, sparsity=0.999, momentum=0.9)


def test_compress_encode_in_cuda_graph():
    # dgc_compress and dgc_encode enqueue kernels only, so a training loop can
    # capture them once (after one ordinary call on the device) and replay the graph every step;
    # the replays must give the oracle's results step after step
    n = 3_000_017
    off = np.array([0, 1_000_000, n])
    kw = dict(mode=dgc.SELECT_SAMPLED, sparsity=0.999, momentum=0.9, seed=4, clip_norm=1.0)
    pd, po = params_pair(**kw)
    comp = Compressor(n, off, pd)
    enc = Encoder(comp.cap, n)
    g_static = torch.zeros(n, dtype=torch.float32, device="cuda")
    u_d, v_d = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    u_h, v_h = np.zeros(n, np.float32), np.zeros(n, np.float32)

    def step():
        comp(g_static, u_d, v_d)
        dgc.dgc_encode(comp.out_idx, comp.out_val, comp.out_count, n, enc.out, enc.out_bytes,
                       enc.status, enc.ws, max_count=comp.cap, out_cap=enc.cap,
                       ws_bytes=enc.ws_bytes)

    grads = [(np.random.default_rng([61, t]).standard_normal(n) * 0.01).astype(np.float32)
             for t in range(4)]
    g_static.copy_(torch.from_numpy(grads[0]))
    step()  # the ordinary first call (sets the streaming kernels' attributes on this device)
    torch.cuda.synchronize()
    oracle.compress(grads[0], u_h, v_h, off, po)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step()
    torch.cuda.synchronize()
    # capture enqueues nothing: the state is still after step 0
    assert same_bits(host_f32(v_d), v_h)
    for t in range(1, 4):
        g_static.copy_(torch.from_numpy(grads[t]))
        graph.replay()
        torch.cuda.synchronize()
        assert comp.status_code() == 0 and dgc.dgc_read_status(enc.status) == 0
        idx, val, _ = comp.results()
        oidx, oval, _ = oracle.compress(grads[t], u_h, v_h, off, po)
        assert np.array_equal(idx, oidx) and same_bits(val, oval), t
        assert same_bits(host_f32(v_d), v_h) and same_bits(host_f32(u_d), u_h), t
        assert enc.message() == oracle.encode(oidx, oval, n)
