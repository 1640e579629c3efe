#!/usr/bin/env python3
"""Throughput of the DGC per-worker compressor on GB300: GB/s of fp32 gradient per step.

A step is one pass of the whole hot path over a fresh synthetic gradient: dgc_compress
(momentum-corrected accumulation, sampled 1% threshold with hierarchical re-selection, index-
ordered compaction, masking) -> dgc_encode (32-bit values + 16-bit zero runs) ->
dgc_decode_accumulate_dev of the message into a dense gradient (the decoder reads the message
size from device memory, so a step needs no host round trip and each of its three calls replays
from a CUDA graph). The workload is the 2^30-entry
(4 GiB) flat bucket: g ~ N(0, 1e-4) with 0.01% fixed outliers x100, momentum 0.9, 99.9%
sparsity; the warm-up steps follow the warm-up schedule 75% -> 93.75% -> 98.4375% -> 99.6%.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank compresses its own bucket on its own GPU (independent replicas,
no collective on the data path); rank 0 prints one JSON line with the max time over ranks.
`--impl reference` times the oracle (the plain CPU restatement used by the tests) on the host on
a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GB/s of fp32 gradient compressed (+% of HBM roofline), 1×GB300, 99.9% sparsity"
UNIT = "GB/s"
WORKLOAD = ("flat bucket of 2^30 fp32 entries (4 GiB), g ~ N(0, 1e-4) with 0.01% fixed "
            "outliers x100; sampled 1% threshold, re-select if |C| > 1.3k; 99.9% sparsity; "
            "compress + encode + decode per step")
WORKLOAD_ADACOMP = ("flat bucket of 2^30 fp32 entries (4 GiB), g ~ N(0, 1e-4) with 0.01% fixed "
                    "outliers x100; AdaComp bins of {} entries; compress + encode + decode per "
                    "step")
SEED = 20240


def _one_segment(n):
    import numpy as np

    return lambda: np.array([0, n], np.int64)


def _workload_segments(name):
    def f():
        import workloads

        return getattr(workloads, name)()
    return f


# the other workloads: segment table, settings beyond sparsity 0.999 and momentum 0.9, name
OTHER_WORKLOADS = {
    "single": (_one_segment(1_048_576), dict(mode=0),
               "single tensor of 1,048,576 fp32 entries ~ N(0, 0.01^2); exact top-k (k = 1049)"),
    "resnet50": (_workload_segments("resnet50_segments"), dict(mode=0, clip_norm=1.0),
                 "ResNet-50-shaped set: 161 tensors, 25,557,032 fp32 entries, per-tensor "
                 "sigma log-uniform in [1e-4, 1e-1]; exact top-k per tensor, clip 1.0 per tensor"),
    "deepspeech": (_workload_segments("deepspeech_segments"),
                   dict(mode=1, sample_ratio=0.01, reselect_factor=1.3),
                   "DeepSpeech-scale bucket: 122,000,000 fp32 entries, Student-t(3) x 1e-3, "
                   "5 x 24M + 2M segments; sampled 1% threshold, re-select if |C| > 1.3k"),
    "learners": (_one_segment(25_557_032), dict(mode=0),
                 "one learner of the aggregation workload: 25,557,032 fp32 entries ~ "
                 "N(0, 0.01^2); exact top-k (k = 25,558)"),
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--n", type=int, default=1 << 30)
    ap.add_argument("--pool", type=int, default=3, help="distinct gradients cycled on device")
    ap.add_argument("--e2e-steps", type=int, default=24)
    ap.add_argument("--cpu-n", type=int, default=1 << 26)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--workload", choices=["bucket1g", "single", "resnet50", "deepspeech",
                                           "learners", "aggregation"], default="bucket1g",
                    help="bucket1g is the headline; the others time the other workloads' steps "
                         "(aggregation: only the 64-learner decode and SGD step)")
    ap.add_argument("--select", choices=["sampled", "adacomp"], default="sampled",
                    help="DGC sampled threshold (the headline) or AdaComp bins of --bin-size")
    ap.add_argument("--bin-size", type=int, default=1000)
    ap.add_argument("--no-graph", action="store_true",
                    help="launch compress and encode call by call instead of replaying graphs")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the single-tensor, ResNet-50, DeepSpeech and aggregation timings "
                         "that follow the headline bucket")
    ap.add_argument("--workload-steps", type=int, default=30)
    ap.add_argument("--l2-fetch", type=int, default=64,
                    help="this process's L2 fetch granularity limit in bytes (0: leave it)")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ ranks and aggregation
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / seconds_max


# ------------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ---------------------------------------------------------------------- roofline inputs
def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def stream_pass_source_hash() -> str:
    """Hash of the streaming kernel's code (compress.cu and dgc_device.cuh without // comments and
    blank lines, so that a comment edit does not orphan the recorded counters)."""
    h = hashlib.sha256()
    for f in ("compress.cu", "dgc_device.cuh"):
        with open(os.path.join(ROOT, "sparsified_gradient_compression_gb300", "csrc", f)) as fh:
            for line in fh:
                code = line.split("//")[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(n: int):
    """DRAM bytes per launch of the streaming pass from the committed ncu summary, scaled to n
    entries; None when the summary is missing or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "stream_pass_sampled_traffic.txt")
    try:
        kv = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("source_sha256_16") != stream_pass_source_hash():
            return None
        per_entry = float(kv["dram_bytes_per_launch"]) / float(kv["entries_per_launch"])
        return per_entry * n
    except Exception:
        return None


# ----------------------------------------------------------------------------- our arm
class Pipeline:
    """Buffers for one worker's step on one GPU, and the step itself (public API calls only)."""

    def __init__(self, n, params, dev, seg_off=None):
        import numpy as np
        import torch

        import sparsified_gradient_compression_gb300 as dgc

        self.dgc, self.n, self.dev = dgc, n, dev
        off = np.array([0, n], np.int64) if seg_off is None else np.asarray(seg_off, np.int64)
        self.nseg = off.size - 1
        self.seg = torch.from_numpy(off).to(dev)
        self.cap = max(dgc.dgc_compress_max_out(n, self.nseg, p) for p in params)
        self.ws_bytes = max(dgc.dgc_compress_workspace(n, self.nseg, p) for p in params)
        self.u = torch.zeros(n, dtype=torch.float32, device=dev)
        self.v = torch.zeros(n, dtype=torch.float32, device=dev)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.out_idx = torch.empty(self.cap, dtype=torch.int32, device=dev)
        self.out_val = torch.empty(self.cap, dtype=torch.float32, device=dev)
        self.out_count = torch.zeros(1, dtype=torch.int64, device=dev)
        self.stats = torch.zeros(self.nseg * dgc.STATS_BYTES, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.msg_cap = dgc.dgc_encode_max_bytes(self.cap, n)
        self.msg = torch.empty(self.msg_cap, dtype=torch.uint8, device=dev)
        self.msg_bytes = torch.zeros(1, dtype=torch.int64, device=dev)
        self.ews_bytes = dgc.dgc_encode_workspace(self.cap)
        self.ews = torch.empty(self.ews_bytes, dtype=torch.uint8, device=dev)
        # the decoder reads the message size from device memory (msg_bytes), its workspace laid
        # out for the largest message the encoder may write
        self.dws_bytes = dgc.dgc_decode_workspace_bound([self.msg_cap], n)
        self.dws = torch.empty(self.dws_bytes, dtype=torch.uint8, device=dev)
        self.dense = torch.empty(n, dtype=torch.float32, device=dev)
        self.nb_host = torch.zeros(1, dtype=torch.int64, pin_memory=True)

    def compress(self, g, p):
        self.dgc.dgc_compress(g, self.u, self.v, self.seg, p, self.out_idx, self.out_val,
                              self.out_count, self.stats, self.status, self.ws, n=self.n,
                              out_cap=self.cap, ws_bytes=self.ws_bytes)

    def encode(self):
        self.dgc.dgc_encode(self.out_idx, self.out_val, self.out_count, self.n, self.msg,
                            self.msg_bytes, self.status, self.ews, max_count=self.cap,
                            out_cap=self.msg_cap, ws_bytes=self.ews_bytes)

    def bound(self, p) -> int:
        """The largest message a compress call with params p can lead to: the decoder's bound."""
        return self.dgc.dgc_encode_max_bytes(
            self.dgc.dgc_compress_max_out(self.n, self.nseg, p), self.n)

    def decode(self, p):
        # the decoder's grids follow the bound on the message, so it is the bound of this
        # step's sparsity (the warm-up schedule's lower sparsities have far larger ones)
        self.dgc.dgc_decode_accumulate_dev([self.msg], self.msg_bytes, [self.bound(p)],
                                           self.dense, self.n, False, self.status, self.dws,
                                           ws_bytes=self.dws_bytes)

    def message_size(self) -> int:
        """The last step's message size, read back to the host (waits for the step)."""
        self.nb_host.copy_(self.msg_bytes)
        return int(self.nb_host.item())

    def capture(self, g, p):
        """CUDA graphs of this pipeline's compress call on g, its encode call and its decode
        call: each enqueues kernels only, the decode taking the message size from
        device memory, so they replay as they were captured, with no host round trip."""
        import torch

        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        graphs = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graphs[0], stream=side):
                self.compress(g, p)
            with torch.cuda.graph(graphs[1], stream=side):
                self.encode()
            with torch.cuda.graph(graphs[2], stream=side):
                self.decode(p)
        torch.cuda.current_stream(self.dev).wait_stream(side)
        return graphs

    def step(self, g, p, ev=None, graphs=None):
        """One step, compress -> encode -> decode, enqueued without waiting on the host; with
        `graphs` (from capture() on the same g and p) the three are graph replays."""
        if ev:
            ev[0].record()
        if graphs:
            graphs[0].replay()
        else:
            self.compress(g, p)
        if ev:
            ev[1].record()
        if graphs:
            graphs[1].replay()
        else:
            self.encode()
        if ev:
            ev[2].record()
        if graphs:
            graphs[2].replay()
        else:
            self.decode(p)
        if ev:
            ev[3].record()

    def time_decode_apply(self, nb, reps=20):
        """The receiving side's alternative to the dense decode: the last message applied as one
        SGD step to a weight vector (dgc_decode_apply), timed alone with CUDA events."""
        import torch

        w = torch.zeros(self.n, dtype=torch.float32, device=self.dev)
        E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        ms = []
        for _ in range(reps + 3):
            a, b = E(), E()
            a.record()
            self.dgc.dgc_decode_apply([self.msg], [nb], w, self.n, 0.01, self.status, self.dws,
                                      ws_bytes=self.dws_bytes)
            b.record()
            b.synchronize()
            ms.append(a.elapsed_time(b))
        del w
        return sorted(ms[3:])[reps // 2]

    def time_quant(self, bits=8, alpha=1000.0, reps=20):
        """The integer-valued variant of the last step's message, outside the step: encode with
        the remainders put back into v (idempotent: the same values again), then decode it to a
        dense array and apply it to a weight vector. Median CUDA-event times of each call."""
        import torch

        dgc = self.dgc
        qmsg = torch.empty(self.msg_cap, dtype=torch.uint8, device=self.dev)
        E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

        def timed(fn):
            ms = []
            for _ in range(reps + 3):
                a, b = E(), E()
                a.record()
                fn()
                b.record()
                b.synchronize()
                ms.append(a.elapsed_time(b))
            return sorted(ms[3:])[reps // 2]

        t_enc = timed(lambda: dgc.dgc_encode_quant(
            self.out_idx, self.out_val, self.out_count, self.n, alpha, bits, self.v, qmsg,
            self.msg_bytes, self.status, self.ews, max_count=self.cap, out_cap=self.msg_cap,
            ws_bytes=self.ews_bytes))
        self.nb_host.copy_(self.msg_bytes)
        nb = int(self.nb_host.item())
        ws_bytes = dgc.dgc_decode_workspace_quant([nb], self.n, bits)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.dev)
        t_dec = timed(lambda: dgc.dgc_decode_accumulate_quant(
            [qmsg], [nb], bits, alpha, self.dense, self.n, False, self.status, ws,
            ws_bytes=ws_bytes))
        w = torch.zeros(self.n, dtype=torch.float32, device=self.dev)
        t_app = timed(lambda: dgc.dgc_decode_apply_quant(
            [qmsg], [nb], bits, alpha, w, self.n, 0.01, self.status, ws, ws_bytes=ws_bytes))
        del w, ws, qmsg
        return {"bits": bits, "alpha": alpha, "message_bytes": nb, "encode_ms": round(t_enc, 4),
                "decode_ms": round(t_dec, 4), "decode_apply_ms": round(t_app, 4)}


    def time_shared(self, p, g, learners=8, reps=20):
        """One index set for all learners, outside the step: a learner's step at the last
        step's set (dgc_compress_shared: the accumulate-only streaming pass, then the gather),
        and the learner-ordered sum of `learners` value vectors (dgc_sum_shared)."""
        import torch

        dgc = self.dgc
        E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        vals = [torch.empty(self.cap, dtype=torch.float32, device=self.dev)
                for _ in range(learners)]

        def timed(fn):
            ms = []
            for _ in range(reps + 3):
                a, b = E(), E()
                a.record()
                fn()
                b.record()
                b.synchronize()
                ms.append(a.elapsed_time(b))
            return sorted(ms[3:])[reps // 2]

        kev = (E(), E())
        dgc.dgc_profile_stream_pass(*kev)  # the shared call marks its streaming pass too
        t_step = timed(lambda: dgc.dgc_compress_shared(
            g, self.u, self.v, self.seg, p, self.out_idx, self.out_count, vals[0], self.status,
            self.ws, n=self.n, max_count=self.cap, ws_bytes=self.ws_bytes))
        dgc.dgc_profile_stream_pass(None, None)
        t_pass = kev[0].elapsed_time(kev[1])
        ws = torch.empty(dgc.dgc_sum_shared_workspace(learners), dtype=torch.uint8,
                         device=self.dev)
        out = torch.empty(self.cap, dtype=torch.float32, device=self.dev)
        t_sum = timed(lambda: dgc.dgc_sum_shared(vals, self.out_count, self.cap, out,
                                                 self.status, ws))
        del vals, out, ws
        return {"compress_shared_ms": round(t_step, 4), "stream_pass_ms": round(t_pass, 4),
                "sum_shared_ms": round(t_sum, 4), "learners": learners}


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import sparsified_gradient_compression_gb300 as dgc
    import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    dgc.build()
    torch.zeros(1, device=dev)  # the context exists before its limit is set
    if args.l2_fetch > 0:  # a context limit of this process (see dgc_set_l2_fetch_granularity)
        dgc.dgc_set_l2_fetch_granularity(args.l2_fetch)
    wl = args.workload
    if wl == "aggregation":  # the 64-learner decode and SGD step alone
        agg = run_aggregation(dev, measured_peak_hbm()[0], reps=args.steps, flush=L2Flush(dev))
        if rank == 0:
            print(json.dumps({"metric": "ms per 64-message decode", "aggregation": agg}),
                  flush=True)
        return
    mode = dgc.SELECT_ADACOMP if args.select == "adacomp" else dgc.SELECT_SAMPLED
    if wl == "bucket1g":  # the headline: one segment, the warm-up schedule, then 99.9%
        n, off = args.n, None
        params = [dgc.make_params(mode=mode, sparsity=s, momentum=0.9, sample_ratio=0.01,
                                  reselect_factor=1.3, seed=SEED + rank, bin_size=args.bin_size)
                  for s in list(workloads.WARMUP_SPARSITY[:4]) + [0.999]]
    else:  # the other workloads at their own settings, 99.9% from the first step
        off = OTHER_WORKLOADS[wl][0]()
        n = int(off[-1])
        kw = OTHER_WORKLOADS[wl][1]
        if args.select == "adacomp":
            kw = dict(kw, mode=dgc.SELECT_ADACOMP)
        params = [dgc.make_params(sparsity=0.999, momentum=0.9, seed=SEED + rank,
                                  bin_size=args.bin_size, **kw)]
    p_main = params[-1]
    pipe = Pipeline(n, params, dev, off)
    # inputs resident in HBM: a pool of distinct gradients, one per step in turn
    pool = []
    for i in range(args.pool):
        pool.append(torch.from_numpy(workloads.gradient(wl, step=i, seed=rank, n=n)).to(dev))

    for i in range(args.warmup):  # the warm-up schedule, then 99.9%
        pipe.step(pool[i % len(pool)], params[min(i, len(params) - 1)])
    torch.cuda.synchronize()
    if dgc.dgc_read_status(pipe.status) != 0:
        raise RuntimeError("warm-up steps reported an error")

    K = args.steps
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    evs = [(E(), E(), E(), E()) for _ in range(K)]
    kev = [(E(), E()) for _ in range(K)]
    graphs, graph_kernels = None, 0
    gkevs = [(E(), E()) for _ in pool]  # the streaming pass's events inside each pool graph
    if not args.no_graph:  # per pool buffer (p_main): one compress, one encode, one decode graph
        torch.cuda.synchronize()
        l0 = dgc.dgc_launch_count()
        graphs = []
        for g, kev_g in zip(pool, gkevs):
            dgc.dgc_profile_stream_pass(*kev_g)  # an event-record node pair in this graph
            graphs.append(pipe.capture(g, p_main))
        dgc.dgc_profile_stream_pass(None, None)
        graph_kernels = (dgc.dgc_launch_count() - l0) // len(pool)  # kernels per step's graphs
        torch.cuda.synchronize()
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(gpu_id)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0 = dgc.dgc_launch_count()
    t_begin, t_end = E(), E()
    t_begin.record()
    t_graph_kernel = []
    # The steps are enqueued back to back. A pool graph's streaming-pass events hold the time of
    # the last step that replayed it: with 3 or more pool buffers the host reads step i - 2's
    # after enqueuing step i (waiting on that step's last event; the graph is not replayed again
    # before step i + 1), so the GPU always has the next step queued.
    lag = 2 if len(pool) >= 3 else 0
    for i in range(K):
        j = (args.warmup + i) % len(pool)
        if graphs:
            pipe.step(pool[j], p_main, evs[i], graphs[j])
            if i >= lag:
                evs[i - lag][3].synchronize()
                kv = gkevs[(args.warmup + i - lag) % len(pool)]
                t_graph_kernel.append(kv[0].elapsed_time(kv[1]))
        else:
            dgc.dgc_profile_stream_pass(kev[i][0], kev[i][1])
            pipe.step(pool[j], p_main, evs[i])
    t_end.record()
    torch.cuda.synchronize()
    if graphs:
        for i in range(max(K - lag, 0), K):
            kv = gkevs[(args.warmup + i) % len(pool)]
            t_graph_kernel.append(kv[0].elapsed_time(kv[1]))
    nb_last = pipe.message_size()
    dgc.dgc_profile_stream_pass(None, None)
    launches = dgc.dgc_launch_count() - launches0 + (K * graph_kernels if graphs else 0)
    clk = clocks.stop()
    barrier()
    if dgc.dgc_read_status(pipe.status) != 0:
        raise RuntimeError("timed steps reported an error")
    sec = t_begin.elapsed_time(t_end) / 1e3
    sec_max = max_over_ranks(sec, dev)
    value = whole_job_value(4.0 * n * K, world, sec_max) / 1e9
    t_compress = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    t_encode = sum(e[1].elapsed_time(e[2]) for e in evs) / K
    t_decode = sum(e[2].elapsed_time(e[3]) for e in evs) / K
    t_kernel = (sum(t_graph_kernel) / K if graphs else
                sum(a.elapsed_time(b) for a, b in kev) / K)
    segst = np.frombuffer(pipe.stats.cpu().numpy().tobytes(), dtype=[
        ("k", "<u8"), ("candidates", "<u8"), ("sent", "<u8"), ("thresh_key", "<u4"),
        ("sample_key", "<u4"), ("reselected", "<u4"), ("clip_scale", "<f4"),
        ("clip_sumsq", "<f8")])
    st = {f: int(segst[f].sum()) for f in ("k", "candidates", "sent")}  # over the segments
    cand = int(st["candidates"])
    # read g, u, v and write u, v; one 4-byte slot per candidate and one count per 2048-entry tile
    alg_bytes = 20.0 * n + 4.0 * cand + 4.0 * ((n + 2047) // 2048)
    peak, peak_kind = measured_peak_hbm()
    achieved = alg_bytes / (t_kernel / 1e3) / 1e9
    traffic = recorded_traffic(n)
    t_apply = pipe.time_decode_apply(nb_last)
    quant = pipe.time_quant()
    if dgc.dgc_read_status(pipe.status) != 0:
        raise RuntimeError("integer-message calls reported an error")
    shared = pipe.time_shared(p_main, pool[0])
    if dgc.dgc_read_status(pipe.status) != 0:
        raise RuntimeError("shared-set calls reported an error")
    shared["stream_pass_frac"] = round(20.0 * n / (shared["stream_pass_ms"] / 1e3) / 1e9 / peak, 4)
    if dgc.dgc_read_status(pipe.status) != 0:
        raise RuntimeError("decode-apply reported an error")

    e2e = None if args.no_e2e else run_e2e(args, pipe, pool, p_main, K)
    cpu = None
    if not args.no_cpu and rank == 0 and world == 1 and wl == "bucket1g":
        cpu = run_cpu_baseline(args.cpu_n, steps=3, select=args.select, bin_size=args.bin_size)
    if wl != "bucket1g":
        workload = OTHER_WORKLOADS[wl][2] + ("" if args.select == "sampled" else
                                             f"; AdaComp bins of {args.bin_size} entries")
    else:
        workload = WORKLOAD if args.select == "sampled" else WORKLOAD_ADACOMP.format(args.bin_size)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(sec_max * 1e3 / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; see workloads/)",
        "config": {"workload": workload, "n": n, "sparsity": 0.999, "k": int(st["k"]),
                   "selection": ("exact", "sampled", "adacomp")[int(p_main.mode)],
                   "momentum": 0.9, "sample_ratio": 0.01, "reselect_factor": 1.3,
                   "segments": pipe.nseg, "l2": f"{4 * n >> 20} MiB per array "
                   f"({'larger' if 4 * n > 129 * 2**20 else 'smaller'} than L2); "
                   f"{len(pool)} distinct gradients cycled",
                   "parallelism": f"{world} independent replicas" if world > 1 else "single GPU",
                   "l2_fetch_granularity_bytes": args.l2_fetch or "driver default",
                   "launch": "compress, encode and decode as CUDA graph replays (captured once "
                             "per gradient buffer; the decoder reads the message size from "
                             "device memory), no host round trip within a step" if graphs else
                             "call by call"},
        "roofline": {"bound": "hbm", "kernel": "k_stream_tma<%d> (accumulate + per-tile compaction)" % (args.select == "adacomp"),
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None if traffic is None else round(traffic),
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one "
                                       "67,108,864-entry launch, scaled to n (an extrapolation "
                                       "from that capture, not a measurement at n)",
                     "alg_bytes": alg_bytes, "kernel_ms": round(t_kernel, 4)},
        "stages_ms": {"compress": round(t_compress, 4), "encode": round(t_encode, 4),
                      "decode": round(t_decode, 4)},
        "decode_apply_ms": round(t_apply, 4),  # outside the step: message -> SGD step on w
        "quant": quant,  # outside the step: the same message as 8-bit integers
        "shared": shared,  # outside the step: one index set for all learners
        "compress_gbs": round(4.0 * n / (t_compress / 1e3) / 1e9, 2),
        # the whole compress call against the same peak: 20 B per entry streamed, 0.12 B per
        # entry of sample (12 B per sample at 1%), 24 B per sent entry (index, value, v, u)
        "compress_roofline_frac": round((20.12 * n + 24.0 * int(st["sent"])) /
                                        (t_compress / 1e3) / 1e9 / peak, 4),
        "message_bytes": nb_last,
        "candidates": cand, "sent": int(st["sent"]),
        "gpu_launches": int(launches), "clocks": clk,
        "e2e": e2e, "cpu_baseline": cpu,
    }
    if wl == "bucket1g" and world == 1 and not args.no_workloads:
        # the other workloads and the aggregation, each at its own settings, after the headline
        # bucket's buffers are released
        del graphs, pool, pipe
        torch.cuda.empty_cache()
        flush = L2Flush(dev)
        out["workloads"] = {name: run_workload(name, dev, peak, args.workload_steps, flush=flush)
                            for name in ("single", "resnet50", "deepspeech")}
        out["aggregation"] = run_aggregation(dev, peak, flush=flush)
        del flush
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_e2e(args, pipe, pool, p, K_dev):
    """The same step through the public API with host buffers: each step's gradient comes from
    pinned host memory and its encoded message goes back to the host. The copy of step i+1's
    gradient runs on a second stream into the other half of a device double buffer while step i
    computes, so the link and the kernels overlap."""
    import torch

    n, dev = pipe.n, pipe.dev
    K = max(1, min(args.e2e_steps, K_dev))
    hosts = []
    for i in range(2):
        h = torch.empty(n, dtype=torch.float32, pin_memory=True)
        h.copy_(pool[i % len(pool)])
        hosts.append(h)
    g_dev = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(2)]
    back = torch.empty(pipe.msg_cap, dtype=torch.uint8, pin_memory=True)
    main = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    landed = [E() for _ in range(K + 1)]
    used = [E() for _ in range(K + 1)]
    began = [E() for _ in range(K + 1)]

    def h2d(i):
        with torch.cuda.stream(copy):
            if i >= 2:
                copy.wait_event(used[i - 2])  # the buffer's previous step is done with it
            began[i].record(copy)
            g_dev[i % 2].copy_(hosts[i % 2], non_blocking=True)
            landed[i].record(copy)

    # two untimed steps to settle the buffers
    for i in range(2):
        h2d(i)
        main.wait_event(landed[i])
        pipe.step(g_dev[i % 2], p)
    torch.cuda.synchronize()
    landed = [E() for _ in range(K + 1)]
    used = [E() for _ in range(K + 1)]
    d2h = 0
    a, b = E(), E()
    a.record(main)
    h2d(0)
    for i in range(K):
        if i + 1 < K:
            h2d(i + 1)
        main.wait_event(landed[i])
        pipe.step(g_dev[i % 2], p)
        nb = pipe.message_size()  # the host copies back exactly the message
        used[i].record(main)
        back[:nb].copy_(pipe.msg[:nb], non_blocking=True)
        d2h += nb + 8  # the message and its size
    b.record(main)
    torch.cuda.synchronize()
    sec = a.elapsed_time(b) / 1e3
    copy_each = [round(began[i].elapsed_time(landed[i]), 2) for i in range(K)]
    copy_ms = sorted(copy_each)
    return {"value": round(4.0 * n * K / sec / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": 4 * n, "d2h_bytes_per_step": int(d2h / K), "steps": K,
            "h2d_ms_median": round(copy_ms[len(copy_ms) // 2], 3),
            "h2d_gbs_median": round(4.0 * n / (copy_ms[len(copy_ms) // 2] / 1e3) / 1e9, 1),
            "h2d_ms_each": copy_each,
            "note": "gradient copied from pinned host memory each step on a second stream, "
                    "overlapped with the previous step's kernels; message copied back"}


# -------------------------------------------------------- the other workloads, aggregation
L2_BYTES = 129 * 2**20


class L2Flush:
    """Writes a buffer twice the size of L2 so that the next timed call starts cold."""

    def __init__(self, dev):
        import torch

        self.buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.fill_(1.0)


def median_ms(fn, reps, flush=None, warm=3):
    """Median CUDA-event time of fn() over `reps` calls after `warm` untimed ones; flush() (if
    given) runs before every call, outside the events."""
    import torch

    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ms = []
    for i in range(warm + reps):
        if flush:
            flush()
        a, b = E(), E()
        a.record()
        fn()
        b.record()
        b.synchronize()
        if i >= warm:
            ms.append(a.elapsed_time(b))
    return statistics.median(ms)


def run_workload(name, dev, peak, steps, warmup=3, flush=None):
    """One of the other workloads at its own settings: `warmup` untimed steps, then `steps`
    timed steps (compress, encode and decode as CUDA graph replays), each step
    timed on its own with CUDA events, L2 flushed before each step when its arrays fit in L2."""
    import numpy as np
    import torch

    import sparsified_gradient_compression_gb300 as dgc
    import workloads

    seg = OTHER_WORKLOADS[name][0]()
    n = int(seg[-1])
    p = dgc.make_params(sparsity=0.999, momentum=0.9, seed=SEED, **OTHER_WORKLOADS[name][1])
    pipe = Pipeline(n, [p], dev, seg)
    pool = [torch.from_numpy(workloads.gradient(name, step=i, seed=0, n=n)).to(dev)
            for i in range(2)]
    for i in range(warmup):
        pipe.step(pool[i % 2], p)
    torch.cuda.synchronize()
    if dgc.dgc_read_status(pipe.status) != 0:
        raise RuntimeError(f"{name}: warm-up steps reported an error")
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    gkev = (E(), E())
    dgc.dgc_profile_stream_pass(*gkev)
    graphs = [pipe.capture(g, p) for g in pool]
    dgc.dgc_profile_stream_pass(None, None)
    torch.cuda.synchronize()
    small = 12 * n < L2_BYTES  # g, u and v together fit in L2
    step_ms, st_ms, kern_ms = [], [], []
    for i in range(steps):
        if small and flush:
            flush()
        ev = (E(), E(), E(), E())
        j = (warmup + i) % 2
        pipe.step(pool[j], p, ev, graphs[j])
        torch.cuda.synchronize()
        step_ms.append(ev[0].elapsed_time(ev[3]))
        st_ms.append((ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2]),
                      ev[2].elapsed_time(ev[3])))
        kern_ms.append(gkev[0].elapsed_time(gkev[1]))
    if dgc.dgc_read_status(pipe.status) != 0:
        raise RuntimeError(f"{name}: timed steps reported an error")
    segst = np.frombuffer(pipe.stats.cpu().numpy().tobytes(), dtype=[
        ("k", "<u8"), ("candidates", "<u8"), ("sent", "<u8"), ("thresh_key", "<u4"),
        ("sample_key", "<u4"), ("reselected", "<u4"), ("clip_scale", "<f4"),
        ("clip_sumsq", "<f8")])
    cand, sent = int(segst["candidates"].sum()), int(segst["sent"].sum())
    t_step = statistics.median(step_ms)
    t_comp = statistics.median(x[0] for x in st_ms)
    t_kern = statistics.median(kern_ms)
    clip = p.clip_norm > 0
    pass_bytes = 20.0 * n + 4.0 * cand + 4.0 * ((n + 2047) // 2048)
    comp_bytes = 20.12 * n + (4.0 * n if clip else 0.0) + 24.0 * sent
    out = {"workload": OTHER_WORKLOADS[name][2], "n": n, "segments": int(seg.size - 1),
           "steps": steps, "warmup": warmup, "ms_per_step": round(t_step, 4),
           "value": round(4.0 * n / (t_step / 1e3) / 1e9, 2), "unit": UNIT,
           "stages_ms": {"compress": round(t_comp, 4),
                         "encode": round(statistics.median(x[1] for x in st_ms), 4),
                         "decode": round(statistics.median(x[2] for x in st_ms), 4)},
           "stream_pass": {"kernel_ms": round(t_kern, 4), "alg_bytes": pass_bytes,
                           "frac": round(pass_bytes / (t_kern / 1e3) / 1e9 / peak, 4)},
           "compress_gbs": round(4.0 * n / (t_comp / 1e3) / 1e9, 2),
           "compress_roofline_frac": round(comp_bytes / (t_comp / 1e3) / 1e9 / peak, 4),
           "compress_alg_bytes": comp_bytes, "candidates": cand, "sent": sent,
           "message_bytes": int(pipe.msg_bytes.item()),
           "l2": ("L2 flushed before every step (g, u, v fit in L2)" if small else
                  f"g, u, v together {12 * n >> 20} MiB, larger than L2"),
           "launch": "compress, encode and decode as CUDA graph replays"}
    del pipe, pool, graphs
    torch.cuda.empty_cache()
    return out


def run_aggregation(dev, peak, W=64, n=25_557_032, reps=20, flush=None):
    """The aggregation workload: W learners each compress their own seeded gradient (momentum
    0.9, exact top-k at 99.9%, first step from zero state) and encode it; the W messages are
    then decoded and summed in learner order into one dense array (dgc_decode_accumulate), and
    applied as one SGD step (dgc_decode_apply). Median CUDA-event times of those two calls, L2
    flushed before each."""
    import numpy as np
    import torch

    import sparsified_gradient_compression_gb300 as dgc
    import workloads

    off = np.array([0, n], np.int64)
    p = dgc.make_params(mode=dgc.SELECT_EXACT, sparsity=0.999, momentum=0.9, seed=SEED)
    pipe = Pipeline(n, [p], dev, off)
    msgs, sizes = [], []
    for w in range(W):
        g = torch.from_numpy(workloads.gradient("learners", 0, learner=w, n=n)).to(dev)
        pipe.u.zero_()
        pipe.v.zero_()
        pipe.compress(g, p)
        pipe.encode()
        nb = int(pipe.msg_bytes.item())
        msgs.append(pipe.msg[:nb].clone())
        sizes.append(nb)
    if dgc.dgc_read_status(pipe.status) != 0:
        raise RuntimeError("aggregation: learners reported an error")
    del pipe, g
    torch.cuda.empty_cache()
    ws_bytes = dgc.dgc_decode_workspace(sizes, n)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dense = torch.empty(n, dtype=torch.float32, device=dev)
    w_vec = torch.zeros(n, dtype=torch.float32, device=dev)
    l0 = dgc.dgc_launch_count()
    t_dec_call = median_ms(lambda: dgc.dgc_decode_accumulate(msgs, sizes, dense, n, False, status,
                                                             ws, ws_bytes=ws_bytes), reps, flush)
    launches_dec = (dgc.dgc_launch_count() - l0) // (reps + 3)
    t_app_call = median_ms(lambda: dgc.dgc_decode_apply(msgs, sizes, w_vec, n, 0.01 / W, status,
                                                        ws, ws_bytes=ws_bytes), reps, flush)
    # the same two calls as a trainer replays them each step: the sizes in device memory (as
    # dgc_encode leaves them), each call captured once into a CUDA graph (the message table
    # travels in the kernels' parameters up to 96 messages)
    t_dec, t_app, launch = t_dec_call, t_app_call, "host calls"
    if W <= 96:
        sizes_dev = torch.tensor(sizes, dtype=torch.int64, device=dev)
        ws_dev = torch.empty(dgc.dgc_decode_workspace_bound(sizes, n), dtype=torch.uint8,
                             device=dev)
        acc_call = lambda: dgc.dgc_decode_accumulate_dev(  # noqa: E731
            msgs, sizes_dev, sizes, dense, n, False, status, ws_dev)
        app_call = lambda: dgc.dgc_decode_apply_dev(  # noqa: E731
            msgs, sizes_dev, sizes, w_vec, n, 0.01 / W, status, ws_dev)
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        graphs = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph())
        with torch.cuda.stream(side):
            acc_call()
            app_call()
            with torch.cuda.graph(graphs[0], stream=side):
                acc_call()
            with torch.cuda.graph(graphs[1], stream=side):
                app_call()
        torch.cuda.current_stream(dev).wait_stream(side)
        t_dec = median_ms(graphs[0].replay, reps, flush)
        t_app = median_ms(graphs[1].replay, reps, flush)
        launch = "CUDA graph replays of dgc_decode_accumulate_dev / dgc_decode_apply_dev"
    if dgc.dgc_read_status(status) != 0:
        raise RuntimeError("aggregation: decode reported an error")
    tokens = sum((s - 32) // 6 for s in sizes)  # values + escapes (the pad is under 6 bytes)
    touched = int((dense != 0).sum().item())  # positions some message reached (sum not 0)
    msg_bytes = float(sum(sizes))
    dec_bytes = msg_bytes + 4.0 * n + 8.0 * tokens
    app_bytes = msg_bytes + 8.0 * tokens + 8.0 * touched
    out = {"workload": f"{W} learners x {n:,} fp32 entries, N(0, 0.01^2) each; messages from "
                       "dgc_compress (exact top-k, 99.9%, momentum 0.9, first step) + dgc_encode;"
                       " decode and sum in learner order 0..W-1",
           "learners": W, "n": n, "message_bytes_total": int(msg_bytes), "tokens": tokens,
           "decode_ms": round(t_dec, 4), "decode_apply_ms": round(t_app, 4),
           "value": round(4.0 * n / (t_dec / 1e3) / 1e9, 2),
           "unit": "GB/s of dense fp32 gradient produced",
           "decode_roofline": {"bound": "hbm", "alg_bytes": dec_bytes,
                               "achieved": round(dec_bytes / (t_dec / 1e3) / 1e9, 1),
                               "frac": round(dec_bytes / (t_dec / 1e3) / 1e9 / peak, 4),
                               "bytes_rule": "messages read + 4 B per dense entry written + "
                                             "8 B per token (position written and read)"},
           "decode_apply_roofline": {"bound": "hbm", "alg_bytes": app_bytes,
                                     "achieved": round(app_bytes / (t_app / 1e3) / 1e9, 1),
                                     "frac": round(app_bytes / (t_app / 1e3) / 1e9 / peak, 4),
                                     "bytes_rule": "messages read + 8 B per token + 8 B per "
                                                   "touched weight (read and write)"},
           "touched": touched, "launches_per_decode": launches_dec, "launch": launch,
           "host_call_ms": {"decode": round(t_dec_call, 4), "decode_apply": round(t_app_call, 4)},
           "l2": "L2 flushed before every call (the 102 MB dense array fits in L2)"}
    del msgs, ws, dense, w_vec
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ CPU baseline / reference
def host_cpu() -> dict:
    """The host CPU's model name (lscpu, else /proc/cpuinfo) and the cores it reports."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu model")):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    import platform

    return {"cpu_model": model or platform.processor() or platform.machine(),
            "nproc": os.cpu_count()}


def run_cpu_baseline(n_cpu: int, steps: int, select: str = "sampled", bin_size: int = 1000):
    """The oracle, single-threaded on one host core, on a bounded sample of the workload:
    an n_cpu-entry bucket with the same recipe (one untimed step, then `steps` timed steps of
    compress + encode + decode at 99.9%)."""
    import numpy as np

    import oracle
    import workloads

    mode = oracle.ADACOMP if select == "adacomp" else oracle.SAMPLED
    p = oracle.make_params(mode, 0.999, 0.9, sample_ratio=0.01, reselect_factor=1.3, seed=SEED,
                           bin_size=bin_size)
    off = np.array([0, n_cpu], np.int64)
    u = np.zeros(n_cpu, np.float32)
    v = np.zeros(n_cpu, np.float32)
    gs = [workloads.gradient("bucket1g", step=i, seed=0, n=n_cpu) for i in range(2)]
    idx, val, _ = oracle.compress(gs[0], u, v, off, p)
    t0 = time.perf_counter()
    for i in range(steps):
        idx, val, _ = oracle.compress(gs[(i + 1) % 2], u, v, off, p)
        m = oracle.encode(idx, val, n_cpu)
        oracle.decode_accumulate([m], n_cpu)
    sec = time.perf_counter() - t0
    return {"value": round(4.0 * n_cpu * steps / sec / 1e9, 4), "unit": UNIT, "cores": 1,
            "kind": "oracle", "seconds": round(sec, 2), **host_cpu(),
            "sample": f"{n_cpu}-entry bucket of the same recipe, {steps} timed steps of "
                      "compress+encode+decode at 99.9% after one untimed step"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    steps = max(1, args.steps)
    # keep the whole run to a few minutes: about 40 ns per entry per step on one core
    n_ref = 1 << 26
    while n_ref > (1 << 16) and steps * n_ref * 40e-9 > 120:
        n_ref >>= 1
    cpu = run_cpu_baseline(n_ref, steps, select=args.select, bin_size=args.bin_size)
    out = {"impl": "reference", "metric": METRIC, "value": cpu["value"], "unit": UNIT,
           "n_gpus": world, "steps": steps, "warmup": args.warmup,
           "ms_per_step": round(cpu["seconds"] * 1e3 / steps, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic (seeded; see workloads/)",
           "config": {"workload": WORKLOAD if args.select == "sampled"
                      else WORKLOAD_ADACOMP.format(args.bin_size), "n": n_ref,
                      "sample_of_n": args.n, "selection": args.select},
           "cpu_baseline": cpu,
           "e2e": {"value": cpu["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return 0
    run_ours(args, world, rank, local)
    return 0


if __name__ == "__main__":
    sys.exit(main())
