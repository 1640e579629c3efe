"""The oracle side of the aggregation workload, one learner per call, for a spawned process pool.

Each of W learners compresses its own seeded gradient stream (25,557,032 entries, N(0, 0.01^2),
momentum 0.9, exact top-k at 99.9%, no clipping) and encodes every step's result; the receiver
decodes and sums the W messages of a step in learner order. The oracle's exact top-k sorts all
entries, about 5 s per learner and step on one core, so the tests run the learners in worker
processes. This module imports neither torch nor the CUDA library: the workers it serves are
started with the spawn method and never touch the GPU.
"""
from __future__ import annotations

import hashlib

import numpy as np

N_LEARNER = 25_557_032


def learner_messages(learner: int, steps: int, n: int = N_LEARNER):
    """The learner's encoded messages for steps 0..steps-1 and SHA-256 digests of its momentum
    and residual after the last step."""
    import oracle
    import workloads

    oracle.lib()
    off = np.array([0, n], np.int64)
    p = oracle.make_params(mode=oracle.EXACT, sparsity=0.999, momentum=0.9)
    u = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    msgs = []
    for t in range(steps):
        g = workloads.gradient("learners", t, learner=learner, n=n)
        idx, val, _ = oracle.compress(g, u, v, off, p)
        msgs.append(oracle.encode(idx, val, n))
    return (msgs, hashlib.sha256(u.tobytes()).hexdigest(),
            hashlib.sha256(v.tobytes()).hexdigest())
