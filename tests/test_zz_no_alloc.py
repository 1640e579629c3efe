"""dgc_compress_noalloc: the compressor entry point for callers that cannot allocate device memory.

Such callers (a framework whose allocator owns all device memory, code running during CUDA graph
capture or in a loop where cudaMalloc is not allowed) cannot pass a workspace; this entry point
works in a scratch array the library keeps on each GPU. Its results must equal those of
dgc_compress with a caller-allocated workspace, call after call, since it runs the same pipeline.

This file is collected last on purpose, and it must pass both on its own in a fresh process (the
first call then also resolves the scratch address) and after every other test.
"""
import numpy as np
import pytest
import torch

import sparsified_gradient_compression_gb300 as dgc
import workloads

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _state(n):
    return torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")


def _outputs(cap, nseg):
    return (torch.empty(cap, dtype=torch.int32, device="cuda"),
            torch.empty(cap, dtype=torch.float32, device="cuda"),
            torch.zeros(1, dtype=torch.int64, device="cuda"),
            torch.zeros(nseg * dgc.STATS_BYTES, dtype=torch.uint8, device="cuda"),
            torch.zeros(1, dtype=torch.int32, device="cuda"))


@pytest.mark.parametrize("mode", [dgc.SELECT_EXACT, dgc.SELECT_SAMPLED])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(mode):
    # the 1,048,576-entry single-tensor workload, 99.9% sparsity, two calls in a row
    dgc.build()
    n = 1_048_576
    off = torch.tensor([0, 600_000, n], dtype=torch.int64, device="cuda")
    p = dgc.make_params(mode=mode, sparsity=0.999, momentum=0.9, sample_ratio=0.01, seed=3)
    cap = dgc.dgc_compress_max_out(n, 2, p)
    ws = torch.empty(dgc.dgc_compress_workspace(n, 2, p), dtype=torch.uint8, device="cuda")
    u_a, v_a = _state(n)
    u_b, v_b = _state(n)
    oa, ob = _outputs(cap, 2), _outputs(cap, 2)
    for step in range(2):
        g = torch.from_numpy(workloads.gradient("single", step)).cuda()
        dgc.dgc_compress(g, u_a, v_a, off, p, oa[0], oa[1], oa[2], oa[3], oa[4], ws)
        dgc.dgc_compress_noalloc(g, u_b, v_b, off, p, ob[0], ob[1], ob[2], ob[3], ob[4])
        assert dgc.dgc_read_status(oa[4]) == 0
        assert dgc.dgc_read_status(ob[4]) == 0
        ca, cb = int(oa[2].item()), int(ob[2].item())
        assert ca == cb and ca > 0
        # bitwise equality: the tolerance every parity test in this suite uses
        assert torch.equal(oa[0][:ca], ob[0][:cb])
        assert torch.equal(oa[1][:ca].view(torch.int32), ob[1][:cb].view(torch.int32))
        assert torch.equal(oa[3], ob[3])
        assert torch.equal(u_a.view(torch.int32), u_b.view(torch.int32))
        assert torch.equal(v_a.view(torch.int32), v_b.view(torch.int32))


class _Problem:
    """One compressor problem run twice side by side: through dgc_compress_noalloc (the shared
    scratch) and through dgc_compress on a workspace of its own, allocated fresh for each call."""

    def __init__(self, n, off, params, gen):
        self.n, self.params, self.gen = n, params, gen
        self.off = torch.tensor(off, dtype=torch.int64, device="cuda")
        self.nseg = len(off) - 1
        self.cap = dgc.dgc_compress_max_out(n, self.nseg, params)
        self.ws_bytes = dgc.dgc_compress_workspace(n, self.nseg, params)
        self.u_a, self.v_a = _state(n)
        self.u_b, self.v_b = _state(n)
        self.step = 0

    def run_and_compare(self):
        g = self.gen(self.step)
        self.step += 1
        oa, ob = _outputs(self.cap, self.nseg), _outputs(self.cap, self.nseg)
        ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device="cuda")
        dgc.dgc_compress(g, self.u_a, self.v_a, self.off, self.params, oa[0], oa[1], oa[2],
                         oa[3], oa[4], ws)
        dgc.dgc_compress_noalloc(g, self.u_b, self.v_b, self.off, self.params, ob[0], ob[1],
                                 ob[2], ob[3], ob[4])
        assert dgc.dgc_read_status(oa[4]) == 0
        assert dgc.dgc_read_status(ob[4]) == 0
        ca, cb = int(oa[2].item()), int(ob[2].item())
        assert ca == cb and ca > 0
        assert torch.equal(oa[0][:ca], ob[0][:cb])
        assert torch.equal(oa[1][:ca].view(torch.int32), ob[1][:cb].view(torch.int32))
        assert torch.equal(oa[3], ob[3])
        assert torch.equal(self.u_a.view(torch.int32), self.u_b.view(torch.int32))
        assert torch.equal(self.v_a.view(torch.int32), self.v_b.view(torch.int32))


def test_noalloc_different_problems_in_turn_share_the_scratch_safely():
    # Problems that leave different things in the shared array for each other: a sampled call
    # (sample-position cache filled for its seed and layout), an exact call with clipping on
    # another segment layout (which moves where the cache sits in the scratch), an AdaComp call
    # (bin maxima), then the first problem again, whose cached positions must be rebuilt or
    # recognised, never reused stale. Each call is compared bitwise with dgc_compress on a
    # workspace of its own.
    dgc.build()
    n_a = 1_048_576

    def grad_a(t):
        return torch.from_numpy(workloads.gradient("single", t)).cuda()

    a = _Problem(n_a, [0, 600_000, n_a],
                 dgc.make_params(mode=dgc.SELECT_SAMPLED, sparsity=0.999, momentum=0.9,
                                 sample_ratio=0.01, seed=3), grad_a)
    n_b = 900_001
    b = _Problem(n_b, [0, 1, 70_000, 70_000, 400_003, n_b],
                 dgc.make_params(mode=dgc.SELECT_EXACT, sparsity=0.99, momentum=0.9,
                                 clip_norm=0.05),
                 lambda t: torch.from_numpy(workloads.misc([71, t], n_b, 0.01)).cuda())
    n_c = 1_000_003
    c = _Problem(n_c, [0, 333_333, n_c],
                 dgc.make_params(mode=dgc.SELECT_ADACOMP, momentum=0.9, bin_size=1000),
                 lambda t: torch.from_numpy(workloads.misc([72, t], n_c, 0.01)).cuda())
    for prob in (a, b, c, a, b, c, a):
        prob.run_and_compare()


def test_noalloc_rejects_problems_larger_than_its_scratch():
    n = 4_000_000  # needs ~32 MiB of scratch, more than the 16 MiB the library holds
    p = dgc.make_params()
    g = torch.zeros(n, device="cuda")
    u, v = _state(n)
    o = _outputs(dgc.dgc_compress_max_out(n, 1, p), 1)
    off = torch.tensor([0, n], dtype=torch.int64, device="cuda")
    with pytest.raises(dgc.DGCError) as e:
        dgc.dgc_compress_noalloc(g, u, v, off, p, o[0], o[1], o[2], o[3], o[4])
    assert e.value.code == dgc.EUNSUPPORTED
    assert dgc.dgc_read_status(o[4]) == 0
    assert not u.any() and not v.any()
