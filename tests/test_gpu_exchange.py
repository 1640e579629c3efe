"""The message exchange's device path on one GPU: a one-rank NCCL group.

With one rank the gather returns this rank's own message, so exchange_and_apply and
exchange_and_decode must give exactly what dgc_decode_apply and dgc_decode_accumulate give on the
message itself, and both must match the oracle. This runs the NCCL collectives on device buffers,
the 16-byte slots and the decode of the received views; the rank order and sizes of several
ranks are covered by the gloo tests on CPU (no call here uses more than one GPU).
"""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
import sparsified_gradient_compression_gb300 as dgc
import workloads
from sparsified_gradient_compression_gb300 import exchange

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture()
def one_rank_nccl():
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    yield
    dist.destroy_process_group()


def test_one_rank_exchange_equals_the_decoders(one_rank_nccl):
    dgc.build()
    n = 1_048_576
    off = np.array([0, n], np.int64)
    g = workloads.gradient("single", 0)
    po = oracle.make_params(mode=oracle.EXACT, sparsity=0.999, momentum=0.9)
    idx, val, _ = oracle.compress(g, np.zeros(n, np.float32), np.zeros(n, np.float32), off, po)
    m = oracle.encode(idx, val, n)
    msg = torch.zeros(len(m) + 100, dtype=torch.uint8, device="cuda")
    msg[: len(m)] = torch.frombuffer(bytearray(m), dtype=torch.uint8).cuda()
    nbytes = torch.tensor([len(m)], dtype=torch.int64, device="cuda")
    ws_bytes = exchange.exchange_workspace_bytes(len(m), 1, n)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    dense = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    sizes = exchange.exchange_and_decode(msg, nbytes, dense, n, status, ws, ws_bytes=ws_bytes)
    assert sizes == [len(m)] and dgc.dgc_read_status(status) == 0
    _, want = oracle.decode_accumulate([m], n)
    assert np.array_equal(dense.cpu().numpy().view(np.uint32), want.view(np.uint32))

    w0 = np.random.Generator(np.random.PCG64([82])).standard_normal(n).astype(np.float32)
    w = torch.from_numpy(w0).cuda()
    sizes = exchange.exchange_and_apply(msg, nbytes, w, n, 0.05, status, ws, ws_bytes=ws_bytes)
    assert sizes == [len(m)] and dgc.dgc_read_status(status) == 0
    _, w_want = oracle.decode_apply([m], n, w0, np.float32(0.05))
    assert np.array_equal(w.cpu().numpy().view(np.uint32), w_want.view(np.uint32))


def test_one_rank_shared_set_exchange_equals_the_oracle(one_rank_nccl):
    # ScaleComp's shared-set path through NCCL on one rank: the set broadcast from rank 0, the
    # value vector at it gathered, and the rank-ordered sum (dgc_sum_shared) on the device; with
    # one rank the sum is +0 + x, which must equal the oracle's bit for bit
    dgc.build()
    n = 1_048_576
    off = np.array([0, n], np.int64)
    g = workloads.gradient("single", 0)
    po = oracle.make_params(mode=oracle.SAMPLED, sparsity=0.999, momentum=0.9, seed=3, leak=0.9)
    sidx, val, _ = oracle.compress(g, np.zeros(n, np.float32), np.zeros(n, np.float32), off, po)
    c = int(sidx.size)
    cap = c + 64
    idx = torch.zeros(cap, dtype=torch.int32, device="cuda")
    idx[:c] = torch.from_numpy(sidx.astype(np.int64)).to(torch.int32).cuda()
    count = torch.tensor([c], dtype=torch.int64, device="cuda")
    assert exchange.broadcast_index_set(idx, count, 0) == c
    assert np.array_equal(idx[:c].cpu().numpy().view(np.uint32), sidx.astype(np.uint32))
    vals = torch.full((cap,), float("nan"), dtype=torch.float32, device="cuda")
    vals[:c] = torch.from_numpy(val).cuda()
    out = torch.full((cap,), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(dgc.dgc_sum_shared_workspace(1), 16), dtype=torch.uint8, device="cuda")
    assert exchange.exchange_shared_sum(vals, count, out, status, ws) == c
    assert dgc.dgc_read_status(status) == 0
    rc, want = oracle.sum_shared([val])
    assert rc == 0
    assert np.array_equal(out[:c].cpu().numpy().view(np.uint32), want.view(np.uint32))
