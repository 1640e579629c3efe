"""The learners' message exchange on CPU: gloo ranks on 127.0.0.1 gather each other's messages.

Each rank compresses and encodes its own gradient with the oracle (the messages differ in size,
one is empty), gathers every rank's message through the package's exchange helper (sizes first,
then the bytes in 16-byte slots), and decodes what it received with the oracle. Every rank must
receive exactly the bytes every other rank sent, in rank order, and its decoded sum and SGD step
must equal the oracle's on the messages themselves, bit for bit. The helper's third step, the
decode on the GPU, is the library's dgc_decode_* call that the GPU tests cover.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from sparsified_gradient_compression_gb300 import exchange

N = 200_003
SPARSITY = (0.999, 0.99, 1.0, 0.9)  # rank 2 sends nothing (an empty, 32-byte message)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _messages(world, steps):
    """Every rank's oracle messages, [step][rank], from its own seeded gradients and state."""
    import oracle
    import workloads

    out = [[None] * world for _ in range(steps)]
    off = np.array([0, N], np.int64)
    for r in range(world):
        p = oracle.make_params(mode=oracle.EXACT, sparsity=SPARSITY[r], momentum=0.9)
        u = np.zeros(N, np.float32)
        v = np.zeros(N, np.float32)
        for t in range(steps):
            g = workloads.misc([80, r, t], N, 0.01)
            idx, val, _ = oracle.compress(g, u, v, off, p)
            out[t][r] = oracle.encode(idx, val, N)
    return out


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist

    import oracle

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        steps = 2
        msgs = _messages(world, steps)
        recv = None
        for t in range(steps):
            mine = msgs[t][rank]
            # this rank's buffer is larger than its message; the bytes past it must not travel
            buf = torch.full((len(mine) + 40,), 0xAB, dtype=torch.uint8)
            buf[: len(mine)] = torch.frombuffer(bytearray(mine), dtype=torch.uint8)
            nbytes = torch.tensor([len(mine)], dtype=torch.int64) if rank % 2 else len(mine)
            views, sizes = exchange.allgather_messages(buf, nbytes, recv=recv)
            assert sizes == [len(m) for m in msgs[t]]
            slot = exchange.slot_bytes(sizes)
            base = views[0].data_ptr()
            for r in range(world):
                assert views[r].numpy().tobytes() == msgs[t][r], (t, r)
                assert (views[r].data_ptr() - base) % 16 == 0 and views[r].data_ptr() % 16 == 0
                assert views[r].data_ptr() - base == r * slot
            got = [v.numpy().tobytes() for v in views]
            rc, dense = oracle.decode_accumulate(got, N)
            rc0, want = oracle.decode_accumulate(msgs[t], N)
            assert rc == 0 and rc0 == 0
            assert np.array_equal(dense.view(np.uint32), want.view(np.uint32))
            w0 = np.random.Generator(np.random.PCG64([81, t])).standard_normal(N).astype(
                np.float32)
            rc, w = oracle.decode_apply(got, N, w0, np.float32(0.1 / world))
            rc0, w_want = oracle.decode_apply(msgs[t], N, w0, np.float32(0.1 / world))
            assert rc == 0 and rc0 == 0
            assert np.array_equal(w.view(np.uint32), w_want.view(np.uint32))
            # the next step reuses a receive buffer large enough for any of its slots
            recv = torch.empty(world * 4096 * 16, dtype=torch.uint8)
        with pytest.raises(ValueError):  # a buffer shorter than the size it claims
            exchange.allgather_messages(torch.zeros(8, dtype=torch.uint8), 64)
        q.put((rank, "ok"))
    except Exception as e:  # reported through the queue, the exit code says the rest
        q.put((rank, repr(e)))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_exchange_messages_and_decode_in_rank_order(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert res == [(r, "ok") for r in range(world)], res
    assert all(p.exitcode == 0 for p in procs)


def test_slot_rule():
    assert exchange.slot_bytes([]) == 16
    assert exchange.slot_bytes([32]) == 32
    assert exchange.slot_bytes([32, 33, 40]) == 48
    assert exchange.slot_bytes([0, 1]) == 16
    assert exchange.slot_bytes([4096 * 16]) == 4096 * 16


def _shared_rank_main(rank, world, port, q):
    # ScaleComp's shared index set across gloo ranks: learner t mod world chooses the set with
    # the oracle's compressor, broadcast_index_set sends it, every other rank sends at it
    # (the oracle's compress_shared) and allgather_values brings every rank's value vector back,
    # rank 0 first. Each rank also runs every learner's steps itself, so it knows what each rank
    # must have sent; its rank-ordered sum of what it received must equal the oracle's sum of
    # those vectors, bit for bit.
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist

    import oracle
    import workloads

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        off = np.array([0, N], np.int64)
        p = oracle.make_params(mode=oracle.SAMPLED, sparsity=0.999, momentum=0.9, seed=5,
                               leak=0.9)
        cap = oracle.max_out(N)
        state = [[np.zeros(N, np.float32), np.zeros(N, np.float32)] for _ in range(world)]
        idx_buf = torch.zeros(cap, dtype=torch.int32)
        count = torch.zeros(1, dtype=torch.int64)
        for t in range(3):
            lead = t % world
            grads = [workloads.misc([83, r, t], N, 0.01) for r in range(world)]
            # every learner's step, as each rank would take it
            sidx, lead_val, _ = oracle.compress(grads[lead], *state[lead], off, p)
            want = [None] * world
            want[lead] = lead_val
            for r in range(world):
                if r != lead:
                    rc, want[r] = oracle.compress_shared(grads[r], *state[r], off, p, sidx)
                    assert rc == 0
            # the set travels from the chooser; the other ranks' buffers start as garbage
            if rank == lead:
                idx_buf[: sidx.size] = torch.from_numpy(sidx.astype(np.int64)).to(torch.int32)
                count[0] = sidx.size
            else:
                idx_buf.fill_(-7)
                count[0] = -1
            c = exchange.broadcast_index_set(idx_buf, count, lead)
            assert c == sidx.size and int(count[0]) == c
            assert np.array_equal(idx_buf[:c].numpy().view(np.uint32), sidx.astype(np.uint32))
            mine = torch.full((c + 5,), float("nan"), dtype=torch.float32)
            mine[:c] = torch.from_numpy(want[rank])
            parts = exchange.allgather_values(mine, c)
            assert len(parts) == world
            for r in range(world):
                assert np.array_equal(parts[r].numpy().view(np.uint32), want[r].view(np.uint32))
            rc, got = oracle.sum_shared([x.numpy() for x in parts])
            rc0, total = oracle.sum_shared(want)
            assert rc == 0 and rc0 == 0
            assert np.array_equal(got.view(np.uint32), total.view(np.uint32))
        with pytest.raises(ValueError):  # a vector shorter than the set
            exchange.allgather_values(torch.zeros(2, dtype=torch.float32), 3)
        q.put((rank, "ok"))
    except Exception as e:  # reported through the queue, the exit code says the rest
        q.put((rank, repr(e)))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_share_an_index_set_and_gather_values_in_rank_order(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shared_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert res == [(r, "ok") for r in range(world)], res
    assert all(p.exitcode == 0 for p in procs)
