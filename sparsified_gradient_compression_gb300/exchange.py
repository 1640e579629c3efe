"""The learners' message exchange: every rank's encoded message to every rank, then one decode.

Synchronous data-parallel SGD sums every learner's update ("[Paper Review] Deep Gradient
Compression", Abstract and Motivation & Objective). The learners' sparse messages cannot be
summed by an all-reduce, since each learner sends its own index set (the all-reduce page,
abstract: most compressed gradients cannot be aggregated with all-reduce). They are gathered
instead, and every rank decodes them in rank order. The exchange is three steps:

1. an all-gather of the message sizes (one int64 per rank), read back to the host, since the
   decoders take message sizes on the host;
2. an all-gather of the bytes, each rank's message in a slot of the largest size rounded up to
   16 bytes, so that one equal-size collective moves every message and every received message
   starts on a 16-byte boundary, as the decoders require;
3. dgc_decode_apply (the SGD step on the weights) or dgc_decode_accumulate (the dense sum) over
   the received messages, rank 0 first, on this rank's GPU.

Steps 1 and 2 are plain torch.distributed collectives (NCCL on GPUs, gloo on host tensors) and
hold none of the method's arithmetic; step 3 runs in the CUDA library. Ranks in the same group
must call these functions in the same order.

ScaleComp's shared index set (ScaleComp, abstract: a compressor whose results add up across
learners, so that the exchange can be all-reduce compatible) takes a different exchange. One
learner chooses the set S (dgc_compress), broadcast_index_set sends S to every rank, the others
send at S (dgc_compress_shared), and exchange_shared_sum adds the learners' value vectors. It
gathers the vectors and adds them in rank order with dgc_sum_shared rather than reducing them in
the collective: a reduction's order of additions is the library's to choose, while the learners'
order gives every rank, and the oracle, the same bits.
"""
from __future__ import annotations

SLOT_ALIGN = 16


def slot_bytes(sizes) -> int:
    """The slot every rank's message is padded to: the largest size rounded up to 16 bytes."""
    m = max((int(s) for s in sizes), default=0)
    return max(SLOT_ALIGN, (m + SLOT_ALIGN - 1) // SLOT_ALIGN * SLOT_ALIGN)


def allgather_sizes(nbytes, group=None, device=None):
    """Every rank's message size in rank order, as host ints. `nbytes` is this rank's size: an
    int, or a one-element int64 tensor (for instance dgc_encode's device-side byte count)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if isinstance(nbytes, torch.Tensor):
        mine = nbytes.reshape(1).to(dtype=torch.int64)
        if device is not None:
            mine = mine.to(device)
    else:
        mine = torch.tensor([int(nbytes)], dtype=torch.int64, device=device)
    parts = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(parts, mine, group=group)
    return [int(p.item()) for p in parts]


def allgather_messages(msg, nbytes, group=None, recv=None):
    """Every rank's encoded message, rank 0 first: (list of uint8 views of the received bytes,
    list of their sizes). `msg` is this rank's message buffer (uint8 tensor on this rank's
    device, at least nbytes long); `recv`, if given, is a uint8 tensor of at least
    world * slot_bytes(sizes) bytes that receives the slots (reused across steps)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    sizes = allgather_sizes(nbytes, group, msg.device)
    me = dist.get_rank(group)
    if msg.numel() < sizes[me]:
        raise ValueError(f"message buffer holds {msg.numel()} bytes, the message {sizes[me]}")
    slot = slot_bytes(sizes)
    send = torch.zeros(slot, dtype=torch.uint8, device=msg.device)
    send[: sizes[me]].copy_(msg.reshape(-1)[: sizes[me]])
    if recv is None:
        recv = torch.empty(world * slot, dtype=torch.uint8, device=msg.device)
    elif recv.numel() < world * slot or recv.dtype != torch.uint8:
        raise ValueError(f"receive buffer needs {world * slot} uint8 entries")
    slots = [recv[r * slot:(r + 1) * slot] for r in range(world)]
    dist.all_gather(slots, send, group=group)
    return [slots[r][: sizes[r]] for r in range(world)], sizes


def exchange_workspace_bytes(max_message_bytes: int, world: int, n: int) -> int:
    """Decoder workspace that serves any exchange of `world` messages of at most
    max_message_bytes each over n entries (dgc_decode_workspace at the worst case)."""
    from . import dgc_decode_workspace

    return dgc_decode_workspace([int(max_message_bytes)] * int(world), n)


def exchange_and_apply(msg, nbytes, w, n: int, lr: float, status, ws, group=None, recv=None,
                       ws_bytes: int | None = None):
    """Gather every rank's message and take the SGD step w <- fma(-lr, sum in rank order, w) on
    this rank's weights (dgc_decode_apply). Returns the received message sizes."""
    from . import dgc_decode_apply

    views, sizes = allgather_messages(msg, nbytes, group, recv)
    dgc_decode_apply(views, sizes, w, n, lr, status, ws, ws_bytes=ws_bytes)
    return sizes


def exchange_and_decode(msg, nbytes, dense, n: int, status, ws, accumulate: bool = False,
                        group=None, recv=None, ws_bytes: int | None = None):
    """Gather every rank's message and sum them in rank order into dense
    (dgc_decode_accumulate). Returns the received message sizes."""
    from . import dgc_decode_accumulate

    views, sizes = allgather_messages(msg, nbytes, group, recv)
    dgc_decode_accumulate(views, sizes, dense, n, accumulate, status, ws, ws_bytes=ws_bytes)
    return sizes


def _as_int32(t):
    """A uint32 or int32 tensor as int32 (the collectives carry int32; the bits are unchanged)."""
    import torch

    if t.dtype == torch.int32:
        return t
    if t.dtype == torch.uint32:
        return t.view(torch.int32)
    raise TypeError(f"index set must be uint32 or int32, not {t.dtype}")


def broadcast_index_set(idx, count, src: int, group=None) -> int:
    """The shared index set chosen on rank `src` to every rank: the count (a one-element int64
    tensor, as dgc_compress writes it), then idx[:count]. Both are written in place on the other
    ranks, whose idx must hold the count; returns the count as a host int."""
    import torch.distributed as dist

    dist.broadcast(count, src, group=group)
    c = int(count.reshape(-1)[0].item())
    if c < 0 or c > idx.numel():
        raise ValueError(f"index set of {c} entries, buffer of {idx.numel()}")
    if c > 0:  # (a leading slice of a flat tensor: contiguous, received in place)
        dist.broadcast(_as_int32(idx.reshape(-1))[:c], src, group=group)
    return c


def allgather_values(vals, count: int, group=None, recv=None):
    """Every rank's value vector at the shared index set, rank 0 first: a list of float32 views
    of `count` entries each. One equal-size all-gather moves them (every rank sends at the same
    set, so every vector has the same length); `recv`, if given, is a float32 tensor of at least
    world * count entries that receives them."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    count = int(count)
    if vals.dtype != torch.float32 or vals.numel() < count:
        raise ValueError(f"value vector needs {count} float32 entries")
    if recv is None:
        recv = torch.empty(max(world * count, 1), dtype=torch.float32, device=vals.device)
    elif recv.dtype != torch.float32 or recv.numel() < world * count:
        raise ValueError(f"receive buffer needs {world * count} float32 entries")
    parts = [recv[r * count:(r + 1) * count] for r in range(world)]
    if count > 0:
        dist.all_gather(parts, vals.reshape(-1)[:count].contiguous(), group=group)
    return parts


def exchange_shared_sum(vals, count, out, status, ws, group=None, recv=None,
                        ws_bytes: int | None = None) -> int:
    """Gather every rank's value vector at the shared index set and add them in rank order into
    out (dgc_sum_shared: out[j] = the rank-ordered sum from +0). `count` is the set's size as a
    one-element device int64 tensor (the same on every rank); `ws` holds
    dgc_sum_shared_workspace(world) bytes. Returns the count."""
    from . import dgc_sum_shared

    c = int(count.reshape(-1)[0].item())
    parts = allgather_values(vals, c, group, recv)
    dgc_sum_shared(parts, count, max(c, 1), out, status, ws, ws_bytes=ws_bytes)
    return c
