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
