"""bench.py's multi-rank logic on CPU: two gloo ranks (127.0.0.1), max-over-ranks timing and the
whole-job throughput, plus the roofline bookkeeping that needs no GPU."""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    bench.barrier()
    seconds = [1.5, 2.0][rank]  # rank 1 is the slow one
    sec_max = bench.max_over_ranks(seconds)
    value = bench.whole_job_value(4.0 * 1000, world, sec_max)
    q.put((rank, sec_max, value))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_report_max_time_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, sec_max, value in res:
        assert sec_max == 2.0
        assert value == 4.0 * 1000 * 2 / 2.0


def test_single_process_aggregation_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_value(10.0, 1, 2.0) == 5.0


def test_traffic_record_ignored_when_source_changed(tmp_path, monkeypatch):
    assert isinstance(bench.stream_pass_source_hash(), str)
    peak, kind = bench.measured_peak_hbm()
    assert peak > 1000 and kind in ("measured", "fallback")
