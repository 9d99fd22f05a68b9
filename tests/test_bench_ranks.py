"""The benchmark's host logic on CPU.  Multi-rank (gloo, two ranks): the step
time is the slowest rank's, the value counts every rank's rows (weak
scaling), and the reference arm runs on rank 0 only.  The traffic lookup:
the captured ratio for the nearest query count, none for a changed source.
No GPU is involved."""
import os
import socket
import types

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = [12.5, 20.0][rank]  # rank 1 is the slower one
        total = bench.max_over_ranks(local_ms, torch.device("cpu"))
        steps, rows = 10, 32 * 2048 * 4
        value = bench.whole_job_rows_per_s(world, rows, total / steps)
        ref = bench.run_reference(types.SimpleNamespace(steps=1, warmup=0), rank, world) \
            if rank == 1 else "skipped"
        q.put((rank, total, value, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_rows():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = {r: (t, v, ref) for r, t, v, ref in got}
    for r in (0, 1):
        t, v, _ = by_rank[r]
        assert t == 20.0                                     # the slowest rank's time
        assert v == pytest.approx(2 * 32 * 2048 * 4 / (2.0 / 1e3))  # both ranks' rows
    assert by_rank[1][2] is None                             # the reference arm: rank 0 only


def test_traffic_ratio_by_query_count_and_stale_source(monkeypatch):
    """A stage's DRAM traffic is its captured ratio x its algorithmic bytes:
    the ratio of the nearest captured query count, and none once the
    kernel's source no longer matches the captured one."""
    import bench
    monkeypatch.setitem(bench.TRAFFIC, "indexer_tc_kernel",
                        ("indexer.cu", bench._src_sha("indexer.cu"), {1: 0.5, 4: 2.0}))
    assert bench.traffic_of("indexer_tc_kernel", 100.0, 1) == 50.0
    assert bench.traffic_of("indexer_tc_kernel", 100.0, 4) == 200.0
    assert bench.traffic_of("indexer_tc_kernel", 100.0, 2) == 50.0   # nearer to 1
    assert bench.traffic_of("indexer_tc_kernel", 100.0, 3) == 200.0  # nearer to 4
    assert bench.traffic_of("indexer_tc_kernel", 100.0, 8) == 200.0
    assert bench.traffic_of("indexer_tc_kernel", 0.0, 1) is None
    monkeypatch.setitem(bench.TRAFFIC, "indexer_tc_kernel", ("indexer.cu", "0" * 16, 1.0))
    assert bench.traffic_of("indexer_tc_kernel", 100.0) is None
    assert bench.traffic_of("no_such_kernel", 100.0) is None
