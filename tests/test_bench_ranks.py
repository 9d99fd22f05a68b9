"""The benchmark's host logic on CPU.  Multi-rank (gloo, two ranks): the step
time is the slowest rank's, the value counts every rank's rows (weak
scaling), and the reference arm runs on rank 0 only.  The traffic lookup:
the captured ratio for the nearest query count, none for a changed source.
The stage rooflines and the choice of the headline stage.  No GPU is
involved."""
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


def test_stage_rooflines_and_the_headline_stage():
    """The bench's per-stage rooflines on a headline-shaped example (64
    requests x 142,000 tokens, 4 queries, K = 2048, 4 layers), with the
    expected figures written out from the definitions: achieved = algorithmic
    bytes (or flops) / stage time, fraction = achieved / peak, share = stage
    time x launches per step / step time; the headline is the largest share,
    and without a host-link peak the copy drops out."""
    import bench
    w = dict(B=64, N=142000, nq=4, K=2048, L=4, P=64, H=128, Hi=64, Di=128)
    misses = 171842.0
    alg = bench.algorithmic(w, misses)
    stage = {"indexer": 0.44, "topk": 0.085, "resolve_plan": 0.045, "miss_copy": 2.8,
             "attention": 0.337, "miss_copy_in_step": 2.39, "miss_copy_in_step_bytes": 450e6}
    peaks = {"hbm": 6784.2, "bf16": 1895.9, "src": "measured"}
    link = {"peak_gbs": 211.0, "source": "memcpy"}
    head, every = bench.roofline(stage, alg, peaks, w, 3.26, link)

    idx_bytes = 64 * 142000 * (128 + 4) + 64 * 4 * 64 * (128 + 4)
    assert every["indexer"]["bound"] == "hbm"
    assert every["indexer"]["achieved"] == pytest.approx(idx_bytes / 0.44e-3 / 1e9)
    assert every["indexer"]["frac"] == pytest.approx(idx_bytes / 0.44e-3 / 1e9 / 6784.2)
    assert every["topk"]["kernel"] == "topk_filter_kernel"  # 256 rows x 9 CTAs: more than a wave
    assert every["topk"]["achieved"] == pytest.approx(
        (64 * 4 * 142000 * 4 + 64 * 4 * 2048 * 4) / 0.085e-3 / 1e9)

    flops = 2 * 64 * 4 * 2048 * 128 * (576 + 512)
    att = every["attention"]
    assert att["kernel"] == "attn_pair_kernel" and att["bound"] == "tensor"
    assert att["achieved"] == pytest.approx(flops / 0.337e-3 / 1e12)
    assert att["frac"] == pytest.approx(flops / 0.337e-3 / 1e12 / 1895.9)
    assert att["share_of_step"] == pytest.approx(0.337 * 4 / 3.26)

    cp = every["miss_copy"]
    assert cp["bound"] == "host_link" and cp["timed"].startswith("in the step")
    assert cp["achieved"] == pytest.approx(450e6 / 2.39e-3 / 1e9)
    assert cp["frac"] == pytest.approx(450e6 / 2.39e-3 / 1e9 / 211.0)
    assert cp["share_of_step"] == pytest.approx(2.39 / 3.26)
    assert cp["us_per_launch"] == pytest.approx(2390.0 / 4)
    assert head is cp  # the largest share

    head, every = bench.roofline(stage, alg, peaks, w, 3.26, None)
    assert "miss_copy" not in every and head is every["attention"]
