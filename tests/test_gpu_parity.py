"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs (bit-exact indices / state / rows; attention within
2e-3 + 1e-2 |ref|).  Sizes are small enough for the oracle, yet span several
tiles, chunks and pages with ragged tails."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mla_kv_fp8_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _hs():
    from sparse_mla_kv_fp8_gb300 import hs
    return hs


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(case, steps=None):
    from harness import Runner
    r = Runner(case)
    try:
        for _ in range(steps or case.steps):
            r.run_step()
        st = r.pool.stats()
        assert st["resident"] == r.stats["resident"]
        assert st["hits"] == r.stats["hits"]
        assert st["misses"] == r.stats["misses"]
        return r.stats
    finally:
        r.close()


def test_tiny_fp32_mixed_32_steps():
    """1 request, N=4096 (+1 per step), K=256, 4x32 fp32 indexer, 16 heads,
    fp32 rows, tail 512, hot 2K=512, 32 steps."""
    from harness import Case
    hs = _hs()
    c = Case("tiny-fp32", B=1, N=4096, K=256, Hi=4, Di=32, idx_fmt=wl.IDX_F32, H=16,
             row_fmt=wl.ROW_F32_2304, L=1, T=512, mode=hs.HS_MIXED, steps=32, append=1)
    stats = _run(c)
    assert stats["misses"] > 0 and stats["hits"] > 0 and stats["resident"] > 0


def test_tiny_fp8_mixed():
    from harness import Case
    hs = _hs()
    c = Case("tiny-fp8", B=1, N=4096, K=256, Hi=4, Di=32, idx_fmt=wl.IDX_E4M3, H=16,
             row_fmt=wl.ROW_E4M3_656, L=1, T=512, mode=hs.HS_MIXED, steps=8, append=1)
    _run(c)


def test_mtp_drawn_recency_zipf_ragged():
    """MTP3 (4 queries), drawn recency/Zipf streams, ragged lengths, 2 layers."""
    from harness import Case
    hs = _hs()
    c = Case("mtp-drawn", B=3, N=[3000, 2500, 3333], K=128, Hi=8, Di=64, H=32, L=2, T=256,
             num_spec=3, mode=hs.HS_MIXED, steps=12, source="recency_zipf", check_attn_every=4)
    stats = _run(c)
    assert stats["misses"] > 0 and stats["hits"] > 0


def test_mtp_indexer_with_scales_and_appends():
    from harness import Case
    hs = _hs()
    c = Case("mtp-indexer", B=2, N=[900, 1234], K=128, Hi=16, Di=32, H=16, L=1, T=128,
             num_spec=3, mode=hs.HS_MIXED, steps=5, append=4, sigma=True)
    _run(c)


def test_zero_residency_fills_on_demand():
    from harness import Case
    hs = _hs()
    c = Case("zero", B=2, N=5000, K=256, Hi=8, Di=32, H=16, L=2, T=0, mode=hs.HS_ZERO,
             steps=10, source="uniform_zipf", check_attn_every=3)
    stats = _run(c)
    assert stats["resident"] == 0 and stats["misses"] > 0


def test_full_residency_real_head_counts():
    """64x128 E4M3 indexer, 128 MLA heads, ragged lengths, full residency."""
    from harness import Case
    hs = _hs()
    c = Case("full", B=3, N=[2000, 700, 4097], K=256, Hi=64, Di=128, H=128, L=2,
             mode=hs.HS_FULL, steps=2)
    stats = _run(c)
    assert stats["misses"] == 0 and stats["hits"] == 0


@pytest.mark.parametrize("num_spec", [0, 3])
def test_fewer_visible_than_k_pads(num_spec):
    from harness import Case
    hs = _hs()
    c = Case("short", B=2, N=[100, 37], K=256, Hi=8, Di=32, H=16, L=1, T=64,
             num_spec=num_spec, mode=hs.HS_MIXED, steps=3, append=num_spec + 1)
    _run(c)


def test_hs_step_matches_separate_calls():
    from harness import Case
    hs = _hs()
    c = Case("step", B=2, N=[3000, 2100], K=256, Hi=16, Di=64, H=32, L=3, T=256,
             mode=hs.HS_MIXED, steps=4, append=1, use_step=True)
    _run(c)


@pytest.mark.parametrize("B,nq,mode", [(5, 4, 1), (6, 1, 2), (2, 2, 1)])
def test_step_with_given_lists(B, nq, mode):
    """hs_step takes the lists to resolve from topk_in when given, while its
    indexer and top-K still run: every step against the oracle, the step's
    own top-K bit-exact against the oracle's indexer, the resolve, hot-buffer
    state, rows and attention against the drawn lists; MTP and one query,
    mixed and zero residency, with appends between steps."""
    from harness import Case
    hs = _hs()
    c = Case("step-given", B=B, N=[1900 + 211 * i for i in range(B)], K=128, Hi=8, Di=32, H=16,
             L=2, T=128, num_spec=nq - 1, mode=mode, steps=4, source="recency_zipf",
             use_step=True, append=1)
    _run(c)


def test_indexer_scores_bit_exact():
    """hs_indexer_score against the oracle's scores, every visible entry."""
    from harness import Case, Runner
    hs = _hs()
    for case in (Case("s-fp8", B=2, N=[1500, 3001], K=64, Hi=64, Di=128, H=16, num_spec=3,
                      sigma=True, mode=hs.HS_FULL),
                 Case("s-f32", B=1, N=777, K=64, Hi=4, Di=32, idx_fmt=wl.IDX_F32, H=16,
                      mode=hs.HS_FULL)):
        r = Runner(case)
        try:
            q, w, _ = r.step_inputs(1)
            stride = r.max_tokens
            sc = torch.full((case.B, r.nq, stride), float("nan"), device=r.dev)
            r.pool.indexer_score(q, w, case.B, r.nq, sc, stride)
            torch.cuda.synchronize()
            for b in range(case.B):
                N = r.N[b]
                ref = oracle.indexer_scores(case.idx_fmt, q[b].cpu().numpy(), w[b].cpu().numpy(),
                                            r.keys[b].cpu().numpy(), r.sig[b].cpu().numpy(), N)
                got = sc[b, :, :N].cpu().numpy()
                for j in range(r.nq):
                    vis = oracle.visible(N, r.nq, j)
                    np.testing.assert_array_equal(got[j, :vis], ref[j, :vis])
        finally:
            r.close()


@pytest.mark.parametrize("Hi,num_spec", [(64, 0), (64, 1), (64, 2), (32, 3), (96, 1), (128, 0)])
def test_indexer_tensor_core_head_and_query_counts(Hi, num_spec):
    """The tensor-core indexer at every epilogue shape: one to four warp
    groups (one per query), the unrolled 64-head reduction and the general
    one (32, 96 and 128 heads), against the oracle's scores bit for bit."""
    from harness import Case, Runner
    hs = _hs()
    case = Case("s-shapes", B=3, N=[1000, 2500, 4097], K=64, Hi=Hi, Di=128, H=16,
                num_spec=num_spec, sigma=True, mode=hs.HS_FULL)
    r = Runner(case)
    try:
        q, w, _ = r.step_inputs(1)
        stride = r.max_tokens
        sc = torch.full((case.B, r.nq, stride), float("nan"), device=r.dev)
        r.pool.indexer_score(q, w, case.B, r.nq, sc, stride)
        torch.cuda.synchronize()
        assert r.pool.get_error() == hs.HS_OK
        for b in range(case.B):
            N = r.N[b]
            ref = oracle.indexer_scores(case.idx_fmt, q[b].cpu().numpy(), w[b].cpu().numpy(),
                                        r.keys[b].cpu().numpy(), r.sig[b].cpu().numpy(), N)
            got = sc[b, :, :N].cpu().numpy()
            for j in range(r.nq):
                vis = oracle.visible(N, r.nq, j)
                np.testing.assert_array_equal(got[j, :vis], ref[j, :vis])
    finally:
        r.close()


@pytest.mark.parametrize("K", [512, 2560])
@pytest.mark.parametrize("max_tokens", [0, 200064, 300032])
def test_topk_ties_and_special_scores(max_tokens, K):
    """hs_topk on crafted scores: heavy ties, +0, negatives, all-equal rows.
    K = 512 takes the one-launch cluster kernel at the smallest capacity
    (20,032 tokens: every row's 2-CTA cluster fits one wave) and the
    sampled-threshold path at the others (rows of at most 8,192 visible
    tokens all candidates, longer rows sampled; the all-equal rows overflow
    the candidate list and take the whole-row select).  K = 2560 takes the
    radix paths, picked by the row capacity: one cluster launch with 16
    keys per thread (20,032) or 32 (200,064), and the multi-kernel radix
    select beyond 262,144."""
    from harness import Case, Runner
    hs = _hs()
    case = Case("topk", B=4, N=[20000, 9000, 300, 16385], K=K, Hi=8, Di=32, H=16,
                num_spec=1, mode=hs.HS_FULL, max_tokens=max_tokens)
    r = Runner(case)
    try:
        stride = r.max_tokens
        g = torch.Generator().manual_seed(3)
        sc = torch.randint(0, 40, (case.B, 2, stride), generator=g).float()
        sc[1] = 0.0                                  # every score equal
        sc[2, 0, :150] = -torch.arange(150).float()  # negatives and -0 area
        sc[3, 1] = torch.randn(stride, generator=g)
        # the K-th largest score is a zero and +0 / -0 alternate among the
        # zeros: equal scores, so the lowest tokens of either sign are taken
        z = torch.zeros(stride)
        z[1::2] = -0.0
        z[:300:3] = torch.arange(1, 101).float()   # 100 positives spread out
        z[7000:9000] = -1.0                          # below the zeros
        sc[0, 1] = z
        sc[3, 0] = -1.0
        sc[3, 0, :5000] = torch.where(torch.arange(5000) % 50 == 0, torch.tensor(2.0),
                                      torch.where(torch.arange(5000) % 2 == 0, torch.tensor(-0.0),
                                                  torch.tensor(0.0)))
        assert (torch.signbit(sc[0, 1]) & (sc[0, 1] == 0)).any()
        sc = sc.to(r.dev)
        out = torch.full((case.B, 2, case.K), -9, dtype=torch.int32, device=r.dev)
        r.pool.topk(sc, stride, case.B, 2, out)
        torch.cuda.synchronize()
        s_np = sc.cpu().numpy()
        for b in range(case.B):
            for j in range(2):
                vis = oracle.visible(r.N[b], 2, j)
                ref = oracle.topk(s_np[b, j], vis, case.K)
                np.testing.assert_array_equal(out[b, j].cpu().numpy(), ref)
    finally:
        r.close()


def test_topk_sampled_threshold_edges():
    """The sampled-threshold top-K where its sample misleads it, against the
    oracle.  With 200,064-token rows and K = 512 the threshold step samples
    16,384 scores of a 131,072-token row, as 2,048 runs of 8 tokens
    [64j + 28, 64j + 36), and aims at 2,048 tokens at or above the 256th
    largest sample; a row keeps at most 8,192 candidates.
      row 0: the samples are distinct and above every other score, so only
             256 tokens reach the threshold (fewer than K): whole-row select;
      row 1: every other sample is 1.0 and every other score 0.0, so exactly
             8,192 tokens reach it (the candidate cap, inclusive): the
             candidate path, with the K-th score tied 8,192 ways;
      row 2: as row 1 with one more 1.0 (8,193 tokens, past the cap): the
             whole-row select, with the same ties;
      row 3: 40,000 equal scores, all candidates: past the cap, whole row;
      row 4: 200,000 normal scores: the candidate path over two bitmap
             windows of 131,072 tokens."""
    from harness import Case, Runner
    hs = _hs()
    N = [131072, 131072, 131072, 40000, 200000]
    case = Case("topk", B=5, N=N, K=512, Hi=8, Di=32, H=16, L=1, num_spec=0,
                mode=hs.HS_FULL, max_tokens=200064)
    r = Runner(case)
    try:
        stride = r.max_tokens
        g = torch.Generator().manual_seed(11)
        sc = torch.full((case.B, 1, stride), -7.0)
        samples = (torch.arange(2048) * 64 + 28).repeat_interleave(8) + torch.arange(8).repeat(2048)
        sc[0, 0, :N[0]] = torch.rand(N[0], generator=g)
        sc[0, 0, samples] = 2.0 + torch.randperm(16384, generator=g).float()
        sc[1, 0, :N[1]] = 0.0
        sc[1, 0, samples[::2]] = 1.0
        sc[2, 0, :N[2]] = 0.0
        sc[2, 0, samples[::2]] = 1.0
        sc[2, 0, 1] = 1.0
        sc[3, 0, :N[3]] = -3.5
        sc[4, 0, :N[4]] = torch.randn(N[4], generator=g)
        sc = sc.to(r.dev)
        out = torch.full((case.B, 1, case.K), -9, dtype=torch.int32, device=r.dev)
        r.pool.topk(sc, stride, case.B, 1, out)
        torch.cuda.synchronize()
        s_np = sc.cpu().numpy()
        for b in range(case.B):
            ref = oracle.topk(s_np[b, 0], N[b], case.K)
            np.testing.assert_array_equal(out[b, 0].cpu().numpy(), ref, err_msg=f"row {b}")
        np.testing.assert_array_equal(out[1, 0].cpu().numpy(), samples[::2][:512].numpy())
        np.testing.assert_array_equal(out[3, 0].cpu().numpy(), np.arange(512))
    finally:
        r.close()


def test_residency_independence_bit_identical():
    """Full, mixed and zero residency give bit-identical outputs for the same
    inputs (the row a query reads is the same bytes wherever it lives)."""
    from harness import Case, Runner
    hs = _hs()
    outs = []
    for mode in (hs.HS_FULL, hs.HS_MIXED, hs.HS_ZERO):
        c = Case("res", B=2, N=[2500, 3100], K=256, Hi=8, Di=32, H=32, L=2, T=256, mode=mode,
                 steps=3)
        r = Runner(c)
        try:
            for s in range(1, 4):
                q, w, qm = r.step_inputs(s)
                topk = torch.empty((2, 1, 256), dtype=torch.int32, device=r.dev)
                rid = torch.empty_like(topk)
                out = torch.empty((2, 2, 1, 32, 512), dtype=torch.bfloat16, device=r.dev)
                r.pool.step(2, 1, q, w, qm, r.tau, out, topk, rid)
            torch.cuda.synchronize()
            outs.append(out.cpu())
        finally:
            r.close()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_graph_capture_replay_equals_eager():
    from harness import Case, Runner
    hs = _hs()
    c = Case("graph", B=2, N=[3000, 2000], K=256, Hi=8, Di=32, H=32, L=2, T=256,
             mode=hs.HS_MIXED, steps=6)
    eager, graph = Runner(c), Runner(c)
    try:
        q, w, qm = eager.step_inputs(1)
        shp = (2, 1, 256)
        bufs = {}
        for name, r in (("eager", eager), ("graph", graph)):
            bufs[name] = dict(q=q.clone(), w=w.clone(), qm=qm.clone(),
                              out=torch.zeros((2, 2, 1, 32, 512), dtype=torch.bfloat16, device=r.dev),
                              topk=torch.zeros(shp, dtype=torch.int32, device=r.dev),
                              rid=torch.zeros(shp, dtype=torch.int32, device=r.dev))
        gbuf = bufs["graph"]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                graph.pool.step(2, 1, gbuf["q"], gbuf["w"], gbuf["qm"], graph.tau, gbuf["out"],
                                gbuf["topk"], gbuf["rid"], stream=s)
        torch.cuda.synchronize()
        for step in range(1, 6):
            qs, ws, qms = eager.step_inputs(step)
            e = bufs["eager"]
            e["q"].copy_(qs), e["w"].copy_(ws), e["qm"].copy_(qms)
            gbuf["q"].copy_(qs), gbuf["w"].copy_(ws), gbuf["qm"].copy_(qms)
            eager.pool.step(2, 1, e["q"], e["w"], e["qm"], eager.tau, e["out"], e["topk"], e["rid"])
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(e["topk"], gbuf["topk"])
            assert torch.equal(e["rid"], gbuf["rid"])
            assert torch.equal(e["out"], gbuf["out"])
            for b in range(2):
                se, sg = eager.pool.dump_state(b), graph.pool.dump_state(b)
                for k in ("hot_map", "slot_token", "stamp", "step"):
                    np.testing.assert_array_equal(se[k], sg[k])
        assert graph.pool.get_error() == hs.HS_OK
        st = graph.pool.stats()
        assert st["misses"] > 0
    finally:
        eager.close()
        graph.close()


def _graph_twins(case, between, steps):
    """Capture one hs_step of `case` as a CUDA graph on one pool and replay it
    for `steps` steps beside eager steps of a twin pool, calling
    between(step, runner) on both before each step; outputs and device state
    must match bit for bit.  Returns the graph pool's counters."""
    from harness import Runner
    hs = _hs()
    eager, graph = Runner(case), Runner(case)
    B, K, H, L = case.B, case.K, case.H, case.L
    try:
        q, w, qm = eager.step_inputs(1)
        shp = (B, 1, K)
        bufs = {}
        for name, r in (("eager", eager), ("graph", graph)):
            bufs[name] = dict(q=q.clone(), w=w.clone(), qm=qm.clone(),
                              out=torch.zeros((L, B, 1, H, 512), dtype=torch.bfloat16, device=r.dev),
                              topk=torch.zeros(shp, dtype=torch.int32, device=r.dev),
                              rid=torch.zeros(shp, dtype=torch.int32, device=r.dev))
        gbuf, e = bufs["graph"], bufs["eager"]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                graph.pool.step(B, 1, gbuf["q"], gbuf["w"], gbuf["qm"], graph.tau, gbuf["out"],
                                gbuf["topk"], gbuf["rid"], stream=s)
        torch.cuda.synchronize()
        for step in range(1, steps + 1):
            for r in (eager, graph):
                between(step, r)
            torch.cuda.synchronize()
            qs, ws, qms = eager.step_inputs(step)
            for buf in (e, gbuf):
                buf["q"].copy_(qs), buf["w"].copy_(ws), buf["qm"].copy_(qms)
            eager.pool.step(B, 1, e["q"], e["w"], e["qm"], eager.tau, e["out"], e["topk"], e["rid"])
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(e["topk"], gbuf["topk"]), f"step {step}: top-K"
            assert torch.equal(e["rid"], gbuf["rid"]), f"step {step}: row ids"
            assert torch.equal(e["out"], gbuf["out"]), f"step {step}: attention"
            for b in range(B):
                se, sg = eager.pool.dump_state(b), graph.pool.dump_state(b)
                for k in ("hot_map", "slot_token", "stamp", "step", "block_table", "seq_len"):
                    np.testing.assert_array_equal(se[k], sg[k], err_msg=f"step {step} req {b}: {k}")
        assert eager.pool.get_error() == hs.HS_OK
        assert graph.pool.get_error() == hs.HS_OK
        return graph.pool.stats()
    finally:
        eager.close()
        graph.close()


def test_graph_replay_stays_valid_across_residency_changes():
    """A step captured as a CUDA graph at full residency replays correctly
    after the requests change residency between replays (full -> mixed ->
    zero -> full): every launch of the step depends only on the pool's
    configuration, the residency lives in device tables.  The replays are
    compared bit for bit with eager steps of a twin pool taking the same
    changes (eager residency changes are checked against the oracle in
    test_residency_round_trips_under_the_oracle)."""
    from harness import Case
    hs = _hs()
    c = Case("graph-modes", B=2, N=[3000, 2000], K=256, Hi=8, Di=32, H=32, L=2, T=256,
             mode=hs.HS_FULL, steps=8)
    flips = {3: hs.HS_MIXED, 5: hs.HS_ZERO, 7: hs.HS_FULL}

    def between(step, r):
        if step in flips:
            for b in range(c.B):
                r.pool.set_mode(b, flips[step])

    st = _graph_twins(c, between, 8)
    assert st["misses"] > 0 and st["resident"] > 0


def test_graph_replay_stays_valid_across_appends():
    """A decode loop replays one captured step graph while every request grows
    by 40 tokens between replays (mixed residency: the tail window slides and
    pages leave it for the host pool): lengths, tables and step counters live
    on the device, so the replays match eager steps of a twin pool bit for
    bit (eager appends are checked against the oracle in
    test_mtp_indexer_with_scales_and_appends)."""
    from harness import Case
    hs = _hs()
    c = Case("graph-append", B=2, N=[3000, 2000], K=256, Hi=8, Di=32, H=32, L=2, T=256,
             mode=hs.HS_MIXED, steps=8, append=40)

    def between(step, r):
        if step > 1:
            for b in range(c.B):
                r.append(b, 40)

    st = _graph_twins(c, between, 8)
    assert st["misses"] > 0 and st["resident"] > 0


def test_out_of_range_index_sets_error_and_recovers():
    from harness import Case, Runner
    hs = _hs()
    c = Case("err", B=1, N=1000, K=64, Hi=8, Di=32, H=16, T=128, mode=hs.HS_MIXED)
    r = Runner(c)
    try:
        topk = torch.arange(64, dtype=torch.int32, device=r.dev).view(1, 1, 64) * 10
        topk[0, 0, -1] = 5000  # outside the request
        rid = torch.zeros_like(topk)
        r.pool.resolve(topk, 1, 1, rid)
        assert r.pool.get_error() == hs.HS_ERR_INDEX_RANGE
        assert (rid == -1).all()
        assert r.pool.get_error() == hs.HS_OK  # read-and-clear
        # not ascending
        bad = torch.arange(64, dtype=torch.int32, device=r.dev).flip(0).view(1, 1, 64).contiguous()
        r.pool.resolve(bad, 1, 1, rid)
        assert r.pool.get_error() == hs.HS_ERR_INDEX_RANGE
        # the pool still works afterwards
        r.run_step()
    finally:
        r.close()


def test_bounded_wait_runs_out_and_context_stays_usable():
    """Failure detection without a fault: a wait whose mbarrier nothing
    completes runs out after its limit, HS_ERR_TIMEOUT lands in the sticky
    error word, and the next calls run normally."""
    from harness import Case, Runner
    hs = _hs()
    r = Runner(Case("after-timeout", B=1, N=600, K=64, Hi=4, Di=32, idx_fmt=wl.IDX_F32, H=16,
                    row_fmt=wl.ROW_F32_2304, T=128, steps=1))
    try:
        with pytest.raises(hs.HSError) as ei:
            r.pool.check_wait_timeout(10)  # limit below the accepted range
        assert ei.value.status == hs.HS_ERR_INVALID_ARG
        r.pool.check_wait_timeout(2_000_000)  # about a millisecond
        torch.cuda.synchronize()
        assert r.pool.get_error() == hs.HS_ERR_TIMEOUT
        assert r.pool.get_error() == hs.HS_OK  # read and cleared
        r.run_step()                          # the context is still usable
    finally:
        r.close()


def test_host_side_capacity_errors():
    hs = _hs()
    cfg = hs.make_config(max_requests=2, max_tokens=1024, top_k=64, num_spec=0, tail_tokens=64,
                         num_mla_layers=1, mla_heads=16, idx_heads=4, idx_dim=32,
                         gpu_blocks=6, host_blocks=3)
    pool = hs.Pool(cfg)
    try:
        rows = wl.mla_rows(0, 0, 0, 400, 1, wl.ROW_E4M3_656, device="cuda")
        keys = wl.idx_keys(0, 0, 0, 400, 32, wl.IDX_E4M3, device="cuda")
        pool.open(0, hs.HS_FULL)
        with pytest.raises(hs.HSError) as ei:
            pool.append(0, rows, keys)  # 7 pages > 6 GPU blocks
        assert ei.value.status == hs.HS_ERR_CAPACITY
        pool.open(1, hs.HS_MIXED)       # leases 2 hot blocks
        with pytest.raises(hs.HSError) as ei:
            pool.append(1, rows, keys)  # 7 host pages > 3 host blocks
        assert ei.value.status == hs.HS_ERR_HOST_POOL_FULL
        with pytest.raises(hs.HSError) as ei:
            pool.open(1, hs.HS_MIXED)   # already open
        assert ei.value.status == hs.HS_ERR_INVALID_ARG
        with pytest.raises(hs.HSError) as ei:
            pool.set_mode(0, 7)         # not a residency mode
        assert ei.value.status == hs.HS_ERR_INVALID_ARG
        with pytest.raises(hs.HSError) as ei:
            pool.resolve(torch.zeros((3, 1, 64), dtype=torch.int32, device="cuda"), 3, 1,
                         torch.zeros((3, 1, 64), dtype=torch.int32, device="cuda"))
        assert ei.value.status == hs.HS_ERR_INVALID_ARG  # B beyond max_requests
        # request 0 holds no token (its append was refused): calls that score,
        # select or resolve its tokens are refused before anything is enqueued
        with pytest.raises(hs.HSError) as ei:
            pool.resolve(torch.zeros((1, 1, 64), dtype=torch.int32, device="cuda"), 1, 1,
                         torch.zeros((1, 1, 64), dtype=torch.int32, device="cuda"))
        assert ei.value.status == hs.HS_ERR_INVALID_ARG
        with pytest.raises(hs.HSError) as ei:
            pool.indexer_topk(torch.zeros((1, 1, 4, 32), dtype=torch.uint8, device="cuda"),
                              torch.ones((1, 1, 4), device="cuda"), 1, 1,
                              torch.zeros((1, 1, 64), dtype=torch.int32, device="cuda"))
        assert ei.value.status == hs.HS_ERR_INVALID_ARG
        # q and out are moved in 16-byte vectors: a misaligned pointer is refused
        # before anything is enqueued
        qm = torch.zeros(16 * 576 + 8, dtype=torch.bfloat16, device="cuda")
        rid = torch.full((1, 1, 64), -1, dtype=torch.int32, device="cuda")
        out = torch.zeros(16 * 512 + 8, dtype=torch.bfloat16, device="cuda")
        for qq, oo in ((qm[1:], out[:-8]), (qm[:-8], out[1:])):
            with pytest.raises(hs.HSError) as ei:
                pool.sparse_mla_decode(0, qq, rid, 1, 1, 0.1, oo, None)
            assert ei.value.status == hs.HS_ERR_INVALID_ARG
        pool.sparse_mla_decode(0, qm[:-8], rid, 1, 1, 0.1, out[:-8], None)  # aligned: accepted
        torch.cuda.synchronize()
        assert pool.get_error() == hs.HS_OK
        pool.close_request(1)
        pool.close_request(0)
        assert pool.free_gpu_blocks() == 6
    finally:
        pool.close()


def test_full_to_mixed_flip_keeps_outputs():
    """A request that flips from full to mixed residency between steps keeps
    producing the oracle's results; its freed blocks return to the pool."""
    from harness import Case, Runner
    hs = _hs()
    c = Case("flip", B=2, N=[2600, 1900], K=128, Hi=8, Di=32, H=16, L=2, T=256, mode=hs.HS_FULL,
             steps=6, append=1)
    r = Runner(c)
    try:
        r.run_step()
        r.run_step()
        free0 = r.pool.free_gpu_blocks()
        r.flip_to_mixed(0)
        assert r.pool.free_gpu_blocks() > free0
        for _ in range(4):
            r.run_step()
    finally:
        r.close()


def test_agentic_growth_flips_under_pool_cap():
    """The agentic growth trace at reduced size: every request starts with a
    long prompt, then each turn appends a prompt and decodes token by token
    with the real indexer top-K.  Appends go through the library's pressure
    policy (hs_append_pressure) into a GPU pool capped so that requests flip
    from full to mixed residency mid-trace; completed pages are pre-copied to
    the host on a side stream after every round of appends, so the flips
    release pages whose host copies came from there.  Then the caller parks
    a request in zero residency and hs_pool_relieve returns the flipped one.
    Flips and returns must be the oracle's reading of the policy; every step
    is compared with the oracle: indices, row locations, hot-buffer state,
    row bytes and attention."""
    from harness import Case, Runner
    hs = _hs()
    r = Runner(Case("agentic", B=4, N=1500, K=256, H=128, L=2, T=256, mode=hs.HS_FULL,
                    max_tokens=1792, gpu_blocks=100, host_blocks=4 * 28 + 4, steps=0))
    pol = oracle.PressurePolicy(cap=100, T=256, P=64, hot_pages=r.C // 64)
    side = torch.cuda.Stream()
    try:
        for b in range(r.c.B):
            pol.open(b)
            assert pol.append(b, 1500) == ([], oracle.OK)
        copied = r.pool.precopy(side)
        assert copied == 4 * (1500 // 64)
        flips = []
        for turn in range(5):
            if turn:
                for b in range(r.c.B):
                    flips += r.append_pressure(b, 60, pol)
                r.pool.precopy(side)
            for _ in range(6):
                r.run_step()
                for b in range(r.c.B):
                    flips += r.append_pressure(b, 1, pol)
                r.pool.precopy(side)
        assert flips == [0]             # the largest, lowest id, and only as many as the cap needs
        assert r.modes.count(hs.HS_FULL) == 3
        st = r.pool.stats()
        assert (st["resident"], st["hits"], st["misses"]) == (
            r.stats["resident"], r.stats["hits"], r.stats["misses"])
        assert r.stats["misses"] > 0
        assert r.relieve(pol) == []     # the pool is still under pressure
        r.set_mode(1, hs.HS_ZERO)       # the caller parks a request: its pages free up
        pol.set_mode(1, oracle.ZERO)
        assert r.relieve(pol) == [0]    # the flipped request comes back
        assert r.pool.free_gpu_blocks() == 100 - pol.used()
        for _ in range(3):
            r.run_step()
            for b in range(r.c.B):
                assert r.append_pressure(b, 1, pol) == []
    finally:
        r.close()


def test_precopy_copies_completed_pages_off_the_append_path():
    """Full residency with a host pool: hs_append writes resident pages to
    the GPU only; hs_precopy enqueues on a side stream the host copy of each
    completed page once (the partial page waits until it completes).  Flips
    right after a pre-copy, which may still be in flight, order themselves
    after it; the steps then read the pre-copied rows from the host pool and
    match the oracle."""
    from harness import Case, Runner
    hs = _hs()
    r = Runner(Case("precopy", B=2, N=[1000, 700], K=128, Hi=8, Di=32, H=16, L=2, T=256,
                    mode=hs.HS_FULL, steps=0, max_tokens=1600))
    side = torch.cuda.Stream()
    P = r.c.P
    try:
        host = r.pool.host_rows_view()          # [host blocks, L, P, R]
        host.fill_(0xAB)                        # nothing written there so far
        r.append(0, 100)
        r.append(1, 30)
        assert r.N == [1100, 730]
        hbt = [r.pool.dump_state(b)["host_block_table"] for b in range(2)]
        for b in range(2):
            for pg in range((r.N[b] + P - 1) // P):
                assert (host[int(hbt[b][pg])] == 0xAB).all(), f"req {b} page {pg} written by append"
        assert r.pool.precopy(side) == 1100 // P + 730 // P
        side.synchronize()
        for b in range(2):
            for pg in range(r.N[b] // P):
                want = r.rows[b][pg * P:(pg + 1) * P].transpose(0, 1).cpu()
                assert torch.equal(host[int(hbt[b][pg])], want), f"req {b} page {pg}"
            assert (host[int(hbt[b][r.N[b] // P])] == 0xAB).all()   # the partial page
        assert r.pool.precopy(side) == 0
        r.append(0, 60)                          # 1160 tokens: page 17 completes
        assert r.pool.precopy(side) == 1
        r.set_mode(0, hs.HS_ZERO)                # straight after the pre-copy
        r.set_mode(1, hs.HS_MIXED)
        for _ in range(3):
            r.run_step()
        assert r.stats["misses"] > 0
    finally:
        r.close()


def test_residency_round_trips_under_the_oracle():
    """Residency changes in every direction between steps (full -> mixed ->
    full, full -> zero -> mixed -> full), with appends in between; every step
    against the oracle (indices, locations, hot-buffer state, row bytes,
    attention), and the GPU pool gets every block back."""
    from harness import Case, Runner
    hs = _hs()
    r = Runner(Case("round-trips", B=2, N=[1500, 900], K=128, Hi=8, Di=32, H=128, L=2, T=256,
                    mode=hs.HS_FULL, append=3, steps=0, max_tokens=1600))
    try:
        free0 = r.pool.free_gpu_blocks()
        plan = [None, (0, hs.HS_MIXED), None, (1, hs.HS_ZERO), None, (0, hs.HS_FULL),
                (1, hs.HS_MIXED), None, (1, hs.HS_FULL), None]
        for item in plan:
            if item is not None:
                r.set_mode(*item)
            r.run_step()
        assert r.modes == [hs.HS_FULL, hs.HS_FULL]
        # back in full residency every page is on the GPU again, no hot buffer held
        pages = sum((n + 63) // 64 for n in r.N)
        assert r.pool.free_gpu_blocks() == free0 - (pages - sum((n + 63) // 64 for n in [1500, 900]))
        assert r.stats["misses"] > 0 and r.stats["hits"] > 0
    finally:
        r.close()


def test_dcp_token_shards_match_the_unsharded_request():
    """Context-parallel decode emulated on one GPU: each of B requests is cut
    into R consecutive token shards held as R pool requests; the indexer and
    top-K run per shard, hs_dcp_topk_merge takes the global top-K over the
    shards' candidates (exactly the oracle's top-K of the whole request) and
    splits it back per shard, each shard resolves and attends over its part,
    and hs_dcp_combine merges the partials by their lse (the oracle's
    attention over the whole top-K, within tolerance)."""
    hs = _hs()
    B, R, K, L, H, P, seed = 2, 3, 256, 1, 128, 64, 5
    lens = [1000, 1024, 980]
    offs = [0, 1000, 2024]
    N = sum(lens)
    dev = torch.device("cuda")
    cfg = hs.make_config(max_requests=R * B, max_tokens=1024, page_tokens=P, top_k=K,
                         num_spec=0, tail_tokens=0, num_mla_layers=L, mla_heads=H, idx_heads=64,
                         idx_dim=128, row_fmt=hs.HS_ROW_E4M3_656, idx_fmt=hs.HS_IDX_E4M3,
                         gpu_blocks=R * B * 16 + 8)
    pool = hs.Pool(cfg, device=dev)
    try:
        truth = [wl.mla_rows(seed, b, 0, N, L, wl.ROW_E4M3_656, device=dev) for b in range(B)]
        keys = [wl.idx_keys(seed, b, 0, N, 128, wl.IDX_E4M3, device=dev) for b in range(B)]
        for r in range(R):
            for b in range(B):
                pool.open(r * B + b, hs.HS_FULL)
                sl = slice(offs[r], offs[r] + lens[r])
                pool.append(r * B + b, truth[b][sl].contiguous(), keys[b][sl].contiguous())
        q = torch.stack([wl.idx_query(seed, b, 1, 1, 64, 128, wl.IDX_E4M3, dev) for b in range(B)])
        w = torch.stack([wl.idx_weights(seed, b, 1, 1, 64, dev) for b in range(B)])
        qm = wl.mla_query(seed, 1, B, 1, H, L, dev)
        stride = 1024
        scores = torch.empty((R * B, 1, stride), dtype=torch.float32, device=dev)
        pool.indexer_score(q.repeat(R, 1, 1, 1).contiguous(), w.repeat(R, 1, 1).contiguous(),
                           R * B, 1, scores, stride)
        local = torch.empty((R * B, 1, K), dtype=torch.int32, device=dev)
        pool.topk(scores, stride, R * B, 1, local)
        topk = torch.full((B, 1, K), -7, dtype=torch.int32, device=dev)
        part = torch.full((R * B, 1, K), -7, dtype=torch.int32, device=dev)
        pool.dcp_topk_merge(scores, stride, local, torch.tensor(offs, dtype=torch.int32, device=dev),
                            R, B, topk, part)
        rid = torch.empty_like(part)
        pool.resolve(part, R * B, 1, rid)
        o_parts = torch.empty((R * B, 1, H, 512), dtype=torch.bfloat16, device=dev)
        lse_parts = torch.empty((R * B, 1, H), dtype=torch.float32, device=dev)
        tau = 1.0 / math.sqrt(576)
        pool.sparse_mla_decode(0, qm[0].repeat(R, 1, 1, 1).contiguous(), rid, R * B, 1, tau,
                               o_parts, lse_parts)
        out = torch.empty((B, 1, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, 1, H), dtype=torch.float32, device=dev)
        hs.dcp_combine(o_parts, lse_parts, R, B, H, out, lse)
        torch.cuda.synchronize()
        assert pool.get_error() == hs.HS_OK
        tk, pt = topk.cpu().numpy(), part.cpu().numpy()
        for b in range(B):
            s_full = oracle.indexer_scores(oracle.IDX_E4M3, q[b].cpu().numpy(), w[b].cpu().numpy(),
                                           keys[b].cpu().numpy(), np.ones(N, np.float32), N)
            ref = oracle.topk(s_full[0], N, K)
            np.testing.assert_array_equal(tk[b, 0], ref)
            for r in range(R):
                mine = ref[(ref >= offs[r]) & (ref < offs[r] + lens[r])] - offs[r]
                want = np.full(K, -1, np.int32)
                want[:len(mine)] = mine
                np.testing.assert_array_equal(pt[r * B + b, 0], want)
            rows = truth[b][torch.from_numpy(ref).long().to(dev), 0].cpu().numpy()
            qb = qm[0, b, 0].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
            o, ls = oracle.attention(oracle.ROW_E4M3_656, qb, rows, tau)
            g = out[b, 0].float().cpu().numpy()
            assert (np.abs(g - o) <= 2e-3 + 1e-2 * np.abs(o)).all(), np.abs(g - o).max()
            gl = lse[b, 0].cpu().numpy()
            assert (np.abs(gl - ls) <= 2e-3 + 1e-2 * np.abs(ls)).all()
    finally:
        pool.close()


def test_dcp_topk_merge_signed_zero_threshold():
    """hs_dcp_topk_merge when the K-th best score is a zero and +0 / -0 are
    mixed across and inside the shards: equal scores, so the merged list is
    the oracle's top-K of the whole row (lower global tokens first)."""
    hs = _hs()
    R, B, K, P = 3, 2, 256, 64
    lens, offs = [500, 640, 450], [0, 500, 1140]
    N = sum(lens)
    dev = torch.device("cuda")
    cfg = hs.make_config(max_requests=R * B, max_tokens=640, page_tokens=P, top_k=K,
                         num_spec=0, tail_tokens=0, num_mla_layers=1, mla_heads=16, idx_heads=8,
                         idx_dim=32, row_fmt=hs.HS_ROW_E4M3_656, idx_fmt=hs.HS_IDX_E4M3,
                         gpu_blocks=R * B * 10 + 4)
    pool = hs.Pool(cfg, device=dev)
    try:
        for r in range(R):
            for b in range(B):
                pool.open(r * B + b, hs.HS_FULL)
                pool.append(r * B + b, wl.mla_rows(0, b, offs[r], lens[r], 1, wl.ROW_E4M3_656, dev),
                            wl.idx_keys(0, b, offs[r], lens[r], 32, wl.IDX_E4M3, dev))
        g = torch.Generator().manual_seed(8)
        whole = torch.zeros((B, N))
        whole[:, ::2] = -0.0
        for b in range(B):
            pos = torch.randperm(N, generator=g)[:90 + 40 * b]
            whole[b, pos] = torch.rand(len(pos), generator=g) + 0.5  # fewer than K positives
            neg = torch.randperm(N, generator=g)[:400]
            whole[b, neg] = -torch.rand(len(neg), generator=g) - 0.5
        stride = 640
        scores = torch.full((R * B, 1, stride), float("nan"))
        for r in range(R):
            for b in range(B):
                scores[r * B + b, 0, :lens[r]] = whole[b, offs[r]:offs[r] + lens[r]]
        scores = scores.to(dev)
        local = torch.empty((R * B, 1, K), dtype=torch.int32, device=dev)
        pool.topk(scores, stride, R * B, 1, local)
        topk = torch.full((B, 1, K), -7, dtype=torch.int32, device=dev)
        part = torch.full((R * B, 1, K), -7, dtype=torch.int32, device=dev)
        pool.dcp_topk_merge(scores, stride, local, torch.tensor(offs, dtype=torch.int32, device=dev),
                            R, B, topk, part)
        torch.cuda.synchronize()
        assert pool.get_error() == hs.HS_OK
        sc = scores.cpu().numpy()
        for r in range(R):
            for b in range(B):
                ref = oracle.topk(sc[r * B + b, 0], lens[r], K)
                np.testing.assert_array_equal(local[r * B + b, 0].cpu().numpy(), ref)
        for b in range(B):
            ref = oracle.topk(whole[b].numpy(), N, K)
            assert (whole[b].numpy()[ref] == 0).any()  # the threshold is a zero
            np.testing.assert_array_equal(topk[b, 0].cpu().numpy(), ref)
    finally:
        pool.close()


def test_hot_buffer_below_nq_k_serves_what_fits():
    """A hot buffer smaller than nq*K (the pages' sizing relaxed): with MTP3
    and 2K slots, zero residency and four disjoint-ish drawn lists per request,
    the first steps find fewer free slots than misses.  Each such step reports
    HS_ERR_CAPACITY, serves the lowest missed tokens that fit, and the
    attention runs over the rows that were read, all exactly as the oracle;
    later steps reuse the slots."""
    from harness import Case, Runner
    hs = _hs()
    r = Runner(Case("short-hot", B=3, N=[3000, 2000, 1200], K=64, Hi=8, Di=32, H=128, L=2,
                    mode=hs.HS_ZERO, num_spec=3, hot_rows=128, source="uniform_zipf",
                    allow_capacity=True, steps=6))
    try:
        for _ in range(6):
            r.run_step()
        assert r.short_steps >= 1
        st = r.pool.stats()
        assert (st["resident"], st["hits"], st["misses"]) == (
            r.stats["resident"], r.stats["hits"], r.stats["misses"])
    finally:
        r.close()


def test_indexer_tensor_core_pipeline_wraps():
    """Enough tiles per CTA that the TMA ring and the two TMEM accumulators
    wrap several times (MTP3: 256 MMA columns, one CTA per SM)."""
    from harness import Case, Runner
    hs = _hs()
    case = Case("s-wrap", B=2, N=[40000, 33333], K=64, Hi=64, Di=128, H=16, num_spec=3,
                sigma=True, mode=hs.HS_FULL)
    r = Runner(case)
    try:
        for s in (1, 2):
            q, w, _ = r.step_inputs(s)
            stride = r.max_tokens
            sc = torch.full((case.B, r.nq, stride), float("nan"), device=r.dev)
            r.pool.indexer_score(q, w, case.B, r.nq, sc, stride)
            torch.cuda.synchronize()
            assert r.pool.get_error() == hs.HS_OK
            for b in range(case.B):
                N = r.N[b]
                ref = oracle.indexer_scores(case.idx_fmt, q[b].cpu().numpy(), w[b].cpu().numpy(),
                                            r.keys[b].cpu().numpy(), r.sig[b].cpu().numpy(), N)
                got = sc[b, :, :N].cpu().numpy()
                for j in range(r.nq):
                    vis = oracle.visible(N, r.nq, j)
                    np.testing.assert_array_equal(got[j, :vis], ref[j, :vis])
    finally:
        r.close()


@pytest.mark.parametrize("name,kw", [
    # split-K over the 2048 rows (few queries), misses from a drawn stream
    ("tc-splits", dict(B=2, N=[5000, 9000], K=2048, Hi=8, Di=32, L=2, T=256, steps=3,
                       source="recency_zipf")),
    # MTP3: four queries per request, ragged lengths
    ("tc-mtp", dict(B=3, N=[2100, 3000, 2600], K=512, Hi=64, Di=128, L=2, T=256, num_spec=3,
                    steps=2)),
    # fewer visible tokens than K: padded entries are skipped
    ("tc-short", dict(B=2, N=[300, 1000], K=512, Hi=8, Di=32, L=1, T=64, steps=2, append=1)),
    # two splits per (query, 64 heads): the pair merges through a 2-CTA cluster
    ("tc-cluster", dict(B=24, N=[2300 + 37 * i for i in range(24)], K=2048, Hi=8, Di=32, L=1,
                        T=256, steps=1, source="recency_zipf")),
    # zero residency, every row arrives through the hot buffer
    ("tc-zero", dict(B=2, N=4000, K=1024, Hi=8, Di=32, L=1, T=0, mode=2, steps=3,
                     source="uniform_zipf")),
    # 64 queries (MTP3 x 16 requests): the latent-split 2-CTA kernel, misses and hits
    ("tc-pair", dict(B=16, N=[1500 + 97 * i for i in range(16)], K=512, Hi=8, Di=32, L=2,
                     T=128, num_spec=3, steps=3, source="recency_zipf", check_attn_every=2)),
])
def test_attention_tensor_core_128_heads(name, kw):
    """128 heads with E4M3 rows: the tcgen05 attention kernel against the oracle."""
    from harness import Case
    hs = _hs()
    kw = dict(kw)
    kw.setdefault("mode", hs.HS_MIXED)
    c = Case(name, H=128, row_fmt=wl.ROW_E4M3_656, **kw)
    _run(c)


def test_resolve_plan_then_miss_copy_equals_resolve():
    """hs_resolve_plan followed by hs_miss_copy (the two halves, here with the
    copy on a second stream ordered by an event) leaves the same row ids,
    hot-buffer state and row bytes as hs_resolve, step after step, against
    the oracle.  Every other step copies layer by layer through
    hs_miss_copy_layers, on a 7-CTA grid for layer 0 and the default one for
    layer 1; empty or out-of-range layer ranges are refused."""
    from harness import Case, Runner
    hs = _hs()
    case = Case("split", B=3, N=[3000, 2500, 4100], K=256, Hi=8, Di=32, H=16, L=2, T=256,
                num_spec=1, mode=hs.HS_MIXED, steps=6, source="recency_zipf")
    a, b = Runner(case), Runner(case)
    try:
        side = torch.cuda.Stream()
        for s in range(1, 7):
            idx = a.drawn(s)
            tk = torch.from_numpy(idx).to(a.dev)
            ra, rb = torch.empty_like(tk), torch.empty_like(tk)
            a.pool.resolve(tk, case.B, 2, ra)
            b.pool.resolve_plan(tk, case.B, 2, rb)
            ev = torch.cuda.Event()
            ev.record()
            side.wait_event(ev)
            if s % 2:
                b.pool.miss_copy(case.B, 2, stream=side)
            else:
                b.pool.miss_copy_layers(case.B, 2, 0, 1, ctas=7, stream=side)
                b.pool.miss_copy_layers(case.B, 2, 1, 2, stream=side)
            torch.cuda.synchronize()
            assert a.pool.get_error() == hs.HS_OK and b.pool.get_error() == hs.HS_OK
            assert torch.equal(ra, rb)
            for r in range(case.B):
                sa, sb = a.pool.dump_state(r), b.pool.dump_state(r)
                for k in ("hot_map", "slot_token", "stamp", "step"):
                    np.testing.assert_array_equal(sa[k], sb[k])
                b._check_rows(r, np.where(idx[r] >= 0, idx[r], -1), rb[r])
        assert a.pool.stats() == b.pool.stats() and b.pool.stats()["misses"] > 0
        for l0, l1, ctas in ((1, 1, 0), (0, 3, 0), (-1, 1, 0), (0, 1, -1)):
            with pytest.raises(hs.HSError):
                b.pool.miss_copy_layers(case.B, 2, l0, l1, ctas=ctas)
    finally:
        a.close()
        b.close()


def test_host_read_probe_copies_pinned_host_memory():
    hs = _hs()
    n = (48 << 20) + 4096
    src = torch.randint(0, 256, (n,), dtype=torch.uint8).pin_memory()
    dst = torch.zeros(n, dtype=torch.uint8, device="cuda")
    hs.host_read_probe(src, dst, n)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src)
    dst.zero_()
    hs.host_read_probe(src, dst, 4096 + 16, ctas=3)
    torch.cuda.synchronize()
    assert torch.equal(dst[:4112].cpu(), src[:4112]) and int(dst[4112:].sum()) == 0


def test_resolve_attend_overlapped_copies_equal_separate_calls():
    """hs_resolve_attend gives bit-identical row ids, state and outputs to
    hs_resolve followed by hs_sparse_mla_decode per layer, eager and replayed
    from a CUDA graph, on a mixed-residency pool with misses every step.  With
    copy timing on (before the capture), every step, eager or replayed,
    leaves one completed span per layer's copy."""
    from harness import Case, Runner
    hs = _hs()
    case = Case("overlap", B=3, N=[3000, 2500, 4100], K=256, Hi=8, Di=32, H=128, L=3, T=256,
                num_spec=1, mode=hs.HS_MIXED, steps=8, source="recency_zipf")
    a, b = Runner(case), Runner(case)
    try:
        B, nq, L, H = case.B, 2, case.L, case.H
        tk = torch.empty((B, nq, case.K), dtype=torch.int32, device=a.dev)
        ra, rb = torch.empty_like(tk), torch.empty_like(tk)
        oa = torch.empty((L, B, nq, H, 512), dtype=torch.bfloat16, device=a.dev)
        ob, la, lb = torch.empty_like(oa), torch.empty((L, B, nq, H), device=a.dev), None
        lb = torch.empty_like(la)
        qm = torch.empty((L, B, nq, H, 576), dtype=torch.bfloat16, device=a.dev)
        st = torch.cuda.Stream()
        graph = None
        b.pool.time_copies(True)
        for s in range(1, 9):
            tk.copy_(torch.from_numpy(a.drawn(s)))
            qm.copy_(a.step_inputs(s)[2])
            a.pool.resolve(tk, B, nq, ra)
            for l in range(L):
                a.pool.sparse_mla_decode(l, qm[l], ra, B, nq, a.tau, oa[l], la[l])
            if s <= 4:
                b.pool.resolve_attend(tk, B, nq, qm, a.tau, ob, rb, lb)
            else:
                if graph is None:
                    torch.cuda.synchronize()
                    graph = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(graph, stream=st):
                        b.pool.resolve_attend(tk, B, nq, qm, a.tau, ob, rb, lb, stream=st)
                graph.replay()
            torch.cuda.synchronize()
            assert a.pool.get_error() == hs.HS_OK and b.pool.get_error() == hs.HS_OK
            assert torch.equal(ra, rb), f"step {s}: row ids"
            assert torch.equal(oa, ob), f"step {s}: outputs"
            assert torch.equal(la, lb), f"step {s}: lse"
            spans = b.pool.copy_times()
            assert len(spans) == L and all(0.0 < t < 1000.0 for t in spans), spans
            for r in range(B):
                sa, sb = a.pool.dump_state(r), b.pool.dump_state(r)
                for k in ("hot_map", "slot_token", "stamp", "step"):
                    np.testing.assert_array_equal(sa[k], sb[k])
        assert a.pool.stats() == b.pool.stats() and b.pool.stats()["misses"] > 0
        # and the outputs of the last step against the oracle
        a._check_attention(qm, ob, lb, a.drawn(8))
    finally:
        a.close()
        b.close()
