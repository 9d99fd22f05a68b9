"""GPU parity at the workloads' full sizes.

Indices, row locations, residency state and copied rows are compared with the
oracle exactly (every step where the oracle can follow, sampled requests where
it cannot); attention is compared on sampled (request, query, layer) triples
within |gpu - ref| <= 2e-3 + 1e-2 |ref|.

  * full residency, 32 requests x 65,536 tokens, K = 2048, 64x128 E4M3
    indexer, 128 heads, 4 layers (the benchmark's workload and launch
    configuration);
  * mixed residency with MTP3: 64 requests x 142,000 tokens, tail 4096, hot
    buffer 5 x 2048, drawn recency/Zipf streams, all 220 decode steps;
  * zero residency: 4 requests x 2^20 tokens, all rows in pinned host memory,
    hot buffers 2 x 2048 filled on demand, drawn uniform/Zipf streams, 64 steps;
  * agentic growth: 16 requests, 13 turns (a 74,160-token prompt, then 753
    prompt tokens per turn), 220 decode steps per turn with the real indexer
    top-K and one appended token per step, GPU pool capped at 20,000 blocks so
    that requests flip from full to mixed residency mid-trace.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mla_kv_fp8_gb300 import workload as wl

pytestmark = pytest.mark.gpu

TAU = 1.0 / math.sqrt(576)
ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module")
def hs():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_mla_kv_fp8_gb300 import hs as mod
    return mod


def _check_attention(rows_truth, qm, out, lse, idx, b, j, l, fmt=oracle.ROW_E4M3_656):
    sel = idx[idx >= 0]
    rr = rows_truth[torch.from_numpy(sel).long().to(rows_truth.device), l].cpu().numpy()
    qb = qm[l, b, j].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    o, ls = oracle.attention(fmt, qb, rr, TAU)
    g = out[l, b, j].float().cpu().numpy()
    err = np.abs(g - o)
    assert (err <= ATOL + RTOL * np.abs(o)).all(), f"attention b{b} j{j} l{l}: max err {err.max():.3g}"
    gl = lse[l, b, j].cpu().numpy()
    assert (np.abs(gl - ls) <= ATOL + RTOL * np.abs(ls)).all()


def test_full_residency_32x65536_benchmark_config(hs):
    import bench
    from fullsize import locate
    w = dict(bench.WORKLOAD)
    dev = torch.device("cuda")
    pool = bench.setup_pool(w, dev)
    B, N, K, L, H, nq, P = w["B"], w["N"], w["K"], w["L"], w["H"], w["nq"], w["P"]
    try:
        q, wt, qm = bench.step_inputs(w, 1, dev)
        out = torch.empty((L, B, nq, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((L, B, nq, H), dtype=torch.float32, device=dev)
        topk = torch.empty((B, nq, K), dtype=torch.int32, device=dev)
        rid = torch.empty_like(topk)
        pool.step(B, nq, q, wt, qm, TAU, out, topk, rid, lse)
        torch.cuda.synchronize()
        assert pool.get_error() == hs.HS_OK
        tk = topk.cpu().numpy()
        # every list: K distinct ascending visible tokens; every row id reads its token in place
        assert (np.diff(tk, axis=-1) > 0).all() and (tk >= 0).all() and (tk < N).all()
        rv = rid.cpu().numpy()
        for b in range(B):
            st = pool.dump_state(b)
            kind, val = locate(rv[b], st["block_table"], st["hot_blocks"], P, pool.cfg.gpu_blocks)
            assert (kind == 1).all() and (val == tk[b]).all()
        # sampled requests: exact top-K against the oracle, attention on every layer
        for b in (0, 17, 31):
            keys = wl.idx_keys(w["seed"], b, 0, N, w["Di"], wl.IDX_E4M3, device=dev).cpu().numpy()
            s = oracle.indexer_scores(oracle.IDX_E4M3, q[b].cpu().numpy(), wt[b].cpu().numpy(),
                                      keys, np.ones(N, np.float32), N)
            ref = oracle.topk(s[0], N, K)
            np.testing.assert_array_equal(tk[b, 0], ref)
            rows = wl.mla_rows(w["seed"], b, 0, N, L, wl.ROW_E4M3_656, device=dev)
            prow = pool.rows_view()
            ids = rid[b, 0].long()
            assert torch.equal(prow[ids // P, :, ids % P], rows[topk[b, 0].long()])
            for l in range(L):
                _check_attention(rows, qm, out, lse, tk[b, 0], b, 0, l)
            del rows
    finally:
        pool.close()


def _setup_host_pool(hs, seed, B, N, K, L, P, T, num_spec, mode, dev):
    """Pool with host copies of every page; truth rows kept on the device."""
    nq = num_spec + 1
    C = (num_spec + 2) * K
    pages = (N + P - 1) // P
    tail_pages = 0 if mode == hs.HS_ZERO else (T + P - 1) // P + 1
    cfg = hs.make_config(max_requests=B, max_tokens=pages * P, page_tokens=P, top_k=K,
                         num_spec=num_spec, tail_tokens=T, num_mla_layers=L, mla_heads=128,
                         idx_heads=64, idx_dim=128, row_fmt=hs.HS_ROW_E4M3_656,
                         idx_fmt=hs.HS_IDX_E4M3, gpu_blocks=B * (tail_pages + C // P) + 8,
                         host_blocks=B * pages)
    pool = hs.Pool(cfg, device=dev)
    truth = []
    for b in range(B):
        pool.open(b, mode)
        r = wl.mla_rows(seed, b, 0, N, L, wl.ROW_E4M3_656, device=dev)
        k = torch.zeros((N, 128), dtype=torch.uint8, device=dev)  # the indexer is not run here
        pool.append(b, r, k)
        truth.append(r)
    torch.cuda.synchronize()
    return pool, truth


def _run_drawn_trace(hs, pool, truth, streams, N, K, L, P, T, mode, nq, check_state_steps,
                     check_attn, seed, rows_every=16):
    from fullsize import locate
    dev = truth[0].device
    B = streams.shape[1]
    C = pool.C
    hot = [oracle.HotState(C, pool.cfg.max_tokens) for _ in range(B)]
    resident = oracle.page_resident(mode, N, T, P)
    tables = [pool.dump_state(b) for b in range(B)]
    for b in range(B):  # residency the oracle expects
        npg = (N + P - 1) // P
        np.testing.assert_array_equal(tables[b]["block_table"][:npg] >= 0, resident[:npg].astype(bool))
    topk = torch.empty((B, nq, K), dtype=torch.int32, device=dev)
    rid = torch.empty_like(topk)
    out = torch.empty((L, B, nq, 128, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((L, B, nq, 128), dtype=torch.float32, device=dev)
    totals = dict(resident=0, hits=0, misses=0)
    pool.reset_stats()
    for si in range(streams.shape[0]):
        s = si + 1
        idx = streams[si]
        topk.copy_(torch.from_numpy(idx))
        qm = wl.mla_query(seed, s, B, nq, 128, L, dev).contiguous()
        pool.resolve(topk, B, nq, rid)
        for l in range(L):
            pool.sparse_mla_decode(l, qm[l], rid, B, nq, TAU, out[l], lse[l])
        torch.cuda.synchronize()
        assert pool.get_error() == hs.HS_OK, f"step {s}"
        rv = rid.cpu().numpy()
        for b in range(B):
            r = hot[b].resolve(resident, P, N, idx[b])
            assert r["status"] == 0
            for key in totals:
                totals[key] += r[key]
            kind, val = locate(rv[b], tables[b]["block_table"], tables[b]["hot_blocks"], P,
                               pool.cfg.gpu_blocks)
            np.testing.assert_array_equal(kind, r["loc_kind"], err_msg=f"step {s} req {b}")
            np.testing.assert_array_equal(val, r["loc_val"], err_msg=f"step {s} req {b}")
        if s in check_state_steps:
            for b in range(B):
                st = pool.dump_state(b)
                np.testing.assert_array_equal(st["slot_token"], hot[b].slot_token)
                np.testing.assert_array_equal(st["stamp"], hot[b].stamp)
                np.testing.assert_array_equal(st["hot_map"], hot[b].hot_map)
                assert int(st["step"][0]) == int(hot[b].step[0])
        if s % rows_every == 1 or s == streams.shape[0]:
            # every selected row of every request holds its token's bytes, all layers
            prow = pool.rows_view()
            for b in range(B):
                sel = topk[b].reshape(-1)
                ok = sel >= 0
                ids = rid[b].reshape(-1)[ok].long()
                assert torch.equal(prow[ids // P, :, ids % P], truth[b][sel[ok].long()]), f"rows step {s} req {b}"
        for (cs, b, j, l) in check_attn:
            if cs == s:
                _check_attention(truth[b], qm, out, lse, idx[b, j], b, j, l)
    st = pool.stats()
    assert (st["resident"], st["hits"], st["misses"]) == (totals["resident"], totals["hits"], totals["misses"])
    assert st["bytes_copied"] == totals["misses"] * L * 656
    return totals


def test_mixed_mtp3_64x142000_220_steps(hs):
    from fullsize import drawn_streams
    B, N, K, L, P, T, ns, seed, steps = 64, 142000, 2048, 4, 64, 4096, 3, 0, 220
    nq = ns + 1
    streams = drawn_streams(seed, B, range(1, steps + 1), nq, N, K, P, "recency_zipf", T)
    dev = torch.device("cuda")
    pool, truth = _setup_host_pool(hs, seed, B, N, K, L, P, T, ns, hs.HS_MIXED, dev)
    try:
        totals = _run_drawn_trace(hs, pool, truth, streams, N, K, L, P, T, hs.HS_MIXED, nq,
                                  check_state_steps={1, 21, 220},
                                  check_attn=[(1, 0, 0, 0), (21, 5, 3, 2), (220, 63, 1, 3)],
                                  seed=seed)
        assert totals["hits"] > 0 and totals["misses"] > 0 and totals["resident"] > 0
    finally:
        pool.close()


def test_zero_residency_4x1M_64_steps(hs):
    from fullsize import drawn_streams
    B, N, K, L, P, seed, steps = 4, 1 << 20, 2048, 4, 64, 0, 64
    streams = drawn_streams(seed, B, range(1, steps + 1), 1, N, K, P, "uniform_zipf", 0)
    dev = torch.device("cuda")
    pool, truth = _setup_host_pool(hs, seed, B, N, K, L, P, 0, 0, hs.HS_ZERO, dev)
    try:
        totals = _run_drawn_trace(hs, pool, truth, streams, N, K, L, P, 0, hs.HS_ZERO, 1,
                                  check_state_steps={1, 64},
                                  check_attn=[(1, 0, 0, 0), (64, 3, 0, 3)], seed=seed,
                                  rows_every=8)
        assert totals["resident"] == 0 and totals["misses"] >= 4 * K
    finally:
        pool.close()


def test_agentic_growth_16x13_turns(hs):
    """The agentic growth trace at full size.  Every append goes through the
    library's pressure policy (hs_append_pressure), whose flips must be the
    oracle's reading of it (oracle.PressurePolicy: when an append does not
    fit, the full-residency request with the most pages flips first); after
    every round of appends the completed pages are pre-copied to the host on
    a side stream (hs_precopy).  Every step: no device error and every
    selected row id of every request reads its own token's bytes (all
    layers, every 8th step; the first and last step of each turn always).
    Two requests (the first to flip and one that flips last or never) are
    followed by the oracle on every step: exact row locations and hot-buffer
    state, and at each turn's first and last step the exact top-K and
    sampled attention.  At the end two requests finish (closed) and
    hs_pool_relieve returns the flipped requests as the reading says; their
    pages are back on the GPU, byte for byte, and one more step over the
    remaining requests matches the oracle."""
    from fullsize import locate
    B, K, L, P, T, H, Hi, Di, seed = 16, 2048, 4, 64, 4096, 128, 64, 128, 0
    prompt0, prompt, decode, turns = 74160, 753, 220, 13
    final = prompt0 + decode + (turns - 1) * (prompt + decode)
    assert final == 86056
    max_tokens = (final + P - 1) // P * P
    pages = max_tokens // P
    dev = torch.device("cuda")
    cfg = hs.make_config(max_requests=B, max_tokens=max_tokens, page_tokens=P, top_k=K, num_spec=0,
                         tail_tokens=T, num_mla_layers=L, mla_heads=H, idx_heads=Hi, idx_dim=Di,
                         row_fmt=hs.HS_ROW_E4M3_656, idx_fmt=hs.HS_IDX_E4M3,
                         gpu_blocks=20000, host_blocks=B * pages)
    pool = hs.Pool(cfg, device=dev)
    C = pool.C
    N = [0] * B
    modes = [hs.HS_FULL] * B
    truth = [wl.mla_rows(seed, b, 0, final, L, wl.ROW_E4M3_656, device=dev) for b in range(B)]
    keys = [wl.idx_keys(seed, b, 0, final, Di, wl.IDX_E4M3, device=dev) for b in range(B)]
    follow = {}   # request -> oracle HotState (from its flip on)
    flips = []
    pol = oracle.PressurePolicy(cap=20000, T=T, P=P, hot_pages=C // P)
    side = torch.cuda.Stream()

    def append(b, n):
        want, status = pol.append(b, n)
        assert status == oracle.OK
        got = pool.append_pressure(b, truth[b][N[b]:N[b] + n], keys[b][N[b]:N[b] + n])
        assert got == want, (b, N[b], got, want)
        for x in got:
            modes[x] = hs.HS_MIXED
            flips.append(x)
            if len(flips) == 1:
                follow[x] = oracle.HotState(C, max_tokens)
        N[b] += n

    for b in range(B):
        pool.open(b, hs.HS_FULL)
        pol.open(b)
        append(b, prompt0)
    assert pool.precopy(side) == B * (prompt0 // P)
    torch.cuda.synchronize()
    last = B - 1  # followed from the start; flips (if at all) late, being the highest id
    follow[last] = None
    topk = torch.empty((B, 1, K), dtype=torch.int32, device=dev)
    rid = torch.empty_like(topk)
    out = torch.empty((L, B, 1, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((L, B, 1, H), dtype=torch.float32, device=dev)
    tau = 1.0 / math.sqrt(576)
    step = 0
    checked_topk = 0
    for turn in range(turns):
        if turn:
            for b in range(B):
                append(b, prompt)
            pool.precopy(side)
        for d in range(decode):
            step += 1
            edge = d == 0 or d == decode - 1
            q = torch.stack([wl.idx_query(seed, b, step, 1, Hi, Di, wl.IDX_E4M3, dev) for b in range(B)])
            w = torch.stack([wl.idx_weights(seed, b, step, 1, Hi, dev) for b in range(B)])
            qm = wl.mla_query(seed, step, B, 1, H, L, dev).contiguous()
            pool.step(B, 1, q.contiguous(), w.contiguous(), qm, tau, out, topk, rid, lse)
            torch.cuda.synchronize()
            assert pool.get_error() == hs.HS_OK, f"turn {turn} step {d}"
            tk = topk.cpu().numpy()
            rv = rid.cpu().numpy()
            if edge or step % 8 == 0:
                prow = pool.rows_view()
                for b in range(B):
                    sel = topk[b, 0]
                    ok = sel >= 0
                    ids = rid[b, 0][ok].long()
                    assert torch.equal(prow[ids // P, :, ids % P], truth[b][sel[ok].long()]), \
                        f"rows turn {turn} step {d} req {b}"
            for b in list(follow):
                if follow[b] is None and modes[b] == hs.HS_MIXED:  # flipped before this step
                    follow[b] = oracle.HotState(C, max_tokens)
                hot = follow[b]
                st = pool.dump_state(b)
                resident = oracle.page_resident(modes[b], N[b], T, P)
                if hot is None:  # still full: every selected token is read in place
                    kind, val = locate(rv[b], st["block_table"], st["hot_blocks"], P, 20000)
                    sel = tk[b] >= 0
                    assert (kind[sel] == 1).all() and (val[sel] == tk[b][sel]).all()
                    continue
                r = hot.resolve(resident, P, N[b], tk[b])
                assert r["status"] == 0
                kind, val = locate(rv[b], st["block_table"], st["hot_blocks"], P, 20000)
                np.testing.assert_array_equal(kind, r["loc_kind"], err_msg=f"turn {turn} step {d} req {b}")
                np.testing.assert_array_equal(val, r["loc_val"], err_msg=f"turn {turn} step {d} req {b}")
                np.testing.assert_array_equal(st["stamp"], hot.stamp)
                np.testing.assert_array_equal(st["slot_token"], hot.slot_token)
            if edge:
                for b in sorted(follow):
                    kb = keys[b][:N[b]].cpu().numpy()
                    sc = oracle.indexer_scores(oracle.IDX_E4M3, q[b].cpu().numpy(), w[b].cpu().numpy(),
                                               kb, np.ones(N[b], np.float32), N[b])
                    np.testing.assert_array_equal(tk[b, 0], oracle.topk(sc[0], N[b], K))
                    checked_topk += 1
                    l = (turn + d) % L
                    _check_attention(truth[b], qm, out, lse, tk[b, 0], b, 0, l)
            for b in range(B):
                append(b, 1)  # the decoded token joins the tail
            pool.precopy(side)
    torch.cuda.synchronize()
    assert N == [final] * B
    assert flips and flips[0] == 0, flips  # every request is the same size: lowest id first
    assert hs.HS_FULL in modes              # only as many flips as the cap needs
    assert checked_topk >= 2 * turns
    # two conversations end; the flipped requests come back as blocks free up
    back = []
    for x in (B - 1, B - 2):
        assert modes[x] == hs.HS_FULL
        pool.close_request(x)
        pol.close(x)
        want = pol.relieve()
        got = pool.relieve()
        assert got == want, (x, got, want)
        back += got
    assert sorted(back) == sorted(flips), (back, flips)
    prow = pool.rows_view()
    for x in back:
        st = pool.dump_state(x)
        bt = st["block_table"][:pages]
        assert (bt >= 0).all() and (st["hot_blocks"] < 0).all()
        tok = torch.arange(final, device=dev)
        blk = torch.from_numpy(bt.astype(np.int64)).to(dev)[tok // P]
        assert torch.equal(prow[blk, :, tok % P], truth[x]), f"request {x} after its return"
    B2 = B - 2
    step += 1
    q = torch.stack([wl.idx_query(seed, b, step, 1, Hi, Di, wl.IDX_E4M3, dev) for b in range(B2)])
    w = torch.stack([wl.idx_weights(seed, b, step, 1, Hi, dev) for b in range(B2)])
    qm = wl.mla_query(seed, step, B2, 1, H, L, dev).contiguous()
    out2, lse2 = out[:, :B2].contiguous(), lse[:, :B2].contiguous()
    topk2, rid2 = topk[:B2].contiguous(), rid[:B2].contiguous()
    pool.step(B2, 1, q.contiguous(), w.contiguous(), qm, tau, out2, topk2, rid2, lse2)
    torch.cuda.synchronize()
    assert pool.get_error() == hs.HS_OK
    for x in back:
        kb = keys[x].cpu().numpy()
        sc = oracle.indexer_scores(oracle.IDX_E4M3, q[x].cpu().numpy(), w[x].cpu().numpy(), kb,
                                   np.ones(final, np.float32), final)
        np.testing.assert_array_equal(topk2[x, 0].cpu().numpy(), oracle.topk(sc[0], final, K))
        _check_attention(truth[x], qm, out2, lse2, topk2[x, 0].cpu().numpy(), x, 0, step % L)
    pool.close()
