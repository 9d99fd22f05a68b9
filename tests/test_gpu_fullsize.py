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
    hot buffers 2 x 2048 filled on demand, drawn uniform/Zipf streams, 64 steps.
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
