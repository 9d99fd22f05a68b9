"""Lockstep runner for the parity tests: the same seeded inputs go to the CUDA
library (through the C ABI binding) and to the CPU oracle; every step's
indices, residency state, copied rows and attention outputs are compared.

Comparison rules: bit-exact for top-K indices, row locations, hot-buffer
state (hot_map, slot_token, stamp, step) and row bytes; attention within
|gpu - ref| <= 2e-3 + 1e-2 |ref| against the fp64 oracle.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

import oracle
from sparse_mla_kv_fp8_gb300 import hs
from sparse_mla_kv_fp8_gb300 import workload as wl

ATOL, RTOL = 2e-3, 1e-2


@dataclasses.dataclass
class Case:
    name: str
    B: int
    N: object               # int or list of ints (tokens per request at start)
    K: int
    Hi: int = 64
    Di: int = 128
    idx_fmt: int = wl.IDX_E4M3
    H: int = 128
    row_fmt: int = wl.ROW_E4M3_656
    L: int = 1
    P: int = 64
    T: int = 0
    mode: int = hs.HS_MIXED
    num_spec: int = 0
    hot_rows: int = 0
    steps: int = 4
    append: int = 0          # tokens appended after each step
    source: str = "indexer"  # or "recency_zipf" / "uniform_zipf"
    seed: int = 0
    sigma: bool = False
    check_attn_every: int = 1
    use_step: bool = False   # call hs_step instead of the separate calls
    gpu_blocks: int = 0      # 0 = enough for the case
    host_blocks: int = 0     # 0 = every page of the case
    max_tokens: int = 0
    allow_capacity: bool = False  # a hot buffer below nq*K may run short: expect HS_ERR_CAPACITY


def _Ns(case):
    return list(case.N) if isinstance(case.N, (list, tuple)) else [case.N] * case.B


class Runner:
    def __init__(self, case: Case, device="cuda"):
        self.c = c = case
        self.dev = torch.device(device)
        self.nq = c.num_spec + 1
        Ns = _Ns(c)
        maxN = max(Ns) + c.steps * c.append
        self.max_tokens = c.max_tokens or ((maxN + c.P - 1) // c.P) * c.P
        pages = sum((n + c.steps * c.append + c.P - 1) // c.P for n in Ns)
        C = c.hot_rows or (c.num_spec + 2) * c.K
        blocks = c.gpu_blocks or (pages + c.B * (C // c.P) + 4)
        host_blocks = c.host_blocks or (pages + 4)  # host copies are always kept
        self.cfg = hs.make_config(max_requests=c.B, max_tokens=self.max_tokens, page_tokens=c.P,
                                  top_k=c.K, num_spec=c.num_spec, tail_tokens=c.T,
                                  num_mla_layers=c.L, mla_heads=c.H, idx_heads=c.Hi, idx_dim=c.Di,
                                  row_fmt=c.row_fmt, idx_fmt=c.idx_fmt, hot_rows=c.hot_rows,
                                  gpu_blocks=blocks, host_blocks=host_blocks)
        self.pool = hs.Pool(self.cfg, device=self.dev)
        self.C = self.pool.C
        self.R = self.pool.R
        self.rows, self.keys, self.sig = [], [], []
        self.N = list(Ns)
        self.hot = [oracle.HotState(self.C, self.max_tokens) for _ in range(c.B)]
        self.modes = [c.mode] * c.B
        for b in range(c.B):
            self.pool.open(b, c.mode)
            r = wl.mla_rows(c.seed, b, 0, Ns[b], c.L, c.row_fmt, device=self.dev)
            k = wl.idx_keys(c.seed, b, 0, Ns[b], c.Di, c.idx_fmt, device=self.dev)
            s = (wl.idx_sigma(Ns[b], self.dev, seed=c.seed, b=b) if c.sigma
                 else wl.idx_sigma(Ns[b], self.dev))
            self.pool.append(b, r, k, s)
            self.rows.append(r)
            self.keys.append(k)
            self.sig.append(s)
        self.step_no = 0
        self.perm = {}
        self.tau = 1.0 / math.sqrt(576)
        self.stats = dict(resident=0, hits=0, misses=0)

    # ---- inputs of one step ----
    def step_inputs(self, s):
        c = self.c
        q = torch.stack([wl.idx_query(c.seed, b, s, self.nq, c.Hi, c.Di, c.idx_fmt, self.dev)
                         for b in range(c.B)]).contiguous()
        w = torch.stack([wl.idx_weights(c.seed, b, s, self.nq, c.Hi, self.dev)
                         for b in range(c.B)]).contiguous()
        qm = wl.mla_query(c.seed, s, c.B, self.nq, c.H, c.L, self.dev).contiguous()
        return q, w, qm

    def drawn(self, s):
        c = self.c
        out = np.empty((c.B, self.nq, c.K), np.int32)
        for b in range(c.B):
            N = self.N[b]
            for j in range(self.nq):
                vis = oracle.visible(N, self.nq, j)
                out[b, j] = wl.drawn_topk(c.seed, b, s, j, vis, c.K, c.P, c.source, c.T)
        return out

    # ---- oracle side ----
    def oracle_topk(self, q, w):
        c = self.c
        qn, wn = q.cpu().numpy(), w.cpu().numpy()
        out = np.empty((c.B, self.nq, c.K), np.int32)
        for b in range(c.B):
            N = self.N[b]
            s = oracle.indexer_scores(c.idx_fmt, qn[b], wn[b], self.keys[b].cpu().numpy(),
                                      self.sig[b].cpu().numpy(), N)
            for j in range(self.nq):
                out[b, j] = oracle.topk(s[j], oracle.visible(N, self.nq, j), c.K)
        return out

    def run_step(self, check_state=True):
        c = self.c
        self.step_no += 1
        s = self.step_no
        q, w, qm = self.step_inputs(s)
        B, nq = c.B, self.nq
        topk = torch.full((B, nq, c.K), -7, dtype=torch.int32, device=self.dev)
        row_id = torch.full((B, nq, c.K), -7, dtype=torch.int32, device=self.dev)
        out = torch.empty((c.L, B, nq, c.H, 512), dtype=torch.bfloat16, device=self.dev)
        lse = torch.empty((c.L, B, nq, c.H), dtype=torch.float32, device=self.dev)
        own_topk = None  # a step fed drawn lists still selects with its own indexer
        if c.source == "indexer":
            ref_idx = self.oracle_topk(q, w)
            if c.use_step:
                self.pool.step(B, nq, q, w, qm, self.tau, out, topk, row_id, lse)
            else:
                self.pool.indexer_topk(q, w, B, nq, topk)
        else:
            ref_idx = self.drawn(s)
            if c.use_step:  # the step's resolve and attention take the drawn lists
                own_topk = self.oracle_topk(q, w)
                tk_in = torch.from_numpy(ref_idx).to(self.dev)
                self.pool.step(B, nq, q, w, qm, self.tau, out, topk, row_id, lse, topk_in=tk_in)
            else:
                topk.copy_(torch.from_numpy(ref_idx).to(self.dev))
        if not c.use_step:
            self.pool.resolve(topk, B, nq, row_id)
            for l in range(c.L):
                self.pool.sparse_mla_decode(l, qm[l], row_id, B, nq, self.tau, out[l], lse[l])
        torch.cuda.synchronize()
        err = self.pool.get_error()
        got_idx = topk.cpu().numpy()
        np.testing.assert_array_equal(got_idx, ref_idx if own_topk is None else own_topk,
                                      err_msg=f"{c.name} step {s}: top-K")
        # oracle resolve
        res = []
        short = False
        for b in range(B):
            resident = oracle.page_resident(self.modes[b], self.N[b], c.T, c.P)
            r = self.hot[b].resolve(resident, c.P, self.N[b], ref_idx[b])
            short |= r["status"] == oracle.ERR_CAPACITY
            assert r["status"] == 0 or (c.allow_capacity and r["status"] == oracle.ERR_CAPACITY)
            res.append(r)
            self.stats["resident"] += r["resident"]
            self.stats["hits"] += r["hits"]
            self.stats["misses"] += r["misses"]
        self.short_steps = getattr(self, "short_steps", 0) + int(short)
        want = hs.HS_ERR_CAPACITY if short else hs.HS_OK
        assert err == want, f"{c.name} step {s}: device status {err}, oracle expects {want}"
        served = [r["loc_kind"] != 0 for r in res]  # entries that read a row
        rid = row_id.cpu().numpy()
        for b in range(B):
            st = self.pool.dump_state(b)
            loc_kind, loc_val = self._locate(rid[b], st)
            np.testing.assert_array_equal(loc_kind, res[b]["loc_kind"],
                                          err_msg=f"{c.name} step {s} req {b}: location kind")
            np.testing.assert_array_equal(loc_val, res[b]["loc_val"],
                                          err_msg=f"{c.name} step {s} req {b}: location")
            if check_state:
                h = self.hot[b]
                np.testing.assert_array_equal(st["slot_token"], h.slot_token)
                np.testing.assert_array_equal(st["stamp"], h.stamp)
                np.testing.assert_array_equal(st["hot_map"], h.hot_map)
                assert int(st["step"][0]) == int(h.step[0])
                resident = oracle.page_resident(self.modes[b], self.N[b], c.T, c.P)
                npg = (self.N[b] + c.P - 1) // c.P
                np.testing.assert_array_equal(st["block_table"][:npg] >= 0, resident[:npg].astype(bool))
            # every resolved row holds the bytes of its token, for every layer
            self._check_rows(b, np.where(served[b], ref_idx[b], -1), row_id[b])
        # attention over the rows each query actually read
        if s % c.check_attn_every == 0 or s == 1:
            self._check_attention(qm, out, lse, np.stack([np.where(served[b], ref_idx[b], -1)
                                                          for b in range(B)]))
        # append
        if c.append:
            for b in range(B):
                self.append(b, c.append)
        return res

    def append(self, b, n, on_capacity=None):
        """Append the next n tokens of request b (rows, keys, scales from the
        generators) to the pool and to the oracle's copy.  When the pool is
        full, on_capacity(b) may make room (it returns False to give up)."""
        c = self.c
        n0 = self.N[b]
        r = wl.mla_rows(c.seed, b, n0, n, c.L, c.row_fmt, device=self.dev)
        k = wl.idx_keys(c.seed, b, n0, n, c.Di, c.idx_fmt, device=self.dev)
        sg = (wl.idx_sigma(n, self.dev, seed=c.seed, b=b, t0=n0) if c.sigma
              else wl.idx_sigma(n, self.dev))
        while True:
            try:
                self.pool.append(b, r, k, sg)
                break
            except hs.HSError as e:
                if e.status != hs.HS_ERR_CAPACITY or on_capacity is None or not on_capacity(b):
                    raise
        self.rows[b] = torch.cat([self.rows[b], r])
        self.keys[b] = torch.cat([self.keys[b], k])
        self.sig[b] = torch.cat([self.sig[b], sg])
        self.N[b] += n

    def append_pressure(self, b, n, policy):
        """Append the next n tokens of request b through the library's
        pressure policy.  The requests it flips must be the ones the oracle's
        reading (oracle.PressurePolicy) flips; they restart with an empty hot
        buffer on the oracle side too."""
        c = self.c
        n0 = self.N[b]
        r = wl.mla_rows(c.seed, b, n0, n, c.L, c.row_fmt, device=self.dev)
        k = wl.idx_keys(c.seed, b, n0, n, c.Di, c.idx_fmt, device=self.dev)
        sg = (wl.idx_sigma(n, self.dev, seed=c.seed, b=b, t0=n0) if c.sigma
              else wl.idx_sigma(n, self.dev))
        want, status = policy.append(b, n)
        assert status == oracle.OK
        got = self.pool.append_pressure(b, r, k, sg)
        assert got == want, f"{c.name}: flips {got}, the policy's reading gives {want}"
        for x in got:
            self.modes[x] = hs.HS_MIXED
            self.hot[x] = oracle.HotState(self.C, self.max_tokens)
        self.rows[b] = torch.cat([self.rows[b], r])
        self.keys[b] = torch.cat([self.keys[b], k])
        self.sig[b] = torch.cat([self.sig[b], sg])
        self.N[b] += n
        return got

    def relieve(self, policy):
        """The library's return of flipped requests, checked against the
        oracle's reading; returned requests read every page in place."""
        want = policy.relieve()
        got = self.pool.relieve()
        assert got == want, f"{self.c.name}: returned {got}, the policy's reading gives {want}"
        for x in got:
            self.modes[x] = hs.HS_FULL
            self.hot[x] = oracle.HotState(self.C, self.max_tokens)
        return got

    def _locate(self, rid, st):
        """Pool row ids -> (kind, value) with the request's own tables:
        1 = resident token, 2 = hot slot, 0 = padding."""
        P = self.c.P
        bt, hb = st["block_table"], st["hot_blocks"]
        page_of = {int(blk): p for p, blk in enumerate(bt) if blk >= 0}
        hot_of = {int(blk): i for i, blk in enumerate(hb) if blk >= 0}
        kind = np.zeros(rid.shape, np.int32)
        val = np.full(rid.shape, -1, np.int32)
        for idx in np.ndindex(rid.shape):
            r = int(rid[idx])
            if r < 0:
                continue
            blk, off = divmod(r, P)
            if blk in page_of:
                kind[idx], val[idx] = 1, page_of[blk] * P + off
            elif blk in hot_of:
                kind[idx], val[idx] = 2, hot_of[blk] * P + off
            else:
                kind[idx], val[idx] = 9, r
        return kind, val

    def _check_rows(self, b, idx, rid):
        c = self.c
        sel = torch.from_numpy(idx.reshape(-1)).to(self.dev).long()
        ids = rid.reshape(-1).long()
        ok = sel >= 0
        assert torch.equal(ok, ids >= 0)
        if not ok.any():
            return
        sel, ids = sel[ok], ids[ok]
        pool = self.pool.rows_view()
        got = pool[ids // c.P, :, ids % c.P]          # [n, L, R]
        want = self.rows[b][sel]                        # [n, L, R]
        assert torch.equal(got, want), f"{c.name} step {self.step_no} req {b}: row bytes differ"

    def _check_attention(self, qm, out, lse, idx):
        c = self.c
        for b in range(c.B):
            for j in range(self.nq):
                sel = idx[b, j][idx[b, j] >= 0]
                for l in range(c.L):
                    qb = qm[l, b, j].view(torch.int16).cpu().numpy().view(np.uint16)
                    rows = self.rows[b][torch.from_numpy(sel).to(self.dev).long(), l].cpu().numpy()
                    o, ls = oracle.attention(c.row_fmt, qb, rows, self.tau)
                    g = out[l, b, j].float().cpu().numpy()
                    bad = np.abs(g - o) > ATOL + RTOL * np.abs(o)
                    assert not bad.any(), (f"{c.name} step {self.step_no} b{b} j{j} l{l}: "
                                           f"{bad.sum()} outside tol, max err "
                                           f"{np.abs(g - o).max():.3g}")
                    gl = lse[l, b, j].cpu().numpy()
                    if len(sel):
                        badl = np.abs(gl - ls) > ATOL + RTOL * np.abs(ls)
                        assert not badl.any(), f"{c.name}: lse outside tol"
                    else:
                        assert np.isneginf(gl).all() and (g == 0).all()

    def flip_to_mixed(self, b):
        """Full -> mixed between steps, on both sides: the oracle's hot buffer
        starts empty and the request's residency becomes the tail window."""
        self.set_mode(b, hs.HS_MIXED)

    def set_mode(self, b, mode):
        """Any residency change between steps, on both sides: the resident
        pages follow the new mode and the hot buffer starts empty."""
        self.pool.set_mode(b, mode)
        self.modes[b] = mode
        self.hot[b] = oracle.HotState(self.C, self.max_tokens)

    def close(self):
        self.pool.close()
