"""Seeded synthetic inputs for the sparse-MLA decode step.

This module only draws numbers and encodes them into the storage formats the
library reads; it holds no step of the decode path (no scoring, selection,
residency logic or attention).  Both the CUDA path and the CPU oracle consume
what it produces.

Every draw is keyed by (seed, field, indices...) through numpy's SeedSequence,
so any piece (one request's keys, one step's queries, one drawn top-K list)
is reproducible on its own.  Large tensors are drawn with torch generators on
the requested device (CPU for oracle-sized cases, CUDA for full-size ones).

Value recipes (why they look the way they do):
  * indexer q and keys take values m/8 with integer |m| <= 8.  Every one of
    the 17 values is exact in E4M3 and in fp32, each product is a multiple of
    2^-6 bounded by 1 in magnitude, so the q.k sums of 128 terms are exact in
    any accumulation order; the head weights are 2^-k (k in 0..3), which keeps
    the weighted sum over 64 heads exact in fp32 too.  The fp32 variant uses
    m/8 with |m| <= 64 (values in [-8, 8]).
  * MLA latent values are N(0,1).  In the FP8 row format the 512 nope dims are
    split into four groups of 128, each group scaled by amax/448 and rounded
    to E4M3 (torch's round-to-nearest-even conversion); the 64 rope dims are
    rounded to bf16.  Layout of the 656-byte row: 512 E4M3 codes | 4 fp32
    scales | 64 bf16.
  * decode queries of the MLA layers are N(0,1) rounded to bf16.
"""
from __future__ import annotations

import numpy as np
import torch

LATENT, NOPE, ROPE = 576, 512, 64
ROW_E4M3_656, ROW_F32_2304 = 0, 1
IDX_E4M3, IDX_F32 = 0, 1

_FIELDS = {
    "idx_q": 1, "idx_w": 2, "idx_k": 3, "idx_sigma": 4, "mla_q": 5, "mla_row": 6,
    "draw": 7, "perm": 8,
}


def subseed(seed: int, field: str, *ix: int) -> int:
    """A 63-bit seed derived from (seed, field, indices)."""
    ss = np.random.SeedSequence([int(seed), _FIELDS[field]] + [int(i) for i in ix])
    return int(ss.generate_state(1, np.uint64)[0] & np.uint64(0x7FFFFFFFFFFFFFFF))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def row_bytes(fmt: int) -> int:
    return 656 if fmt == ROW_E4M3_656 else 2304


# --------------------------------------------------------------------------
# indexer inputs
# --------------------------------------------------------------------------
def _small_ints(shape, bound: int, seed: int, device) -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randint(-bound, bound + 1, shape, generator=g, device=device, dtype=torch.int32)


def idx_values(shape, fmt: int, seed: int, device="cpu") -> torch.Tensor:
    """Indexer q or key elements: E4M3 codes (uint8) of m/8, |m| <= 8, or fp32
    m/8 with |m| <= 64."""
    if fmt == IDX_E4M3:
        m = _small_ints(shape, 8, seed, device).to(torch.float32) / 8.0
        return m.to(torch.float8_e4m3fn).view(torch.uint8)
    m = _small_ints(shape, 64, seed, device).to(torch.float32) / 8.0
    return m


def idx_query(seed: int, b: int, step: int, nq: int, Hi: int, Di: int, fmt: int, device="cpu"):
    return idx_values((nq, Hi, Di), fmt, subseed(seed, "idx_q", b, step), device)


def idx_weights(seed: int, b: int, step: int, nq: int, Hi: int, device="cpu") -> torch.Tensor:
    """Head weights 2^-k, k uniform in {0,1,2,3}."""
    g = _gen(subseed(seed, "idx_w", b, step), device)
    k = torch.randint(0, 4, (nq, Hi), generator=g, device=device)
    return torch.pow(2.0, -k.to(torch.float32))


def idx_keys(seed: int, b: int, t0: int, n: int, Di: int, fmt: int, device="cpu"):
    """Keys of tokens [t0, t0+n) of request b (drawn per 4096-token block so
    that any range regenerates identically)."""
    out = []
    blk = 4096
    t = t0
    while t < t0 + n:
        base = (t // blk) * blk
        full = idx_values((blk, Di), fmt, subseed(seed, "idx_k", b, base // blk), device)
        lo, hi = t - base, min(t0 + n - base, blk)
        out.append(full[lo:hi])
        t = base + hi
    if not out:
        return idx_values((0, Di), fmt, 0, device)
    return torch.cat(out, 0)


def idx_sigma(n: int, device="cpu", seed: int | None = None, b: int = 0, t0: int = 0):
    """Per-token key scale.  Ones by default; with a seed, powers of two in
    {1/2, 1, 2} (still exact)."""
    if seed is None:
        return torch.ones(n, dtype=torch.float32, device=device)
    g = _gen(subseed(seed, "idx_sigma", b, t0), device)
    e = torch.randint(-1, 2, (n,), generator=g, device=device)
    return torch.pow(2.0, e.to(torch.float32))


# --------------------------------------------------------------------------
# MLA latent rows and queries
# --------------------------------------------------------------------------
def encode_rows(x: torch.Tensor, fmt: int) -> torch.Tensor:
    """[..., 576] float32 -> [..., R] uint8 stored rows."""
    if fmt == ROW_F32_2304:
        return x.to(torch.float32).contiguous().view(torch.uint8).reshape(*x.shape[:-1], 2304)
    lead = x.shape[:-1]
    nope = x[..., :NOPE].reshape(*lead, 4, 128).to(torch.float32)
    amax = nope.abs().amax(-1, keepdim=True).clamp_min(1e-30)
    scale = amax / 448.0
    codes = (nope / scale).to(torch.float8_e4m3fn).view(torch.uint8).reshape(*lead, NOPE)
    sc = scale.reshape(*lead, 4).contiguous().view(torch.uint8).reshape(*lead, 16)
    rope = x[..., NOPE:].to(torch.bfloat16).contiguous().view(torch.uint8).reshape(*lead, 128)
    return torch.cat([codes, sc, rope], -1).contiguous()


def mla_rows(seed: int, b: int, t0: int, n: int, L: int, fmt: int, device="cpu") -> torch.Tensor:
    """Stored latent rows of tokens [t0, t0+n) of request b, all L layers:
    [n, L, R] uint8 (drawn per 1024-token block for range independence)."""
    blk = 1024
    out = []
    t = t0
    while t < t0 + n:
        base = (t // blk) * blk
        lo, hi = t - base, min(t0 + n - base, blk)
        g = _gen(subseed(seed, "mla_row", b, base // blk), device)
        x = torch.randn((blk, L, LATENT), generator=g, device=device, dtype=torch.float32)
        out.append(encode_rows(x[lo:hi], fmt))
        t = base + hi
    if not out:
        return torch.empty((0, L, row_bytes(fmt)), dtype=torch.uint8, device=device)
    return torch.cat(out, 0)


def mla_query(seed: int, step: int, B: int, nq: int, H: int, L: int, device="cpu") -> torch.Tensor:
    """Decode queries of the L MLA layers: [L, B, nq, H, 576] bf16."""
    g = _gen(subseed(seed, "mla_q", step), device)
    return torch.randn((L, B, nq, H, LATENT), generator=g, device=device).to(torch.bfloat16)


# --------------------------------------------------------------------------
# drawn top-K streams (stand-ins for the agentic traces, which are not here)
# --------------------------------------------------------------------------
def zipf_cdf(n: int, a: float = 1.1) -> np.ndarray:
    w = np.arange(1, n + 1, dtype=np.float64) ** (-a)
    c = np.cumsum(w)
    return c / c[-1]


def page_perm(seed: int, b: int, npages: int) -> np.ndarray:
    return np.random.default_rng(subseed(seed, "perm", b)).permutation(npages)


def _distinct_fill(chosen: np.ndarray, target: int, draw, rng, cap_iters=1000) -> np.ndarray:
    """Append draws to `chosen` (first occurrences, in draw order, skipping
    tokens already there) until it holds `target` tokens."""
    it = 0
    while chosen.shape[0] < target and it < cap_iters:
        need = target - chosen.shape[0]
        cand = draw(rng, 4 * need + 256)
        cand = cand[~np.isin(cand, chosen)]
        if cand.shape[0]:
            _, first = np.unique(cand, return_index=True)
            cand = cand[np.sort(first)][:need]
            chosen = np.concatenate([chosen, cand.astype(np.int64)])
        it += 1
    return chosen


def drawn_topk(seed: int, b: int, step: int, j: int, vis: int, K: int, P: int,
               kind: str, tail_tokens: int = 0, perm: np.ndarray | None = None,
               cdf: np.ndarray | None = None) -> np.ndarray:
    """K distinct tokens of [0, vis), ascending, -1 padded if vis < K.

    kind "recency_zipf": half the tokens from a page-geometric law,
      p(d) ~ (1 - 1/64)^d over the page distance d from the newest page, half
      from Zipf(1.1) over the pages older than the tail window, ranked by a
      fixed per-request permutation; token uniform inside its page.
    kind "uniform_zipf": half uniform over all pages, half Zipf(1.1) over all
      pages under the per-request permutation.
    The two halves are disjoint: the second half skips tokens already drawn."""
    out = np.full(K, -1, np.int32)
    if vis <= K:
        out[:vis] = np.arange(vis, dtype=np.int32)
        return out
    rng = np.random.default_rng(subseed(seed, "draw", b, step, j))
    npages = (vis + P - 1) // P
    newest = npages - 1
    if kind == "recency_zipf":
        older = max(vis - tail_tokens, 0) // P
    else:
        older = npages
    older = max(older, 1)
    if perm is None:
        perm = page_perm(seed, b, older)
    perm = perm[perm < older] if perm.shape[0] != older else perm
    if cdf is None or cdf.shape[0] != older:
        cdf = zipf_cdf(older)

    def in_page(rng, pages):
        t = pages * P + rng.integers(0, P, pages.shape[0])
        return t[t < vis]

    if kind == "recency_zipf":
        q = 1.0 - 1.0 / 64.0

        def first(rng, n):
            d = rng.geometric(1.0 - q, n) - 1  # support 0,1,2,...
            d = d[d <= newest]
            return in_page(rng, newest - d)
    else:
        def first(rng, n):
            return in_page(rng, rng.integers(0, npages, n))

    def second(rng, n):
        r = np.searchsorted(cdf, rng.random(n), side="right")
        r = np.minimum(r, older - 1)
        return in_page(rng, perm[r])

    chosen = np.zeros(0, np.int64)
    chosen = _distinct_fill(chosen, K // 2, first, rng)
    chosen = _distinct_fill(chosen, K, second, rng)
    if chosen.shape[0] < K:  # tiny contexts: top up uniformly
        chosen = _distinct_fill(chosen, K, lambda r, n: r.integers(0, vis, n), rng)
    out[:] = np.sort(chosen[:K].astype(np.int32))
    return out


def _streams_worker(args):
    seed, b, steps, nq, N, K, P, kind, T = args
    older = (max(N - T, 0) // P) if kind == "recency_zipf" else (N + P - 1) // P
    perm = page_perm(seed, b, max(older, 1))
    cdf = zipf_cdf(perm.shape[0])
    out = np.empty((len(steps), nq, K), np.int32)
    for i, s in enumerate(steps):
        for j in range(nq):
            vis = N - nq + j + 1
            out[i, j] = drawn_topk(seed, b, s, j, vis, K, P, kind, T, perm, cdf)
    return out


def drawn_streams(seed: int, B: int, steps, nq: int, N: int, K: int, P: int, kind: str,
                  T: int = 0, procs: int | None = None) -> np.ndarray:
    """[len(steps)][B][nq][K] drawn top-K lists of B requests of N tokens,
    generated in parallel by spawned worker processes (which never touch
    CUDA, so they may start after the caller's first GPU call)."""
    import multiprocessing as mp
    import os
    steps = list(steps)
    procs = procs or max(1, min(B, len(os.sched_getaffinity(0))))
    args = [(seed, b, steps, nq, N, K, P, kind, T) for b in range(B)]
    if procs == 1:
        per_req = [_streams_worker(a) for a in args]
    else:
        with mp.get_context("spawn").Pool(procs) as pool:
            per_req = pool.map(_streams_worker, args)
    return np.stack(per_req, axis=1)
