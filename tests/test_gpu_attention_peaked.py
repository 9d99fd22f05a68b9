"""GPU parity of the sparse MLA decode on peaked softmaxes.

Queries of some heads are built as multiples of rows that sit late in their
top-K list, so that the running maximum of those heads grows chunk after
chunk (the tensor-core kernel keeps a reference maximum and rescales its
accumulators only when a later chunk raises it by more than 2^8: these
heads force that rescale, several times for some), and one row carries
nearly all of a head's softmax weight.  Other heads keep N(0,1) queries.
Every output is compared with the fp64 oracle within 2e-3 + 1e-2 |ref|.

The shapes pick the kernel routes by themselves: two requests over K = 2048
split every query's rows over many CTAs (partials + combine kernel); 32
queries take two row ranges per query (a 2-CTA cluster that merges in
distributed shared memory); 64 or more queries (x 128-head groups) take the
kernel that splits the latent dims over a 2-CTA cluster (with 80 queries one
range each; 64 queries with K = 704; 256 heads as two head groups); 16 heads
(not a multiple of 64) take the CUDA-core kernel.

Sources: "Un contexte d'un million sur huit H200", « Les trois états de
résidence » (attention reads only the selected rows); "vLLM sert GLM-5.3 en
contexte 1M sur 16 H200", « Comment s'y prendre » (K = 2048 selected tokens).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mla_kv_fp8_gb300 import workload as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _peaked_queries(rng, deq, ent, H, K):
    """[H, 576] float64 queries for one (request, query).  deq[k] is the
    dequantised row of list entry k (576 values), ent the number of valid
    entries.  Heads 8m + i for small i get the patterns below; the rest stay
    N(0,1) (some scaled up)."""
    q = rng.standard_normal((H, 576))
    last = ent - 1
    mid = ent // 2
    for base in range(0, H, 64 if H >= 64 else H):
        pats = {
            # one extreme peak on the very last entry
            0: [(1.0, last)],
            # a maximum that grows three times, chunk after chunk
            1: [(0.2, min(130, last)), (0.35, min(mid + 3, last)), (0.6, last)],
            # moderate peak in the middle
            2: [(0.5, mid)],
            # peak in the first chunk, then nothing larger
            3: [(0.8, 0)],
            # two equal peaks far apart (weight split in half)
            4: [(0.7, min(5, last)), (0.7, last)],
            # strongly disfavoured row: a negative multiple
            5: [(-1.0, mid)],
        }
        for i, pat in pats.items():
            h = base + i
            if h >= H:
                continue
            v = np.zeros(576)
            for a, k in pat:
                v += a * deq[k]
            q[h] = v + 0.05 * rng.standard_normal(576)
        for h in range(base + 6, min(base + 12, H)):
            q[h] *= 3.0  # a wider spread of scores
    return q


def _run(B, nq, H, K, N, seed):
    from sparse_mla_kv_fp8_gb300 import hs
    dev = torch.device("cuda")
    P, L = 64, 1
    pages = (N + P - 1) // P
    cfg = hs.make_config(max_requests=B, max_tokens=pages * P, page_tokens=P, top_k=K,
                         num_spec=nq - 1, tail_tokens=0, num_mla_layers=L, mla_heads=H,
                         idx_heads=8, idx_dim=32, row_fmt=hs.HS_ROW_E4M3_656,
                         idx_fmt=hs.HS_IDX_E4M3, gpu_blocks=B * pages + 4)
    pool = hs.Pool(cfg, device=dev)
    try:
        rows = []
        for b in range(B):
            pool.open(b, hs.HS_FULL)
            r = wl.mla_rows(seed, b, 0, N, L, wl.ROW_E4M3_656, device=dev)
            pool.append(b, r, wl.idx_keys(seed, b, 0, N, 32, wl.IDX_E4M3, device=dev))
            rows.append(r)
        rng = np.random.default_rng(seed)
        topk = np.full((B, nq, K), -1, np.int32)
        for b in range(B):
            for j in range(nq):
                vis = oracle.visible(N, nq, j)
                n = min(K, vis) if (b + j) % 3 else min(K, vis) - 37  # a ragged list now and then
                topk[b, j, :n] = np.sort(rng.choice(vis, n, replace=False))
        tk = torch.from_numpy(topk).to(dev)
        rid = torch.empty_like(tk)
        pool.resolve(tk, B, nq, rid)
        q = np.empty((B, nq, H, 576))
        for b in range(B):
            for j in range(nq):
                sel = topk[b, j][topk[b, j] >= 0]
                deq = oracle.dequant_rows(oracle.ROW_E4M3_656, rows[b][torch.from_numpy(sel).long().to(dev), 0].cpu().numpy())
                q[b, j] = _peaked_queries(rng, deq, len(sel), H, K)
        qb = torch.from_numpy(q).to(torch.float32).to(torch.bfloat16).to(dev).contiguous()
        out = torch.empty((B, nq, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, nq, H), dtype=torch.float32, device=dev)
        tau = 1.0 / math.sqrt(576)
        pool.sparse_mla_decode(0, qb, rid, B, nq, tau, out, lse)
        torch.cuda.synchronize()
        assert pool.get_error() == hs.HS_OK
        checked = 0
        peak_weight = 0.0
        for b in range(B):
            for j in range(nq):
                if B * nq > 8 and (b * nq + j) % 7 not in (0, 3):
                    continue  # a sample of the queries at the larger shapes
                sel = topk[b, j][topk[b, j] >= 0]
                r = rows[b][torch.from_numpy(sel).long().to(dev), 0].cpu().numpy()
                qbits = qb[b, j].view(torch.int16).cpu().numpy().view(np.uint16)
                o, ls = oracle.attention(oracle.ROW_E4M3_656, qbits, r, tau)
                g = out[b, j].float().cpu().numpy()
                err = np.abs(g - o)
                bad = err > ATOL + RTOL * np.abs(o)
                assert not bad.any(), (f"B{B} H{H} b{b} j{j}: {bad.sum()} outside tol, heads "
                                       f"{sorted(set(np.nonzero(bad)[0].tolist()))[:8]}, max err "
                                       f"{err.max():.3g}")
                gl = lse[b, j].cpu().numpy()
                assert (np.abs(gl - ls) <= ATOL + RTOL * np.abs(ls)).all()
                # how peaked the softmax of head 0 is (the pattern's point)
                deq = oracle.dequant_rows(oracle.ROW_E4M3_656, r)
                qf = np.array([oracle.bf16(int(x)) for x in qbits[0]])
                z = deq @ qf * tau
                w = np.exp(z - z.max())
                peak_weight = max(peak_weight, w.max() / w.sum())
                checked += 1
        assert checked > 0
        assert peak_weight > 0.99
    finally:
        pool.close()


@pytest.mark.parametrize("B,nq,H,K,N", [
    (2, 1, 128, 2048, 5000),    # many row ranges per query: partials + combine
    (32, 1, 128, 2048, 2600),   # two ranges per query: the 2-CTA cluster merge
    (20, 4, 128, 2048, 2300),   # one range per query (MTP3: 80 queries)
    (3, 1, 128, 704, 1500),     # K not a multiple of the 128-row chunk
    (3, 2, 16, 512, 1400),      # 16 heads: the CUDA-core kernel
    (64, 1, 128, 704, 1500),    # 64 queries: the 2-CTA latent-split kernel, ragged K
    (17, 4, 256, 1024, 1800),   # 256 heads: two 128-head groups per query (68 x 2 groups)
])
def test_peaked_softmax_and_rescale(B, nq, H, K, N):
    _run(B, nq, H, K, N, seed=11 + B)


def test_fp16_range_is_reported():
    """The tensor-core attention computes in fp16: a row whose group scale
    would carry E4M3 values beyond 65504, or a query value beyond it, sets
    HS_ERR_RANGE in the sticky error word; in-range inputs do not."""
    from sparse_mla_kv_fp8_gb300 import hs
    dev = torch.device("cuda")
    B, H, K, N, P = 2, 128, 256, 600, 64
    cfg = hs.make_config(max_requests=B, max_tokens=640, page_tokens=P, top_k=K, num_spec=0,
                         tail_tokens=0, num_mla_layers=1, mla_heads=H, idx_heads=8, idx_dim=32,
                         row_fmt=hs.HS_ROW_E4M3_656, idx_fmt=hs.HS_IDX_E4M3, gpu_blocks=24)
    pool = hs.Pool(cfg, device=dev)
    try:
        for b in range(B):
            pool.open(b, hs.HS_FULL)
            r = wl.mla_rows(3, b, 0, N, 1, wl.ROW_E4M3_656, device=dev)
            if b == 1:
                sc = r[77, 0, 512:528].clone().view(torch.float32)
                sc[2] = 200.0  # 448 * 200 > 65504
                r[77, 0, 512:528] = sc.view(torch.uint8)
            pool.append(b, r, wl.idx_keys(3, b, 0, N, 32, wl.IDX_E4M3, device=dev))
        tk = torch.stack([torch.arange(0, 2 * K, 2, dtype=torch.int32)] * B)[:, None].to(dev)
        rid = torch.empty_like(tk)
        pool.resolve(tk, B, 1, rid)
        q = wl.mla_query(3, 1, B, 1, H, 1, dev)[0].contiguous()
        out = torch.empty((B, 1, H, 512), dtype=torch.bfloat16, device=dev)
        # request 0 alone: in range
        pool.sparse_mla_decode(0, q[:1].contiguous(), rid[:1].contiguous(), 1, 1, 0.04, out[:1])
        assert pool.get_error() == hs.HS_OK
        # request 1 reads row 76 or 77? entries are even tokens: 76 is read, 77 is not
        pool.sparse_mla_decode(0, q, rid, B, 1, 0.04, out)
        assert pool.get_error() == hs.HS_OK
        tk2 = tk.clone()
        tk2[1, 0, 38] = 77  # between 76 and 78: still ascending
        pool.resolve(tk2, B, 1, rid)
        pool.sparse_mla_decode(0, q, rid, B, 1, 0.04, out)
        assert pool.get_error() == hs.HS_ERR_RANGE
        # a query value beyond fp16's range
        q2 = q.clone()
        q2[0, 0, 5, 100] = 70000.0
        pool.resolve(tk, B, 1, rid)
        pool.sparse_mla_decode(0, q2, rid, B, 1, 0.04, out)
        assert pool.get_error() == hs.HS_ERR_RANGE
        pool.sparse_mla_decode(0, q, rid, B, 1, 0.04, out)
        assert pool.get_error() == hs.HS_OK
    finally:
        pool.close()
