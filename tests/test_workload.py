"""The seeded input generators that both the oracle tests and the CUDA path
consume (``sparse_mla_kv_fp8_gb300/workload.py``), on CPU: any token range
regenerates identically, and the drawn top-K streams that stand in for the
agentic traces have the recipe's structure.  They hold none of the method's
arithmetic; these tests check only what they promise."""
import numpy as np
import pytest
import torch

from sparse_mla_kv_fp8_gb300 import workload as wl


@pytest.mark.parametrize("t0,n", [(0, 1), (4090, 20), (5000, 9000), (12287, 2)])
def test_indexer_keys_regenerate_by_range(t0, n):
    whole = wl.idx_keys(3, 1, 0, 16384, 128, wl.IDX_E4M3)
    part = wl.idx_keys(3, 1, t0, n, 128, wl.IDX_E4M3)
    assert torch.equal(part, whole[t0:t0 + n])
    assert not torch.equal(wl.idx_keys(3, 2, t0, n, 128, wl.IDX_E4M3), part)  # another request


@pytest.mark.parametrize("t0,n", [(0, 3), (1020, 10), (1500, 2000)])
def test_latent_rows_regenerate_by_range(t0, n):
    whole = wl.mla_rows(5, 0, 0, 4096, 2, wl.ROW_E4M3_656)
    part = wl.mla_rows(5, 0, t0, n, 2, wl.ROW_E4M3_656)
    assert part.shape == (n, 2, 656)
    assert torch.equal(part, whole[t0:t0 + n])


@pytest.mark.parametrize("kind", ["recency_zipf", "uniform_zipf"])
def test_drawn_lists_are_k_distinct_visible_tokens_in_order(kind):
    P, K, vis, T = 64, 2048, 142000 - 3, 4096
    a = wl.drawn_topk(0, 7, 21, 0, vis, K, P, kind, T)
    assert a.shape == (K,) and a.dtype == np.int32
    assert (np.diff(a) > 0).all() and a[0] >= 0 and a[-1] < vis
    assert np.array_equal(a, wl.drawn_topk(0, 7, 21, 0, vis, K, P, kind, T))  # seeded
    assert not np.array_equal(a, wl.drawn_topk(0, 7, 22, 0, vis, K, P, kind, T))  # next step


def test_drawn_lists_cover_everything_when_k_does():
    a = wl.drawn_topk(0, 0, 1, 0, 100, 128, 64, "recency_zipf", 64)
    assert a[:100].tolist() == list(range(100)) and (a[100:] == -1).all()


def test_recency_zipf_mix():
    """Half the tokens from a page-geometric law over the distance from the
    newest page (mean about 63 pages), half Zipf(1.1) over the pages older
    than the tail window: most of the first half lies within 256 pages of
    the newest, and a good part of the list lies far behind it."""
    P, K, vis, T = 64, 2048, 142000, 4096
    a = wl.drawn_topk(1, 3, 40, 0, vis, K, P, "recency_zipf", T)
    newest = (vis - 1) // P
    near = (newest - a // P) <= 256
    assert near.sum() >= 0.45 * K
    assert (~near).sum() >= 0.2 * K
    b = wl.drawn_topk(1, 3, 40, 0, vis, K, P, "uniform_zipf", T)
    assert ((newest - b // P) <= 256).sum() < 0.3 * K  # no recency half there


def test_streams_are_the_per_list_draws():
    P, K, N, nq, T = 64, 256, 20000, 2, 1024
    s = wl.drawn_streams(0, 3, [1, 2], nq, N, K, P, "recency_zipf", T, procs=1)
    assert s.shape == (2, 3, nq, K)
    for i, step in enumerate([1, 2]):
        for b in range(3):
            for j in range(nq):
                want = wl.drawn_topk(0, b, step, j, N - nq + j + 1, K, P, "recency_zipf", T)
                assert np.array_equal(s[i, b, j], want)
