"""The allocation-free top-K entry point (hs_topk_noalloc).

It exists for callers that cannot allocate device memory (an engine that
reserved most of the GPU for its own pool, host code that must avoid the
synchronising allocation calls): its scratch is a static area inside the
library.  These tests call it through the C ABI: twice in a row on different
scores against the pool-based hs_topk and the oracle (indices are integers:
bit-exact); at its limits (64 rows, rows of 2^20 tokens) against the oracle;
with lengths beyond max_tokens, which it clamps; and with oversize requests,
which it refuses.  The file is collected last so that a stopping run has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hs():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_mla_kv_fp8_gb300 import hs as mod
    return mod


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_topk_matches_pool_topk_twice(hs):
    from harness import Case, Runner
    B, nq, K = 3, 2, 512
    case = Case("noalloc", B=B, N=[20000, 9000, 300], K=K, Hi=8, Di=32, H=16, num_spec=nq - 1,
                mode=hs.HS_FULL)
    r = Runner(case)
    try:
        stride = r.max_tokens
        seq = torch.tensor(r.N, dtype=torch.int32, device=r.dev)
        stream = torch.cuda.current_stream()
        for call in range(2):
            g = torch.Generator().manual_seed(100 + call)
            sc = torch.randint(0, 50 + 20 * call, (B, nq, stride), generator=g).float()
            if call == 1:
                sc[0, 1] = torch.randn(stride, generator=g)  # distinct values on one row
            sc = sc.to(r.dev)
            ref = torch.full((B, nq, K), -9, dtype=torch.int32, device=r.dev)
            got = torch.full((B, nq, K), -9, dtype=torch.int32, device=r.dev)
            r.pool.topk(sc, stride, B, nq, ref)
            st = hs.hs_topk_noalloc(_ptr(sc), stride, _ptr(seq), B, nq, K, stride, _ptr(got),
                                    ctypes.c_void_p(stream.cuda_stream))
            assert st == hs.HS_OK
            torch.cuda.synchronize()
            assert torch.equal(got, ref), f"call {call}: differs from hs_topk"
            s_np, g_np = sc.cpu().numpy(), got.cpu().numpy()
            for b in range(B):
                for j in range(nq):
                    want = oracle.topk(s_np[b, j], oracle.visible(r.N[b], nq, j), K)
                    np.testing.assert_array_equal(g_np[b, j], want)
            # the 300-token request: query 0 sees 299 tokens, query 1 sees 300
            assert (got[2, :, 300:] == -1).all() and int(got[2, 0, 299]) == -1
            assert int(got[2, 1, 299]) == 299
    finally:
        r.close()


def test_noalloc_topk_refuses_beyond_its_scratch(hs):
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # 65 rows > 64
    assert hs.hs_topk_noalloc(_ptr(dummy), 1 << 20, _ptr(dummy), 65, 1, 8, 1 << 20, _ptr(dummy),
                              s) == hs.HS_ERR_CAPACITY
    # more tokens than the scratch covers
    assert hs.hs_topk_noalloc(_ptr(dummy), (1 << 20) + 1, _ptr(dummy), 1, 1, 8, (1 << 20) + 1,
                              _ptr(dummy), s) == hs.HS_ERR_CAPACITY
    # malformed arguments
    assert hs.hs_topk_noalloc(None, 10, _ptr(dummy), 1, 1, 8, 10, _ptr(dummy),
                              s) == hs.HS_ERR_INVALID_ARG
    assert hs.hs_topk_noalloc(_ptr(dummy), 5, _ptr(dummy), 1, 1, 8, 10, _ptr(dummy),
                              s) == hs.HS_ERR_INVALID_ARG


def test_noalloc_topk_at_its_limits_against_the_oracle(hs):
    """64 rows (16 requests x MTP3) with rows of up to 2^20 tokens: the most
    the static scratch covers.  Scores are small integers (heavy ties at the
    threshold), one row distinct values."""
    B, nq, K, T = 16, 4, 2048, 1 << 20
    dev = torch.device("cuda")
    lens = [T, T - 5, 70000, 2049, 2051, 300000, 8192, 8193] + [4096 + 1000 * i for i in range(8)]
    seq = torch.tensor(lens, dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev).manual_seed(7)
    sc = torch.randint(0, 3000, (B, nq, T), generator=g, device=dev).float()
    sc[1, 2] = torch.randn(T, generator=g, device=dev)
    got = torch.full((B, nq, K), -9, dtype=torch.int32, device=dev)
    for call in range(2):  # the second call reuses the scratch the first left behind
        if call == 1:
            sc[5] = -sc[5]
        st = hs.hs_topk_noalloc(_ptr(sc), T, _ptr(seq), B, nq, K, T, _ptr(got),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == hs.HS_OK
        torch.cuda.synchronize()
        s_np, g_np = sc.cpu().numpy(), got.cpu().numpy()
        rows = [(b, j) for b in range(B) for j in range(nq)]
        if call == 1:
            rows = [(5, j) for j in range(nq)] + [(0, 0), (1, 2)]
        for b, j in rows:
            want = oracle.topk(s_np[b, j], oracle.visible(lens[b], nq, j), K)
            np.testing.assert_array_equal(g_np[b, j], want, err_msg=f"call {call} row {b},{j}")


def test_noalloc_topk_clamps_lengths_beyond_max_tokens(hs):
    """A seq_len[b] beyond max_tokens (a caller's device data the library
    cannot check on the host) is clamped on the device: the query sees at most
    max_tokens tokens, and the scores past max_tokens (here the largest of
    the row, in the padding of a wider buffer) are never read or selected."""
    B, nq, K, M, stride = 3, 2, 256, 5000, 8192
    dev = torch.device("cuda")
    seq = torch.tensor([M + 2000, M + 1, 900], dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev).manual_seed(9)
    sc = torch.randint(0, 100, (B, nq, stride), generator=g, device=dev).float()
    sc[:, :, M:] = 1e30  # padding: must not be read
    got = torch.full((B, nq, K), -9, dtype=torch.int32, device=dev)
    st = hs.hs_topk_noalloc(_ptr(sc), stride, _ptr(seq), B, nq, K, M, _ptr(got),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == hs.HS_OK
    torch.cuda.synchronize()
    s_np, g_np = sc.cpu().numpy(), got.cpu().numpy()
    for b in range(B):
        for j in range(nq):
            vis = min(oracle.visible(int(seq[b]), nq, j), M)
            np.testing.assert_array_equal(g_np[b, j], oracle.topk(s_np[b, j], vis, K))
            assert g_np[b, j].max() < M
