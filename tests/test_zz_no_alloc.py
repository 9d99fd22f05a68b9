"""The allocation-free top-K entry point (hs_topk_noalloc).

It exists for callers that cannot allocate device memory (an engine that
reserved most of the GPU for its own pool, host code that must avoid the
synchronising allocation calls): its scratch is a static area inside the
library.  This test calls it through the C ABI twice in a row, on different
scores, and checks both results against the pool-based hs_topk (indices are
integers: bit-exact), then checks that oversize requests are refused.  It is
collected last so that a stopping run has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

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
