"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against a closed form, a brute force, an
independent library routine, a hand-worked example or an invariant the
pages state, so that a plausible slip (a dropped term, a wrong sign or index,
a transposed operand) fails at least one of them.  No GPU is used.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_mla_kv_fp8_gb300 import workload as wl

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _json(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def test_e4m3_ocp_code_points():
    for code, val in _json("e4m3_ocp_points.json")["points"]:
        got = oracle.e4m3(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), code


def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])


def test_bf16_matches_torch():
    bits = torch.arange(0, 65536, 97, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    for i, b in enumerate(bits.numpy().astype(np.uint16)):
        got = oracle.bf16(int(b))
        if math.isnan(ref[i]):
            assert math.isnan(got)
        else:
            assert got == ref[i]


def test_dequant_row_e4m3_layout():
    # codes i -> a known value per position, a distinct scale per 128-group
    row = np.zeros(656, np.uint8)
    codes = np.array([0x38, 0xB8, 0x40, 0x30] * 128, np.uint8)  # 1, -1, 2, 0.5
    row[:512] = codes
    scales = np.array([0.5, 2.0, 3.0, -1.25], np.float32)
    row[512:528] = scales.view(np.uint8)
    rope = torch.linspace(-3, 3, 64).to(torch.bfloat16)
    row[528:656] = rope.view(torch.uint8).numpy()
    got = oracle.dequant_rows(oracle.ROW_E4M3_656, row[None])[0]
    base = np.array([1.0, -1.0, 2.0, 0.5] * 128)
    want = np.concatenate([base * np.repeat(scales.astype(np.float64), 128),
                           rope.to(torch.float64).numpy()])
    np.testing.assert_array_equal(got, want)


def test_dequant_row_f32_layout():
    x = np.random.default_rng(1).standard_normal(576).astype(np.float32)
    got = oracle.dequant_rows(oracle.ROW_F32_2304, x.view(np.uint8)[None])[0]
    np.testing.assert_array_equal(got, x.astype(np.float64))


def test_generator_rows_roundtrip_within_e4m3_step():
    """The FP8 rows the generator encodes decode to within half an E4M3 step of
    the N(0,1) draw (sanity of the layout both sides read)."""
    g = torch.Generator().manual_seed(3)
    x = torch.randn((5, 576), generator=g)
    rows = wl.encode_rows(x, wl.ROW_E4M3_656).numpy()
    y = oracle.dequant_rows(oracle.ROW_E4M3_656, rows)
    nope_err = np.abs(y[:, :512] - x[:, :512].double().numpy())
    amax = x[:, :512].abs().reshape(5, 4, 128).amax(-1).double().numpy()
    # E4M3 relative step is 2^-3; half of it times the largest magnitude in range
    bound = np.repeat(amax, 128, axis=1) * (2 ** -4) + 1e-12
    assert (nope_err <= bound).all()
    np.testing.assert_array_equal(y[:, 512:], x[:, 512:].to(torch.bfloat16).double().numpy())


# --------------------------------------------------------------------------
# indexer: exact integer recomputation
# --------------------------------------------------------------------------
def _int_recompute(qi, ki, wk, sig_e, N, nq, relu_gate=True):
    """Closed form in integers.  q = qi/8, k = ki/8, w = 2^-wk, sigma = 2^sig_e:
    s = sum_h 2^-wk * max(2^sig_e * (qi.ki)/64, 0), returned as an exact
    rational via integers scaled by 2^(6+3+1).  relu_gate=False drops the
    max (the identity gate)."""
    dots = np.einsum("jhd,td->jht", qi.astype(np.int64), ki.astype(np.int64))  # units 2^-6
    relu = np.maximum(dots, 0) if relu_gate else dots
    # term = 2^-wk * 2^sig_e * dot * 2^-6 ; scale everything by 2^10
    scale = (2 ** (3 - wk))[:, :, None].astype(np.int64)           # 2^-wk * 2^3
    sig = (2 ** (sig_e + 1))[None, None, :].astype(np.int64)      # 2^sig_e * 2^1
    s_int = (relu * scale * sig).sum(1)                            # units 2^-(6+3+1)
    s = s_int.astype(np.float64) / 2.0 ** 10
    for j in range(nq):
        s[j, N - nq + j + 1:] = -np.inf
    return s


@pytest.mark.parametrize("fmt,Hi,Di,bound,nq,N,sig", [
    (oracle.IDX_E4M3, 8, 32, 8, 1, 50, False),
    (oracle.IDX_E4M3, 4, 16, 8, 4, 37, True),
    (oracle.IDX_F32, 4, 32, 64, 1, 64, False),
    (oracle.IDX_F32, 3, 8, 64, 2, 21, True),
])
def test_indexer_scores_exact_int64(fmt, Hi, Di, bound, nq, N, sig):
    rng = np.random.default_rng(7)
    qi = rng.integers(-bound, bound + 1, (nq, Hi, Di))
    ki = rng.integers(-bound, bound + 1, (N, Di))
    wk = rng.integers(0, 4, (nq, Hi))
    sig_e = rng.integers(-1, 2, N) if sig else np.zeros(N, np.int64)
    w = (2.0 ** -wk).astype(np.float32)
    sigma = (2.0 ** sig_e).astype(np.float32)
    if fmt == oracle.IDX_E4M3:
        q = torch.from_numpy(qi / 8.0).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        k = torch.from_numpy(ki / 8.0).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    else:
        q = (qi / 8.0).astype(np.float32)
        k = (ki / 8.0).astype(np.float32)
    got = oracle.indexer_scores(fmt, q, w, k, sigma, N)
    want = _int_recompute(qi, ki, wk, sig_e, N, nq)
    np.testing.assert_array_equal(got.astype(np.float64), want)


def test_visibility_reading_matches_the_scored_tokens():
    """oracle.visible (the reading the harnesses use: query j of nq sees
    [0, N - nq + j + 1)) names exactly the tokens the indexer scores, which
    the integer recomputation above pins; the last query sees every token."""
    rng = np.random.default_rng(3)
    for nq, N in ((1, 9), (2, 12), (4, 11)):
        q = rng.standard_normal((nq, 2, 8)).astype(np.float32)
        k = rng.standard_normal((N, 8)).astype(np.float32)
        w = np.ones((nq, 2), np.float32)
        s = oracle.indexer_scores(oracle.IDX_F32, q, w, k, np.ones(N, np.float32), N)
        for j in range(nq):
            v = oracle.visible(N, nq, j)
            assert np.isfinite(s[j, :v]).all() and np.isneginf(s[j, v:]).all()
        assert oracle.visible(N, nq, nq - 1) == N


def test_indexer_identity_gate_build(tmp_path):
    """The oracle built with -DHSO_IDENTITY_GATE (the other plain reading of the
    gate) against the same integer closed form without the max; the default
    build reports the ReLU gate."""
    import ctypes
    import subprocess
    lib_path = str(tmp_path / "liboracle_identity.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    "-DHSO_IDENTITY_GATE", os.path.join(os.path.dirname(oracle.__file__), "hs_oracle.c"), "-o",
                    lib_path, "-lm"], check=True)
    lib = ctypes.CDLL(lib_path)
    assert lib.hso_gate_is_identity() == 1
    assert oracle._load().hso_gate_is_identity() == 0
    rng = np.random.default_rng(11)
    nq, Hi, Di, N = 2, 4, 32, 40
    qi = rng.integers(-8, 9, (nq, Hi, Di))
    ki = rng.integers(-8, 9, (N, Di))
    wk = rng.integers(0, 4, (nq, Hi))
    sig_e = rng.integers(-1, 2, N)
    q = np.ascontiguousarray(torch.from_numpy(qi / 8.0).float().to(torch.float8_e4m3fn)
                             .view(torch.uint8).numpy())
    k = np.ascontiguousarray(torch.from_numpy(ki / 8.0).float().to(torch.float8_e4m3fn)
                             .view(torch.uint8).numpy())
    w = np.ascontiguousarray((2.0 ** -wk).astype(np.float32))
    sigma = np.ascontiguousarray((2.0 ** sig_e).astype(np.float32))
    out = np.empty((nq, N), np.float32)
    p = lambda a: ctypes.c_void_p(a.ctypes.data)
    lib.hso_indexer_scores(ctypes.c_int(oracle.IDX_E4M3), p(q), p(w), p(k), p(sigma),
                           ctypes.c_int(N), ctypes.c_int(nq), ctypes.c_int(Hi), ctypes.c_int(Di),
                           p(out))
    want = _int_recompute(qi, ki, wk, sig_e, N, nq, relu_gate=False)
    np.testing.assert_array_equal(out.astype(np.float64), want)
    assert (want[np.isfinite(want)] < 0).any()  # the identity gate keeps negative terms


def test_indexer_generator_values_are_exact_grid():
    """The generator's E4M3 indexer values are exactly m/8, |m| <= 8."""
    v = wl.idx_values((4096,), wl.IDX_E4M3, 11).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    m = v * 8
    assert np.array_equal(m, np.round(m)) and np.abs(m).max() <= 8
    f = wl.idx_values((4096,), wl.IDX_F32, 11).double().numpy() * 8
    assert np.array_equal(f, np.round(f)) and np.abs(f).max() <= 64


# --------------------------------------------------------------------------
# top-K
# --------------------------------------------------------------------------
def _brute_topk(s, vis, K):
    """Enumerate every subset of size min(K, vis); keep the one where each
    chosen score beats each unchosen one, ties going to the lower index."""
    m = min(K, vis)
    found = []
    for sub in itertools.combinations(range(vis), m):
        ss = set(sub)
        ok = True
        for a in sub:
            for b in range(vis):
                if b in ss:
                    continue
                if s[a] < s[b] or (s[a] == s[b] and a > b):
                    ok = False
                    break
            if not ok:
                break
        if ok:
            found.append(sub)
    assert len(found) == 1
    out = np.full(K, -1, np.int32)
    out[:m] = sorted(found[0])
    return out


@pytest.mark.parametrize("seed", range(12))
def test_topk_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 11))
    vis = int(rng.integers(0, n + 1))
    K = int(rng.integers(1, 6))
    s = rng.integers(0, 4, n).astype(np.float32)  # many ties
    if seed % 3 == 0:
        s = rng.standard_normal(n).astype(np.float32)
    got = oracle.topk(s, vis, K)
    np.testing.assert_array_equal(got, _brute_topk(s, vis, K))


@pytest.mark.parametrize("seed", range(6))
def test_topk_signed_zeros_tie(seed):
    """-0 and +0 are equal scores: they tie like any other equal scores and
    go to the lower index (brute force on tiny rows of +-0 and +-1)."""
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(4, 11))
    s = np.zeros(n, np.float32)
    s[rng.random(n) < 0.5] = -0.0
    s[rng.integers(0, n, 2)] = rng.choice(np.array([1.0, -1.0], np.float32), 2)
    s[rng.integers(0, n)] = -0.0
    assert np.signbit(s[s == 0]).any()
    K = int(rng.integers(1, n))
    got = oracle.topk(s, n, K)
    np.testing.assert_array_equal(got, _brute_topk(s, n, K))


def test_topk_invariants_large_with_ties():
    rng = np.random.default_rng(5)
    N, K = 5000, 777
    s = rng.integers(0, 50, N).astype(np.float32)
    got = oracle.topk(s, N, K)
    assert (np.diff(got) > 0).all() and len(got) == K
    sel = np.zeros(N, bool)
    sel[got] = True
    thr = s[sel].min()
    assert (s[~sel] <= thr).all()
    # ties at the threshold: chosen ones have lower indices than unchosen ones
    tie_in = np.nonzero(sel & (s == thr))[0]
    tie_out = np.nonzero(~sel & (s == thr))[0]
    if len(tie_out):
        assert tie_in.max() < tie_out.min()


def test_topk_k_at_least_visible_selects_all():
    s = np.random.default_rng(0).standard_normal(30).astype(np.float32)
    got = oracle.topk(s, 20, 32)
    np.testing.assert_array_equal(got[:20], np.arange(20))
    assert (got[20:] == -1).all()


# --------------------------------------------------------------------------
# resolve / LRU
# --------------------------------------------------------------------------
def test_resolve_hand_worked_example():
    ex = _json("resolve_hand_example.json")
    P, N, C = ex["P"], ex["N"], ex["C"]
    resident = np.zeros((N + P - 1) // P, np.uint8)
    resident[ex["resident_pages"]] = 1
    np.testing.assert_array_equal(resident, oracle.page_resident(oracle.MIXED, N, ex["T"], P))
    st = oracle.HotState(C, N)
    for i, step in enumerate(ex["steps"]):
        r = st.resolve(resident, P, N, np.array([step["idx"]], np.int32))
        assert r["status"] == 0
        assert r["loc_kind"][0].tolist() == step["kind"], i
        assert r["loc_val"][0].tolist() == step["val"], i
        assert [[int(a), int(b)] for a, b in zip(r["miss_tok"], r["miss_slot"])] == step["misses"], i
        assert st.slot_token.tolist() == step["slot_token"], i
        assert st.stamp.tolist() == step["stamp"], i
        assert int(st.step[0]) == i + 1
    bad = ex["then_out_of_range"]
    r = st.resolve(resident, P, N, np.array([bad["idx"]], np.int32))
    assert r["status"] == bad["status"]


class HistoryLRU:
    """Independent formulation of the same policy: no stamps are kept; the
    last use of a slot is found by scanning a full access log."""

    def __init__(self, C):
        self.C = C
        self.log = []  # (step, slot)
        self.token_of = {}  # slot -> token
        self.step = 0

    def last_use(self, c):
        t = 0
        for s, cc in self.log:
            if cc == c:
                t = max(t, s)
        return t

    def resolve(self, resident, P, idx):
        self.step += 1
        U = sorted(set(int(x) for x in idx.ravel() if x >= 0))
        slot_of_tok = {t: c for c, t in self.token_of.items()}
        where = {}
        misses = []
        for u in U:
            if resident[u // P]:
                where[u] = (1, u)
            elif u in slot_of_tok:
                self.log.append((self.step, slot_of_tok[u]))
                where[u] = (2, slot_of_tok[u])
            else:
                misses.append(u)
        free = [c for c in range(self.C) if self.last_use(c) < self.step]
        free.sort(key=lambda c: (self.last_use(c), c))
        victims = sorted(free[:len(misses)])
        assert len(victims) == len(misses)
        for u, c in zip(misses, victims):
            self.token_of[c] = u
            self.log.append((self.step, c))
            where[u] = (2, c)
        return where, list(zip(misses, victims))


@pytest.mark.parametrize("nq,K,C,mode", [(1, 8, 16, oracle.MIXED), (2, 6, 18, oracle.MIXED),
                                         (4, 4, 20, oracle.ZERO), (1, 8, 8, oracle.MIXED)])
def test_resolve_matches_history_replay(nq, K, C, mode):
    rng = np.random.default_rng(nq * 100 + K)
    P, N, T = 4, 64, 12
    resident = oracle.page_resident(mode, N, T, P)
    st = oracle.HotState(C, N)
    ref = HistoryLRU(C)
    hot_before = set()
    zipf_p = np.zeros(N)
    zipf_p[rng.permutation(N)] = np.arange(1, N + 1, dtype=np.float64) ** -1.1
    zipf_p /= zipf_p.sum()
    total_hits = total_misses = evictions = 0
    for step in range(40):
        # skewed draws so that hits, misses and evictions all happen
        idx = np.full((nq, K), -1, np.int32)
        for j in range(nq):
            # four steps in five draw from a Zipf law over a fixed permutation
            # (repeats: hits and refreshed stamps), the fifth uniformly (a
            # burst of misses that evicts)
            pool = rng.choice(N, size=K, replace=False, p=None if step % 5 == 4 else zipf_p)
            idx[j] = np.sort(pool)
        r = st.resolve(resident, P, N, idx)
        assert r["status"] == 0
        where, pairs = ref.resolve(resident, P, idx)
        for j in range(nq):
            for k in range(K):
                u = idx[j, k]
                assert (r["loc_kind"][j, k], r["loc_val"][j, k]) == where[int(u)]
        assert list(zip(r["miss_tok"].tolist(), r["miss_slot"].tolist())) == pairs
        # invariants: tail tokens never enter the hot buffer; occupancy <= C;
        # misses = |U \ (resident u hot before)|; hot_map and slot_token agree
        U = set(int(x) for x in idx.ravel())
        nonres = {u for u in U if not resident[u // P]}
        assert r["misses"] == len(nonres - hot_before)
        held = [t for t in st.slot_token.tolist() if t >= 0]
        assert len(held) <= C and len(set(held)) == len(held)
        assert all(not resident[t // P] for t in held)
        for c, t in enumerate(st.slot_token.tolist()):
            if t >= 0:
                assert st.hot_map[t] == c
        assert (st.hot_map >= 0).sum() == len(held)
        evictions += len(hot_before - set(held))
        total_hits += r["hits"]
        total_misses += r["misses"]
        hot_before = set(held)
    # the draws did what they are for
    assert total_hits > 0 and total_misses > 0 and evictions > 0


def test_resolve_full_residency_never_misses():
    P, N = 8, 200
    st = oracle.HotState(16, N)
    res = oracle.page_resident(oracle.FULL, N, 0, P)
    rng = np.random.default_rng(2)
    for _ in range(10):
        idx = np.sort(rng.choice(N, 8, replace=False)).astype(np.int32)[None]
        r = st.resolve(res, P, N, idx)
        assert r["misses"] == 0 and r["hits"] == 0 and r["resident"] == 8
        assert (r["loc_kind"] == 1).all() and (r["loc_val"] == idx).all()


def test_resolve_capacity_error_when_buffer_too_small():
    """Four misses, three slots: a capacity error, handled gracefully (our
    reading: the pages plan to relax the hot-buffer sizing and say nothing
    about a shortfall).  The three lowest tokens take the three slots, token
    13 reads nothing, and the step counts."""
    P, N = 4, 64
    st = oracle.HotState(3, N)
    res = oracle.page_resident(oracle.ZERO, N, 0, P)
    r = st.resolve(res, P, N, np.array([[1, 5, 9, 13]], np.int32))
    assert r["status"] == oracle.ERR_CAPACITY
    assert r["loc_kind"].tolist() == [[2, 2, 2, 0]]
    assert r["loc_val"].tolist() == [[0, 1, 2, -1]]
    assert (r["misses"], r["hits"], r["resident"]) == (3, 0, 0)
    assert st.slot_token.tolist() == [1, 5, 9] and st.hot_map[13] == -1
    assert int(st.step[0]) == 1
    # next step: 13 and 1 again; 1 hits (stamp 2), 13 takes the oldest slot
    # not used in this step (slot 1: stamp 1, lower than slot 2's)
    r = st.resolve(res, P, N, np.array([[1, 13, -1, -1]], np.int32))
    assert r["status"] == 0
    assert r["loc_kind"].tolist() == [[2, 2, 0, 0]]
    assert r["loc_val"].tolist() == [[0, 1, -1, -1]]
    assert st.slot_token.tolist() == [1, 13, 9] and st.hot_map[5] == -1


def test_resolve_shortfall_never_evicts_rows_of_this_step():
    """Under a hot-buffer shortfall (fewer free-able slots than misses; the
    capacity error of our reading), a slot that this step already uses is
    never a victim ("Les trois états de résidence": a hit refreshes its LRU
    entry, so it is the most recent use), and every entry that the step
    locates in the hot buffer still holds its token when the step ends.
    Hand-worked, then as an invariant over random shortfalls."""
    P, N = 4, 64
    res = oracle.page_resident(oracle.ZERO, N, 0, P)
    st = oracle.HotState(2, N)
    r = st.resolve(res, P, N, np.array([[1, 5, -1]], np.int32))
    assert r["status"] == 0 and st.slot_token.tolist() == [1, 5]
    # step 2: 1 hits slot 0 (stamp 2); the misses 9 and 13 find one slot of
    # an earlier step (slot 1): 9 takes it, 13 reads nothing, slot 0 keeps 1
    r = st.resolve(res, P, N, np.array([[1, 9, 13]], np.int32))
    assert r["status"] == oracle.ERR_CAPACITY
    assert r["loc_kind"].tolist() == [[2, 2, 0]]
    assert r["loc_val"].tolist() == [[0, 1, -1]]
    assert st.slot_token.tolist() == [1, 9]
    assert (st.hot_map[1], st.hot_map[9], st.hot_map[5], st.hot_map[13]) == (0, 1, -1, -1)
    rng = np.random.default_rng(21)
    shortfalls = 0
    for C in (3, 5, 8):
        st = oracle.HotState(C, N)
        for _ in range(40):
            idx = np.stack([np.sort(rng.choice(16, 4, replace=False)) for _ in range(2)]).astype(np.int32)
            r = st.resolve(res, P, N, idx)
            assert r["status"] in (0, oracle.ERR_CAPACITY)
            shortfalls += r["status"] == oracle.ERR_CAPACITY
            for j, k in zip(*np.nonzero(r["loc_kind"] == 2)):
                assert st.slot_token[r["loc_val"][j, k]] == idx[j, k]
    assert shortfalls > 0


def test_resolve_capacity_rule_always_has_victims():
    """With C = (num_spec+2)*K the victims always exist (union <= nq*K = C-K)."""
    rng = np.random.default_rng(9)
    P, N = 4, 400
    for nq in (1, 2, 4):
        K = 16
        C = (nq + 1) * K
        st = oracle.HotState(C, N)
        res = oracle.page_resident(oracle.ZERO, N, 0, P)
        for _ in range(30):
            idx = np.stack([np.sort(rng.choice(N, K, replace=False)) for _ in range(nq)]).astype(np.int32)
            assert st.resolve(res, P, N, idx)["status"] == 0


def test_page_resident_tail_window():
    P, T = 64, 4096
    for N in (4096, 4097, 5000, 142000):
        r = oracle.page_resident(oracle.MIXED, N, T, P)
        npages = (N + P - 1) // P
        for p in range(npages):
            assert bool(r[p]) == ((p + 1) * P > N - T)
        # the tail covers at least the last T tokens
        assert all(r[t // P] for t in range(max(N - T, 0), N))
    assert oracle.page_resident(oracle.ZERO, 1000, T, P).sum() == 0
    assert oracle.page_resident(oracle.FULL, 1000, T, P).sum() == (1000 + 63) // 64


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def _rows_and_dense(fmt, n, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, 576), generator=g)
    rows = wl.encode_rows(x, fmt)
    if fmt == oracle.ROW_E4M3_656:
        codes = rows[:, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
        sc = rows[:, 512:528].contiguous().view(torch.float32).to(torch.float64)
        rope = rows[:, 528:].contiguous().view(torch.bfloat16).to(torch.float64)
        kv = torch.cat([codes * sc.repeat_interleave(128, 1), rope], 1)
    else:
        kv = rows.contiguous().view(torch.float32).to(torch.float64)
    return rows.numpy(), kv


@pytest.mark.parametrize("fmt", [oracle.ROW_E4M3_656, oracle.ROW_F32_2304])
def test_attention_k_ge_n_equals_dense_sdpa(fmt):
    """When the selection covers every token (K >= N) sparse attention is
    dense attention ("Comment s'y prendre": prompts inside the 2048 selected
    tokens take the dense path).  Reference: torch SDPA in fp64."""
    n, H = 37, 6
    rows, kv = _rows_and_dense(fmt, n, 4)
    q = torch.randn((H, 576), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    tau = 1.0 / math.sqrt(576)
    o, lse = oracle.attention(fmt, q.view(torch.int16).numpy().view(np.uint16), rows, tau)
    qd = q.to(torch.float64)[None, :, None, :].expand(1, H, 1, 576)
    kd = kv[None, None].expand(1, H, n, 576)
    vd = kv[:, :512][None, None].expand(1, H, n, 512)
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, scale=tau)[0, :, 0]
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)
    ref_lse = torch.logsumexp(tau * (q.to(torch.float64) @ kv.T), 1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_attention_masked_equals_gathered():
    n, H = 50, 4
    rows, _ = _rows_and_dense(oracle.ROW_E4M3_656, n, 8)
    q = torch.randn((H, 576), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    qb = q.view(torch.int16).numpy().view(np.uint16)
    mask = np.zeros(n, np.uint8)
    sel = [0, 3, 4, 17, 30, 49]
    mask[sel] = 1
    o1, l1 = oracle.attention(oracle.ROW_E4M3_656, qb, rows, 0.05, mask)
    o2, l2 = oracle.attention(oracle.ROW_E4M3_656, qb, rows[sel], 0.05)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-14)


def test_attention_closed_forms():
    rows, kv = _rows_and_dense(oracle.ROW_F32_2304, 5, 10)
    kv = kv.numpy()
    q = torch.randn((3, 576), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    qb = q.view(torch.int16).numpy().view(np.uint16)
    # one row: output is that row's value part, lse is its score
    o, lse = oracle.attention(oracle.ROW_F32_2304, qb, rows[2:3], 0.1)
    np.testing.assert_allclose(o, np.repeat(kv[2:3, :512], 3, 0), rtol=0, atol=0)
    np.testing.assert_allclose(lse, 0.1 * (q.double().numpy() @ kv[2]), rtol=1e-14)
    # equal scores (q = 0): output is the mean of the rows, lse = log(n)
    z = np.zeros((2, 576), np.uint16)
    o, lse = oracle.attention(oracle.ROW_F32_2304, z, rows, 0.1)
    np.testing.assert_allclose(o, np.repeat(kv[:, :512].mean(0, keepdims=True), 2, 0), rtol=1e-14)
    np.testing.assert_allclose(lse, np.log(5), rtol=1e-15)
    # nothing selected
    o, lse = oracle.attention(oracle.ROW_F32_2304, qb, rows, 0.1, np.zeros(5, np.uint8))
    assert (o == 0).all() and np.isneginf(lse).all()


def test_hot_buffer_sizing_follows_the_printed_rule():
    """The pages print the hot-buffer sizes: 2 x top-K rows per request, and
    (num_speculative_tokens + 2) x top-K under MTP (fixture constants, each
    cited).  The library derives C from the config when hot_rows = 0: its
    arena size must equal that of a config stating C explicitly by the
    printed rule, and differ from one stating a neighbouring size.  The
    oracle's resolve must then always find victims at that C, even when every
    step's nq lists are disjoint from each other and from the last step's."""
    from sparse_mla_kv_fp8_gb300 import build, hs
    build.build()
    pc = _json("page_constants.json")
    K = pc["top_k"]["value"]
    for ns, C in ((0, pc["hot_rows_per_topk_default"]["value"] * K),
                  (pc["mtp_speculative_tokens"]["value"],
                   (pc["mtp_speculative_tokens"]["value"] + pc["hot_rows_per_topk_mtp_offset"]["value"]) * K)):
        base = dict(max_requests=2, max_tokens=16384, page_tokens=64, top_k=K, num_spec=ns,
                    tail_tokens=4096, num_mla_layers=4, mla_heads=128, idx_heads=64, idx_dim=128,
                    gpu_blocks=600, host_blocks=600)
        derived = hs.required_bytes(hs.make_config(**base))
        assert derived == hs.required_bytes(hs.make_config(hot_rows=C, **base))
        assert derived != hs.required_bytes(hs.make_config(hot_rows=C - 64, **base))
        assert derived != hs.required_bytes(hs.make_config(hot_rows=C + 64, **base))
    # C = (ns + 2) K at the MTP3 sizing, scaled down to K = 8 so the oracle
    # runs quickly; adversarial lists: every query of every step new
    ns = pc["mtp_speculative_tokens"]["value"]
    nq, k = ns + 1, 8
    Cs = (ns + pc["hot_rows_per_topk_mtp_offset"]["value"]) * k
    P, N = 4, 4000
    st = oracle.HotState(Cs, N)
    res = oracle.page_resident(oracle.ZERO, N, 0, P)
    t = 0
    for _ in range(20):
        idx = np.arange(t, t + nq * k, dtype=np.int32).reshape(nq, k)
        t += nq * k
        r = st.resolve(res, P, N, idx)
        assert r["status"] == 0 and r["misses"] == nq * k


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_topk_of_shard_candidates_equals_topk_of_the_whole(seed):
    """The property the context-parallel merge rests on: the top-K of a row
    is the top-K of the union of its shards' top-K lists (ties to the lower
    token, with heavy ties in the scores)."""
    rng = np.random.default_rng(seed)
    N, K = 700, 64
    s = rng.integers(0, 30, N).astype(np.float32)  # many equal scores
    whole = oracle.topk(s, N, K)
    cuts = sorted(rng.choice(np.arange(1, N), 3, replace=False).tolist())
    bounds = [0] + cuts + [N]
    cand = []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        loc = oracle.topk(s[lo:hi], hi - lo, K)
        cand += [lo + t for t in loc if t >= 0]
    cand = np.array(cand)
    order = np.lexsort((cand, -s[cand]))  # score descending, then token ascending
    merged = np.sort(cand[order[:K]])
    np.testing.assert_array_equal(merged, whole)


@pytest.mark.parametrize("nq", [1, 4])
def test_zero_residency_start_gives_full_residency_outputs(nq):
    """Resolve + attention in the oracle, run from a zero-residency start and
    from full residency over the same top-K lists: each entry reads a row
    from its own place (the truth for a resident page, a hot-buffer slot
    filled by the miss copies otherwise), and the attention outputs are
    identical step after step ("Les trois états de résidence": a request
    that starts with empty slots receives its rows as the indexer asks for
    them).  The hot buffer is simulated as slot arrays filled with the host
    rows of the misses; a wrong slot, a missed copy or a stale entry changes
    the output."""
    rng = np.random.default_rng(nq)
    P, N, K, H = 8, 400, 24, 4
    C = (nq + 1) * K
    g = torch.Generator().manual_seed(31)
    truth = wl.encode_rows(torch.randn((N, 576), generator=g), oracle.ROW_E4M3_656).numpy()
    hot = {oracle.ZERO: oracle.HotState(C, N), oracle.FULL: oracle.HotState(C, N),
           oracle.MIXED: oracle.HotState(C, N)}
    slots = {m: np.zeros((C, truth.shape[1]), np.uint8) for m in hot}
    tau = 1.0 / math.sqrt(576)
    hits = 0
    for step in range(12):
        idx = np.full((nq, K), -1, np.int32)
        for j in range(nq):
            lo = 0 if step % 3 else 200  # revisit a region: hits after misses
            n = K if j % 2 == 0 else K - 5
            idx[j, :n] = np.sort(rng.choice(np.arange(lo, lo + 200), n, replace=False))
        q = torch.randn((nq, H, 576), generator=g).to(torch.bfloat16)
        outs = {}
        for mode, st in hot.items():
            res = oracle.page_resident(mode, N, 64, P)
            r = st.resolve(res, P, N, idx)
            assert r["status"] == 0
            for u, c in zip(r["miss_tok"], r["miss_slot"]):
                slots[mode][c] = truth[u]  # the miss copy: exactly one row
            if mode == oracle.ZERO:
                hits += r["hits"]
            per_q = []
            for j in range(nq):
                rows = []
                for k in range(K):
                    kind, val = r["loc_kind"][j, k], r["loc_val"][j, k]
                    if kind == 1:
                        rows.append(truth[val])
                    elif kind == 2:
                        rows.append(slots[mode][val])
                rows = np.stack(rows)
                qb = q[j].view(torch.int16).numpy().view(np.uint16)
                per_q.append(oracle.attention(oracle.ROW_E4M3_656, qb, rows, tau))
            outs[mode] = per_q
        for j in range(nq):
            for mode in (oracle.ZERO, oracle.MIXED):
                np.testing.assert_array_equal(outs[mode][j][0], outs[oracle.FULL][j][0])
                np.testing.assert_array_equal(outs[mode][j][1], outs[oracle.FULL][j][1])
            # and equal to the attention over the selected truth rows
            sel = idx[j][idx[j] >= 0]
            qb = q[j].view(torch.int16).numpy().view(np.uint16)
            o, l = oracle.attention(oracle.ROW_E4M3_656, qb, truth[sel], tau)
            np.testing.assert_array_equal(outs[oracle.FULL][j][0], o)
    assert hits > 0


# --------------------------------------------------------------------------
# pool pressure reading ("Ce qui se passe": offload only under real pressure)
# --------------------------------------------------------------------------
def test_pressure_policy_hand_worked_example():
    """Cap 10 blocks, P = 4, T = 4, hot buffer 2 blocks, three requests opened
    in full residency.  Worked by hand:
      r0 += 12 -> 3 pages (3 used); r1 += 16 -> 4 pages (7); r2 += 8 -> 2 (9).
      r2 += 8 would need 3 + 4 + 4 = 11 blocks.  Flips that free blocks: r1
      (mixed: tail page 3 + 2 hot = 3 < 4); not r0 (page 2 + 2 hot = 3 = 3)
      nor r2 (page 1 + 2 hot = 3 > 2).  Flip r1: 3 + 3 + 4 = 10 fits.
      r0 += 4 would need 4 + 3 + 4 = 11; only r2 frees blocks (3 < 4): flip
      r2, 4 + 3 + 3 = 10 fits.
      Nothing returns while the pool is full.  Close r0 (6 used, 2 open):
      r2 (last flipped) needs 1 more block + 2 spare <= 4 free: back; then
      r1 needs 1 + 2 <= 3 free: back (8 used)."""
    pol = oracle.PressurePolicy(cap=10, T=4, P=4, hot_pages=2)
    for r in range(3):
        pol.open(r)
    assert pol.append(0, 12) == ([], oracle.OK)
    assert pol.append(1, 16) == ([], oracle.OK)
    assert pol.append(2, 8) == ([], oracle.OK)
    assert pol.used() == 9
    assert pol.append(2, 8) == ([1], oracle.OK)
    assert pol.used() == 10
    assert pol.append(0, 4) == ([2], oracle.OK)
    assert pol.used() == 10
    assert pol.mode == {0: oracle.FULL, 1: oracle.MIXED, 2: oracle.MIXED}
    assert pol.relieve() == []
    pol.close(0)
    assert pol.used() == 6
    assert pol.relieve() == [2, 1]
    assert pol.used() == 8 and pol.flipped == []


def test_pressure_policy_flips_the_most_pages_and_keeps_a_margin():
    """Cap 23 blocks, P = 4, T = 8, hot buffer 2 blocks.  Worked by hand:
      r0 += 20 -> 5 pages; r1 += 40 -> 10; r2 += 28 -> 7 (22 used).
      r0 += 8 would need 22 - 5 + 7 = 24.  Every request's flip frees blocks
      (mixed: its last two pages + 2 hot = 4, against 5, 10 and 7): the one
      with the most pages, r1, flips: 5 + 4 + 7 = 16, and the append fits
      (18 used, 5 free).
      r1's return adds 10 - 4 = 6 blocks.  With 5 free, nothing returns.
      Close r2 and reopen it with 20 tokens (16 used, 7 free, 3 open): 7
      covers the 6 blocks but not the margin of one block per open request
      (6 + 3 = 9), so nothing returns.  Close r2 again (11 used, 12 free, 2
      open): 6 + 2 <= 12, r1 returns (17 used)."""
    pol = oracle.PressurePolicy(cap=23, T=8, P=4, hot_pages=2)
    for r in range(3):
        pol.open(r)
    assert pol.append(0, 20) == ([], oracle.OK)
    assert pol.append(1, 40) == ([], oracle.OK)
    assert pol.append(2, 28) == ([], oracle.OK)
    assert pol.used() == 22
    assert pol.append(0, 8) == ([1], oracle.OK)
    assert pol.used() == 18
    assert pol.relieve() == []
    pol.close(2)
    pol.open(2)
    assert pol.append(2, 20) == ([], oracle.OK)
    assert pol.used() == 16
    assert pol.relieve() == []
    pol.close(2)
    assert pol.used() == 11
    assert pol.relieve() == [1]
    assert pol.used() == 17 and pol.flipped == []


def test_pressure_policy_capacity_when_no_flip_frees_blocks():
    """Short requests hold fewer pages than a hot buffer: no flip lowers the
    count, so an append past the cap fails and nothing flips."""
    pol = oracle.PressurePolicy(cap=4, T=4, P=4, hot_pages=2)
    pol.open(0)
    pol.open(1)
    assert pol.append(0, 8) == ([], oracle.OK)    # 2 pages
    assert pol.append(1, 8) == ([], oracle.OK)    # 2 pages, pool full
    # a flip of either would hold page 1 + 2 hot = 3 > 2 blocks
    assert pol.append(1, 1) == ([], oracle.ERR_CAPACITY)
    assert pol.N == {0: 8, 1: 8} and pol.used() == 4


def test_pressure_policy_agentic_trace_first_flip_closed_form():
    """Sixteen equal requests of the agentic growth trace (74,160 prompt
    tokens, then 220 decoded and 753 prompt tokens per turn) in a pool of
    20,000 blocks of 64 tokens: 16 x 1,250 pages = 16 x 80,000 tokens fill it
    exactly.  Before turn 7 a request holds 74,160 + 220 + 5 x 973 = 79,245
    tokens, 79,998 after turn 7's prompt; decode appends go request by
    request, so the first append past 80,000 tokens is request 0's third
    decoded token of turn 7, and the largest full request (all tie at 1,250
    pages) is request 0 itself."""
    P, T, hot = 64, 4096, 4096 // 64
    pol = oracle.PressurePolicy(cap=20000, T=T, P=P, hot_pages=hot)
    for b in range(16):
        pol.open(b)
        assert pol.append(b, 74160) == ([], oracle.OK)
    first = None
    for turn in range(7):
        if turn:
            for b in range(16):
                f, st = pol.append(b, 753)
                assert st == oracle.OK and not f
        for d in range(220):
            for b in range(16):
                f, st = pol.append(b, 1)
                assert st == oracle.OK
                if f:
                    first = (turn, d, b, f)
                    break
            if first:
                break
        if first:
            break
    assert first == (6, 2, 0, [0])
    # the flip keeps request 0's tail window (pages 1186..1250) and a hot buffer
    assert pol.blocks(0) == (1250 - (80001 - T) // P + 1) + hot == 129


@pytest.mark.parametrize("seed", range(6))
def test_pressure_policy_flips_only_under_pressure(seed):
    """Random growth traces: an append that fits flips nothing; one that
    does not, flips until it fits, each flip lowering the blocks in use; the
    pool never goes past its cap; a capacity error leaves the request's
    length unchanged and no flip would free a block."""
    rng = np.random.default_rng(seed)
    P, T, hot = 8, 16, 3
    cap = int(rng.integers(40, 90))
    pol = oracle.PressurePolicy(cap=cap, T=T, P=P, hot_pages=hot)
    for r in range(5):
        pol.open(r)
    for _ in range(300):
        r = int(rng.integers(0, 5))
        n = int(rng.integers(1, 40))
        used0 = pol.used()
        fits = used0 - pol.blocks(r) + pol.blocks(r, N=pol.N[r] + n) <= cap
        before = dict(pol.mode), dict(pol.N)
        flips, st = pol.append(r, n)
        assert pol.used() <= cap
        if fits:
            assert flips == [] and st == oracle.OK and pol.N[r] == before[1][r] + n
            continue
        assert flips or st == oracle.ERR_CAPACITY
        # replay the flips one by one: each lowers the count
        mode, used = dict(before[0]), used0
        for x in flips:
            assert mode[x] == oracle.FULL
            gain = (oracle.gpu_blocks(oracle.FULL, before[1][x], T, P, hot)
                    - oracle.gpu_blocks(oracle.MIXED, before[1][x], T, P, hot))
            assert gain > 0
            mode[x] = oracle.MIXED
            used -= gain
        if st == oracle.ERR_CAPACITY:
            assert pol.N[r] == before[1][r]
            assert all(pol.blocks(x, oracle.MIXED) >= pol.blocks(x, oracle.FULL)
                       for x in pol.mode if pol.mode[x] == oracle.FULL)
        else:
            assert pol.N[r] == before[1][r] + n
        if rng.random() < 0.1:
            back = pol.relieve()
            assert pol.used() + len(pol.mode) <= cap or not back
