"""Plain CPU oracle for the Hybrid HiSparse sparse-MLA decode step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
never loads it, and it shares no code with the CUDA path: the arithmetic lives
in ``hs_oracle.c`` (plain C, fp64), this module only marshals numpy arrays
into it and holds the residency reading below.

Sources: the pages "Un contexte d'un million sur huit H200" (sections "Ce qui
se passe", "Les trois états de résidence", "Ce qu'il faut en retenir") and
"vLLM sert GLM-5.3 en contexte 1M sur 16 H200" (section "Comment s'y
prendre").  Each function names the passage it follows.

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_pins.py`` (none is unpinned).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hs_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# status codes (same numbering as the library's hs_status)
OK, ERR_CAPACITY, ERR_INDEX_RANGE = 0, 3, 5
# formats
ROW_E4M3_656, ROW_F32_2304 = 0, 1
IDX_E4M3, IDX_F32 = 0, 1
# residency modes
FULL, MIXED, ZERO = 0, 1, 2

LATENT, NOPE = 576, 512


def build() -> str:
    """Compile ``hs_oracle.c`` into ``liboracle.so`` with gcc (plain -O2, no
    fast-math, no FP contraction, OpenMP over independent outputs)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        lib.hso_e4m3.restype = ctypes.c_double
        lib.hso_e4m3.argtypes = [ctypes.c_uint8]
        lib.hso_bf16.restype = ctypes.c_double
        lib.hso_bf16.argtypes = [ctypes.c_uint16]
        lib.hso_row_bytes.restype = i32
        lib.hso_row_bytes.argtypes = [i32]
        lib.hso_dequant_row.restype = None
        lib.hso_dequant_row.argtypes = [i32, P, P]
        lib.hso_indexer_scores.restype = None
        lib.hso_indexer_scores.argtypes = [i32, P, P, P, P, i32, i32, i32, i32, P]
        lib.hso_topk.restype = None
        lib.hso_topk.argtypes = [P, i32, i32, P]
        lib.hso_resolve.restype = i32
        lib.hso_resolve.argtypes = [P, P, P, P, i32, P, i32, i32, P, i32, i32,
                                    P, P, P, P, P, P]
        lib.hso_attention.restype = None
        lib.hso_attention.argtypes = [i32, P, i32, P, P, i32, ctypes.c_double, P, P]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def row_bytes(fmt: int) -> int:
    return 656 if fmt == ROW_E4M3_656 else 2304


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def e4m3(code: int) -> float:
    """OCP FP8 E4M3FN decode of one byte."""
    return _load().hso_e4m3(int(code) & 0xFF)


def bf16(bits: int) -> float:
    return _load().hso_bf16(int(bits) & 0xFFFF)


def dequant_rows(fmt: int, rows: np.ndarray) -> np.ndarray:
    """Stored rows [n, R] uint8 -> [n, 576] float64 (reading of the FP8 latent
    row: 512 E4M3 nope codes, four fp32 group scales, 64 bf16 rope dims)."""
    lib = _load()
    rows = np.ascontiguousarray(rows, dtype=np.uint8).reshape(-1, row_bytes(fmt))
    out = np.empty((rows.shape[0], LATENT), np.float64)
    for i in range(rows.shape[0]):
        lib.hso_dequant_row(fmt, ctypes.c_void_p(rows[i].ctypes.data),
                            ctypes.c_void_p(out[i].ctypes.data))
    return out


# --------------------------------------------------------------------------
# indexer + top-K  ("Ce qui se passe"; "Comment s'y prendre")
# --------------------------------------------------------------------------
def indexer_scores(idx_fmt: int, q: np.ndarray, w: np.ndarray, keys: np.ndarray,
                   sigma: np.ndarray, N: int) -> np.ndarray:
    """s[j][t] = sum_h w[j,h] * ReLU(sigma[t] * q[j,h,:].k[t,:]) for the tokens
    query j sees, -inf elsewhere.  q [nq,Hi,Di], w [nq,Hi] fp32, keys [>=N,Di],
    sigma [>=N] fp32; elements are fp32 or E4M3 bytes per idx_fmt."""
    nq, Hi, Di = q.shape
    dt = np.uint8 if idx_fmt == IDX_E4M3 else np.float32
    q = np.ascontiguousarray(q, dtype=dt)
    keys = np.ascontiguousarray(keys[:N], dtype=dt)
    w = np.ascontiguousarray(w, dtype=np.float32)
    sigma = np.ascontiguousarray(sigma[:N], dtype=np.float32)
    s = np.empty((nq, N), np.float32)
    _load().hso_indexer_scores(idx_fmt, _ptr(q), _ptr(w), _ptr(keys), _ptr(sigma),
                               N, nq, Hi, Di, _ptr(s))
    return s


def visible(N: int, nq: int, j: int) -> int:
    """Tokens query j of a step sees: [0, N - nq + j + 1) (reading: the cache
    already holds the step's nq tokens; each query sees up to itself)."""
    return N - nq + j + 1


def topk(s_row: np.ndarray, vis: int, K: int) -> np.ndarray:
    """K largest of s_row[:vis], ties to the lower index, ascending, -1 padded."""
    s_row = np.ascontiguousarray(s_row[:max(vis, 0)], dtype=np.float32)
    out = np.empty(K, np.int32)
    _load().hso_topk(_ptr(s_row) if vis > 0 else None, vis, K, _ptr(out))
    return out


# --------------------------------------------------------------------------
# residency reading  ("Les trois états de résidence")
# --------------------------------------------------------------------------
def page_resident(mode: int, N: int, T: int, P: int) -> np.ndarray:
    """Pages read in place on the GPU for a request of N tokens.
    full: every page; mixed: the tail window, i.e. pages p with
    (p+1)*P > N - T (whole pages, reading); zero: none."""
    npages = (N + P - 1) // P
    res = np.zeros(max(npages, 1), np.uint8)
    if mode == FULL:
        res[:npages] = 1
    elif mode == MIXED:
        first = max(N - T, 0) // P
        res[first:npages] = 1
    return res


class HotState:
    """Explicit LRU map of one request's hot buffer (C slots).

    hot_map[t] = slot or -1; slot_token[c] = token or -1; stamp[c] = step of
    last use (0 = never); step = last resolved step (steps count from 1)."""

    def __init__(self, C: int, max_tokens: int):
        self.C = C
        self.hot_map = np.full(max_tokens, -1, np.int32)
        self.slot_token = np.full(C, -1, np.int32)
        self.stamp = np.zeros(C, np.uint32)
        self.step = np.zeros(1, np.uint32)

    def copy(self) -> "HotState":
        h = HotState.__new__(HotState)
        h.C = self.C
        h.hot_map = self.hot_map.copy()
        h.slot_token = self.slot_token.copy()
        h.stamp = self.stamp.copy()
        h.step = self.step.copy()
        return h

    def resolve(self, resident: np.ndarray, P: int, N: int, idx: np.ndarray) -> dict:
        """Fused resolve of one request for one step (see hs_oracle.c)."""
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        nq, K = idx.shape
        resident = np.ascontiguousarray(resident, dtype=np.uint8)
        loc_kind = np.zeros((nq, K), np.int32)
        loc_val = np.zeros((nq, K), np.int32)
        miss_tok = np.zeros(nq * K + 1, np.int32)
        miss_slot = np.zeros(nq * K + 1, np.int32)
        n_miss = np.zeros(1, np.int32)
        counts = np.zeros(3, np.int32)
        st = _load().hso_resolve(_ptr(self.hot_map), _ptr(self.slot_token), _ptr(self.stamp),
                                 _ptr(self.step), self.C, _ptr(resident), P, N, _ptr(idx),
                                 nq, K, _ptr(loc_kind), _ptr(loc_val), _ptr(miss_tok),
                                 _ptr(miss_slot), _ptr(n_miss), _ptr(counts))
        m = int(n_miss[0])
        return dict(status=int(st), loc_kind=loc_kind, loc_val=loc_val,
                    miss_tok=miss_tok[:m].copy(), miss_slot=miss_slot[:m].copy(),
                    resident=int(counts[0]), hits=int(counts[1]), misses=int(counts[2]))


# --------------------------------------------------------------------------
# pool pressure  ("Ce qui se passe": the cache stays on the GPU while there is
# room and is offloaded only under real pressure; the pages give no policy,
# so the rule below is a reading)
# --------------------------------------------------------------------------
def gpu_blocks(mode: int, N: int, T: int, P: int, hot_pages: int) -> int:
    """GPU blocks a request of N tokens holds in `mode`: its resident pages
    (page_resident), plus its hot buffer of hot_pages blocks unless it is in
    full residency."""
    npages = (N + P - 1) // P
    return int(page_resident(mode, N, T, P)[:npages].sum()) + (0 if mode == FULL else hot_pages)


class PressurePolicy:
    """Block accounting of a device pool of `cap` blocks shared by requests,
    and the pressure reading.

    An append that would take the blocks in use past `cap` first flips to
    mixed residency the full-residency request with the most pages among
    those whose flip lowers its block count (lower id on ties), again and
    again until the append fits.  relieve() returns flipped requests to full
    residency, the last flipped first, while the free blocks cover the blocks
    the return adds plus one block per open request; it stops at the first
    that does not fit.  A request set by hand or closed leaves the policy."""

    def __init__(self, cap: int, T: int, P: int, hot_pages: int):
        self.cap, self.T, self.P, self.hot_pages = cap, T, P, hot_pages
        self.mode: dict[int, int] = {}
        self.N: dict[int, int] = {}
        self.flipped: list[int] = []

    def blocks(self, r: int, mode: int | None = None, N: int | None = None) -> int:
        return gpu_blocks(self.mode[r] if mode is None else mode, self.N[r] if N is None else N,
                          self.T, self.P, self.hot_pages)

    def used(self) -> int:
        return sum(self.blocks(r) for r in self.mode)

    def open(self, r: int, mode: int = FULL):
        self.mode[r], self.N[r] = mode, 0

    def close(self, r: int):
        del self.mode[r], self.N[r]
        if r in self.flipped:
            self.flipped.remove(r)

    def set_mode(self, r: int, mode: int):
        self.mode[r] = mode
        if r in self.flipped:
            self.flipped.remove(r)

    def append(self, r: int, n: int):
        """Returns (flipped ids in order, status)."""
        flips = []
        while self.used() - self.blocks(r) + self.blocks(r, N=self.N[r] + n) > self.cap:
            cands = [x for x in sorted(self.mode) if self.mode[x] == FULL
                     and self.blocks(x, MIXED) < self.blocks(x, FULL)]
            if not cands:
                return flips, ERR_CAPACITY
            most = max((self.N[x] + self.P - 1) // self.P for x in cands)
            x = min(x for x in cands if (self.N[x] + self.P - 1) // self.P == most)
            self.mode[x] = MIXED
            self.flipped.append(x)
            flips.append(x)
        self.N[r] += n
        return flips, OK

    def relieve(self) -> list[int]:
        back = []
        while self.flipped:
            x = self.flipped[-1]
            need = self.blocks(x, FULL) - self.blocks(x)
            if self.cap - self.used() < need + len(self.mode):
                break
            self.mode[x] = FULL
            self.flipped.pop()
            back.append(x)
        return back


# --------------------------------------------------------------------------
# sparse MLA attention  ("Ce qui se passe")
# --------------------------------------------------------------------------
def attention(fmt: int, q_bf16: np.ndarray, rows: np.ndarray, tau: float,
              mask: np.ndarray | None = None):
    """Dense-masked absorbed-MLA attention of one query over stored rows.
    q_bf16: [H,576] uint16 bf16 bits; rows: [n,R] uint8; mask: [n] (None =
    all rows in).  Returns (o [H,512] float64, lse [H] float64, natural log)."""
    q_bf16 = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    H = q_bf16.shape[0]
    rows = np.ascontiguousarray(rows, dtype=np.uint8).reshape(-1, row_bytes(fmt))
    n = rows.shape[0]
    o = np.empty((H, NOPE), np.float64)
    lse = np.empty(H, np.float64)
    m = None
    if mask is not None:
        m = np.ascontiguousarray(mask, dtype=np.uint8)
    _load().hso_attention(fmt, _ptr(q_bf16), H, _ptr(rows) if n else None,
                          _ptr(m) if m is not None else None, n, float(tau),
                          _ptr(o), _ptr(lse))
    return o, lse


def omp_threads() -> int:
    """Threads the oracle's OpenMP loops use (OMP_NUM_THREADS, else the CPU
    affinity set)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        return int(env)
    return len(os.sched_getaffinity(0))
