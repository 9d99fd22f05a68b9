"""Helpers for the full-size GPU parity tests: vectorised row-location
translation and stream generation in a spawn pool (started before any CUDA
work in the worker processes; the workers never touch CUDA)."""
from __future__ import annotations

import numpy as np


def locate(rid: np.ndarray, block_table: np.ndarray, hot_blocks: np.ndarray, P: int,
           nblocks: int):
    """Pool row ids -> (kind, value): 1 = resident token, 2 = hot slot,
    0 = padding, 9 = a row that belongs to neither."""
    page_of = np.full(nblocks, -1, np.int64)
    sel = block_table >= 0
    page_of[block_table[sel]] = np.nonzero(sel)[0]
    hot_of = np.full(nblocks, -1, np.int64)
    selh = hot_blocks >= 0
    hot_of[hot_blocks[selh]] = np.nonzero(selh)[0]
    valid = rid >= 0
    blk = np.where(valid, rid // P, 0)
    off = np.where(valid, rid % P, 0)
    pg, hp = page_of[blk], hot_of[blk]
    kind = np.where(~valid, 0, np.where(pg >= 0, 1, np.where(hp >= 0, 2, 9)))
    val = np.where(kind == 1, pg * P + off, np.where(kind == 2, hp * P + off, -1))
    return kind.astype(np.int32), val.astype(np.int32)


def drawn_streams(seed, B, steps, nq, N, K, P, kind, T=0, procs=None):
    """[len(steps)][B][nq][K] drawn top-K lists, generated in parallel."""
    from sparse_mla_kv_fp8_gb300 import workload as wl
    return wl.drawn_streams(seed, B, steps, nq, N, K, P, kind, T, procs)
