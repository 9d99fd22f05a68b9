"""Thin ctypes binding of libhs (include/hs.h), with the same names.

Argument marshalling only: every step of the decode path runs in the CUDA
library.  Importing this module raises ImportError when libhs.so has not been
built (``python -c "import __graft_entry__ as g; g.build()"``); there is no
fallback of any kind.

``Pool`` is a convenience owner of the two arenas (torch tensors: device
memory and pinned host memory) and of the opaque pool handle.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhs.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)

# ---- enums (include/hs.h) ----
HS_OK, HS_ERR_INVALID_ARG, HS_ERR_ARENA_TOO_SMALL, HS_ERR_CAPACITY = 0, 1, 2, 3
HS_ERR_HOST_POOL_FULL, HS_ERR_INDEX_RANGE, HS_ERR_TIMEOUT, HS_ERR_CUDA = 4, 5, 6, 7
HS_ERR_RANGE = 8
HS_ROW_E4M3_656, HS_ROW_F32_2304 = 0, 1
HS_IDX_E4M3, HS_IDX_F32 = 0, 1
HS_FULL, HS_MIXED, HS_ZERO = 0, 1, 2

_i32, _i64, _u32, _sz, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t, ctypes.c_void_p
_f32 = ctypes.c_float


class hs_pool_config(ctypes.Structure):
    _fields_ = [("max_requests", _i32), ("max_tokens", _i32), ("page_tokens", _i32),
                ("top_k", _i32), ("num_spec", _i32), ("tail_tokens", _i32),
                ("num_mla_layers", _i32), ("mla_heads", _i32), ("idx_heads", _i32),
                ("idx_dim", _i32), ("row_fmt", _i32), ("idx_fmt", _i32), ("hot_rows", _i32),
                ("reserved", _i32), ("gpu_blocks", _i64), ("host_blocks", _i64)]


class hs_stats(ctypes.Structure):
    _fields_ = [("resident", ctypes.c_uint64), ("hits", ctypes.c_uint64),
                ("misses", ctypes.c_uint64), ("bytes_copied", ctypes.c_uint64)]


class hs_layout(ctypes.Structure):
    _fields_ = [(n, _sz) for n in ("rows", "idx_keys", "idx_scale", "block_table",
                                   "host_block_table", "hot_map", "slot_token", "stamp",
                                   "hot_blocks", "seq_len", "req_step", "row_bytes",
                                   "max_pages", "hot_rows", "total")]


class hs_step_args(ctypes.Structure):
    _fields_ = [("B", _i32), ("nq", _i32), ("q_idx", _vp), ("w_idx", _vp), ("q_mla", _vp),
                ("softmax_scale", _f32), ("out", _vp), ("lse", _vp), ("topk", _vp),
                ("row_id", _vp), ("topk_in", _vp)]


def _decl(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_P = _vp
hs_pool_required_bytes = _decl("hs_pool_required_bytes", _i32,
                               [ctypes.POINTER(hs_pool_config), ctypes.POINTER(_sz), ctypes.POINTER(_sz)])
hs_pool_create = _decl("hs_pool_create", _i32,
                       [ctypes.POINTER(hs_pool_config), _P, _sz, _P, _sz, ctypes.POINTER(_P)])
hs_pool_destroy = _decl("hs_pool_destroy", None, [_P])
hs_pool_get_layout = _decl("hs_pool_get_layout", _i32, [_P, ctypes.POINTER(hs_layout)])
hs_pool_free_gpu_blocks = _decl("hs_pool_free_gpu_blocks", _i64, [_P])
hs_request_open = _decl("hs_request_open", _i32, [_P, _i32, _i32])
hs_append = _decl("hs_append", _i32, [_P, _i32, _P, _P, _P, _i32, _P])
hs_request_set_mode = _decl("hs_request_set_mode", _i32, [_P, _i32, _i32, _P])
hs_request_close = _decl("hs_request_close", _i32, [_P, _i32])
hs_precopy = _decl("hs_precopy", _i32, [_P, _P, _P])
hs_append_pressure = _decl("hs_append_pressure", _i32, [_P, _i32, _P, _P, _P, _i32, _P, _P, _P])
hs_pool_relieve = _decl("hs_pool_relieve", _i32, [_P, _P, _P, _P])
hs_indexer_score = _decl("hs_indexer_score", _i32, [_P, _P, _P, _i32, _i32, _P, _i64, _P])
hs_topk = _decl("hs_topk", _i32, [_P, _P, _i64, _i32, _i32, _P, _P])
hs_indexer_topk = _decl("hs_indexer_topk", _i32, [_P, _P, _P, _i32, _i32, _P, _P])
hs_resolve = _decl("hs_resolve", _i32, [_P, _P, _i32, _i32, _P, _P])
hs_resolve_plan = _decl("hs_resolve_plan", _i32, [_P, _P, _i32, _i32, _P, _P])
hs_miss_copy = _decl("hs_miss_copy", _i32, [_P, _i32, _i32, _P])
hs_miss_copy_layers = _decl("hs_miss_copy_layers", _i32, [_P, _i32, _i32, _i32, _i32, _i32, _P])
hs_pool_time_copies = _decl("hs_pool_time_copies", _i32, [_P, _i32])
hs_pool_copy_times = _decl("hs_pool_copy_times", _i32, [_P, ctypes.POINTER(ctypes.c_float), _i32])
hs_host_read_probe = _decl("hs_host_read_probe", _i32, [_P, _P, _sz, _i32, _P])
hs_sparse_mla_decode = _decl("hs_sparse_mla_decode", _i32,
                             [_P, _i32, _P, _P, _i32, _i32, _f32, _P, _P, _P])
hs_step = _decl("hs_step", _i32, [_P, ctypes.POINTER(hs_step_args), _P])
hs_resolve_attend = _decl("hs_resolve_attend", _i32,
                          [_P, _P, _i32, _i32, _P, _f32, _P, _P, _P, _P])
hs_pool_get_error = _decl("hs_pool_get_error", _i32, [_P, ctypes.POINTER(_i32)])
hs_pool_stats = _decl("hs_pool_stats", _i32, [_P, ctypes.POINTER(hs_stats)])
hs_pool_reset_stats = _decl("hs_pool_reset_stats", _i32, [_P])
hs_pool_dump_state = _decl("hs_pool_dump_state", _i32, [_P, _i32, _P, _P, _P, _P, _P, _P, _P, _P])
hs_pool_load_state = _decl("hs_pool_load_state", _i32, [_P, _i32, _P, _P, _P, _u32])
hs_topk_noalloc = _decl("hs_topk_noalloc", _i32, [_P, _i64, _P, _i32, _i32, _i32, _i32, _P, _P])
hs_check_wait_timeout = _decl("hs_check_wait_timeout", _i32, [_P, _i64, _P])
hs_dcp_topk_merge = _decl("hs_dcp_topk_merge", _i32, [_P, _P, _i64, _P, _P, _i32, _i32, _P, _P, _P])
hs_dcp_combine = _decl("hs_dcp_combine", _i32, [_P, _P, _i32, _i32, _i32, _P, _P, _P])
hs_step_kernel_count = _decl("hs_step_kernel_count", _i32, [_P, _i32, _i32])
hs_status_string = _decl("hs_status_string", ctypes.c_char_p, [_i32])
hs_abi_version = _decl("hs_abi_version", _i32, [])


class HSError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {hs_status_string(status).decode()} ({status})")


def check(status: int, what: str = "hs call") -> None:
    if status != HS_OK:
        raise HSError(status, what)


def host_read_probe(host_src, dev_dst, nbytes, ctas=0, stream=None):
    """Zero-copy read of pinned host memory into device memory (host-link probe)."""
    check(hs_host_read_probe(_ptr(host_src, "host_src"), _dev(dev_dst, "dev_dst"), nbytes, ctas,
                             _stream(stream)), "hs_host_read_probe")


def dcp_combine(o_parts, lse_parts, R, rows, H, out, lse=None, stream=None):
    check(hs_dcp_combine(_dev(o_parts, "o_parts"), _dev(lse_parts, "lse_parts"), R, rows, H,
                         _dev(out, "out"), _dev(lse, "lse"), _stream(stream)), "hs_dcp_combine")


def make_config(**kw) -> hs_pool_config:
    c = hs_pool_config()
    defaults = dict(page_tokens=64, num_spec=0, tail_tokens=0, num_mla_layers=1, hot_rows=0,
                    row_fmt=HS_ROW_E4M3_656, idx_fmt=HS_IDX_E4M3, host_blocks=0, reserved=0)
    defaults.update(kw)
    for k, v in defaults.items():
        setattr(c, k, int(v))
    return c


def required_bytes(cfg: hs_pool_config):
    d, h = _sz(), _sz()
    check(hs_pool_required_bytes(ctypes.byref(cfg), ctypes.byref(d), ctypes.byref(h)),
          "hs_pool_required_bytes")
    return d.value, h.value


def _ptr(t, what="argument"):
    """Pointer of a contiguous tensor in host or device memory (None -> NULL)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError(f"{what}: expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _dev(t, what="argument"):
    """Pointer of a contiguous CUDA tensor, for the header's "dev" arguments
    (None -> NULL): a host tensor here is rejected before anything runs."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what}: expected a CUDA tensor (a device pointer), got {t.device}")
    return _ptr(t, what)


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Pool:
    """Owns the arenas (torch device tensor + pinned host tensor) and the pool."""

    def __init__(self, cfg: hs_pool_config, device="cuda"):
        import torch
        self.cfg = cfg
        dev_bytes, host_bytes = required_bytes(cfg)
        self.dev_bytes, self.host_bytes = dev_bytes, host_bytes
        self.arena = torch.empty(dev_bytes, dtype=torch.uint8, device=device)
        self.host_arena = (torch.empty(host_bytes, dtype=torch.uint8, pin_memory=True)
                           if host_bytes else None)
        h = ctypes.c_void_p()
        check(hs_pool_create(ctypes.byref(cfg), _dev(self.arena, "arena"), dev_bytes,
                             _ptr(self.host_arena, "host arena"), host_bytes, ctypes.byref(h)),
              "hs_pool_create")
        self.handle = h
        lay = hs_layout()
        check(hs_pool_get_layout(self.handle, ctypes.byref(lay)), "hs_pool_get_layout")
        self.layout = lay
        self.R = int(lay.row_bytes)
        self.C = int(lay.hot_rows)
        self.max_pages = int(lay.max_pages)
        self.nq_max = cfg.num_spec + 1

    def close(self):
        if getattr(self, "handle", None):
            hs_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- lifecycle ----
    def open(self, req: int, mode: int):
        check(hs_request_open(self.handle, req, mode), "hs_request_open")

    def append(self, req: int, rows, keys, scale=None, stream=None):
        n = rows.shape[0]
        check(hs_append(self.handle, req, _ptr(rows, "rows"), _ptr(keys, "keys"),
                        _ptr(scale, "scale"), n, _stream(stream)), "hs_append")

    def set_mode(self, req: int, mode: int, stream=None):
        check(hs_request_set_mode(self.handle, req, mode, _stream(stream)), "hs_request_set_mode")

    def close_request(self, req: int):
        check(hs_request_close(self.handle, req), "hs_request_close")

    def precopy(self, stream=None) -> int:
        """Enqueue the host pre-copy of completed resident pages on `stream`;
        returns the number of pages enqueued (nothing is waited for)."""
        n = ctypes.c_int64()
        check(hs_precopy(self.handle, _stream(stream), ctypes.byref(n)), "hs_precopy")
        return n.value

    def append_pressure(self, req: int, rows, keys, scale=None, stream=None) -> list:
        """Append under the pressure policy; returns the requests it flipped."""
        n = rows.shape[0]
        ids = (_i32 * self.cfg.max_requests)()
        nf = _i32()
        check(hs_append_pressure(self.handle, req, _ptr(rows, "rows"), _ptr(keys, "keys"),
                                 _ptr(scale, "scale"), n, _stream(stream), ids, ctypes.byref(nf)),
              "hs_append_pressure")
        return list(ids[:nf.value])

    def relieve(self, stream=None) -> list:
        """Return policy-flipped requests to full residency while blocks allow;
        returns the requests restored."""
        ids = (_i32 * self.cfg.max_requests)()
        nr = _i32()
        check(hs_pool_relieve(self.handle, _stream(stream), ids, ctypes.byref(nr)),
              "hs_pool_relieve")
        return list(ids[:nr.value])

    def free_gpu_blocks(self) -> int:
        return int(hs_pool_free_gpu_blocks(self.handle))

    # ---- decode-step calls ----
    def indexer_score(self, q, w, B, nq, scores, stride, stream=None):
        check(hs_indexer_score(self.handle, _dev(q, "q"), _dev(w, "w"), B, nq,
                               _dev(scores, "scores"), stride, _stream(stream)), "hs_indexer_score")

    def topk(self, scores, stride, B, nq, out, stream=None):
        check(hs_topk(self.handle, _dev(scores, "scores"), stride, B, nq, _dev(out, "out"),
                      _stream(stream)), "hs_topk")

    def indexer_topk(self, q, w, B, nq, out, stream=None):
        check(hs_indexer_topk(self.handle, _dev(q, "q"), _dev(w, "w"), B, nq, _dev(out, "out"),
                              _stream(stream)), "hs_indexer_topk")

    def resolve(self, topk, B, nq, row_id, stream=None):
        check(hs_resolve(self.handle, _dev(topk, "topk"), B, nq, _dev(row_id, "row_id"),
                         _stream(stream)), "hs_resolve")

    def resolve_plan(self, topk, B, nq, row_id, stream=None):
        check(hs_resolve_plan(self.handle, _dev(topk, "topk"), B, nq, _dev(row_id, "row_id"),
                              _stream(stream)), "hs_resolve_plan")

    def miss_copy(self, B, nq, stream=None):
        check(hs_miss_copy(self.handle, B, nq, _stream(stream)), "hs_miss_copy")

    def time_copies(self, enable=True):
        check(hs_pool_time_copies(self.handle, 1 if enable else 0), "hs_pool_time_copies")

    def copy_times(self, n=None):
        """Per-layer durations (ms) of the last recorded step's side-stream copies."""
        n = self.cfg.num_mla_layers if n is None else n
        buf = (ctypes.c_float * max(n, 1))()
        check(hs_pool_copy_times(self.handle, buf, n), "hs_pool_copy_times")
        return [buf[i] for i in range(n)]

    def miss_copy_layers(self, B, nq, layer_begin, layer_end, ctas=0, stream=None):
        check(hs_miss_copy_layers(self.handle, B, nq, layer_begin, layer_end, ctas, _stream(stream)),
              "hs_miss_copy_layers")

    def sparse_mla_decode(self, layer, q, row_id, B, nq, scale, out, lse=None, stream=None):
        check(hs_sparse_mla_decode(self.handle, layer, _dev(q, "q"), _dev(row_id, "row_id"), B, nq,
                                   scale, _dev(out, "out"), _dev(lse, "lse"), _stream(stream)),
              "hs_sparse_mla_decode")

    def dcp_topk_merge(self, scores, stride, local_topk, offsets, R, rows, topk, part_topk,
                       stream=None):
        check(hs_dcp_topk_merge(self.handle, _dev(scores, "scores"), stride,
                                _dev(local_topk, "local_topk"), _dev(offsets, "offsets"), R, rows,
                                _dev(topk, "topk"), _dev(part_topk, "part_topk"), _stream(stream)),
              "hs_dcp_topk_merge")

    def check_wait_timeout(self, limit_cycles, stream=None):
        check(hs_check_wait_timeout(self.handle, limit_cycles, _stream(stream)),
              "hs_check_wait_timeout")

    def step(self, B, nq, q_idx, w_idx, q_mla, scale, out, topk, row_id, lse=None, stream=None,
             topk_in=None):
        a = hs_step_args(B=B, nq=nq, q_idx=_dev(q_idx, "q_idx"), w_idx=_dev(w_idx, "w_idx"),
                         q_mla=_dev(q_mla, "q_mla"), softmax_scale=scale, out=_dev(out, "out"),
                         lse=_dev(lse, "lse"), topk=_dev(topk, "topk"), row_id=_dev(row_id, "row_id"),
                         topk_in=_dev(topk_in, "topk_in"))
        check(hs_step(self.handle, ctypes.byref(a), _stream(stream)), "hs_step")

    def resolve_attend(self, topk, B, nq, q_mla, scale, out, row_id, lse=None, stream=None):
        check(hs_resolve_attend(self.handle, _dev(topk, "topk"), B, nq, _dev(q_mla, "q_mla"), scale,
                                _dev(out, "out"), _dev(lse, "lse"), _dev(row_id, "row_id"),
                                _stream(stream)), "hs_resolve_attend")

    def step_kernel_count(self, B, nq) -> int:
        return int(hs_step_kernel_count(self.handle, B, nq))

    # ---- introspection ----
    def get_error(self) -> int:
        v = _i32()
        check(hs_pool_get_error(self.handle, ctypes.byref(v)), "hs_pool_get_error")
        return v.value

    def stats(self) -> dict:
        s = hs_stats()
        check(hs_pool_stats(self.handle, ctypes.byref(s)), "hs_pool_stats")
        return dict(resident=s.resident, hits=s.hits, misses=s.misses, bytes_copied=s.bytes_copied)

    def reset_stats(self):
        check(hs_pool_reset_stats(self.handle), "hs_pool_reset_stats")

    def dump_state(self, req: int) -> dict:
        import numpy as np
        c = self.cfg
        out = dict(hot_map=np.empty(c.max_tokens, np.int32), slot_token=np.empty(self.C, np.int32),
                   stamp=np.empty(self.C, np.uint32), block_table=np.empty(self.max_pages, np.int32),
                   host_block_table=np.empty(self.max_pages, np.int32),
                   hot_blocks=np.empty(self.C // c.page_tokens, np.int32),
                   step=np.empty(1, np.uint32), seq_len=np.empty(1, np.int32))
        ptrs = [ctypes.c_void_p(out[k].ctypes.data) for k in
                ("hot_map", "slot_token", "stamp", "block_table", "host_block_table", "hot_blocks",
                 "step", "seq_len")]
        check(hs_pool_dump_state(self.handle, req, *ptrs), "hs_pool_dump_state")
        return out

    def load_state(self, req, hot_map, slot_token, stamp, step):
        import numpy as np
        hm = np.ascontiguousarray(hot_map, np.int32)
        st = np.ascontiguousarray(slot_token, np.int32)
        sp = np.ascontiguousarray(stamp, np.uint32)
        check(hs_pool_load_state(self.handle, req, ctypes.c_void_p(hm.ctypes.data),
                                 ctypes.c_void_p(st.ctypes.data), ctypes.c_void_p(sp.ctypes.data),
                                 int(step)), "hs_pool_load_state")

    # ---- views of pool memory (for tests) ----
    def rows_view(self):
        """The device block pool as [gpu_blocks, L, P, R] uint8."""
        c, L = self.cfg, self.cfg.num_mla_layers
        n = c.gpu_blocks * L * c.page_tokens * self.R
        return self.arena[self.layout.rows:self.layout.rows + n].view(
            c.gpu_blocks, L, c.page_tokens, self.R)

    def host_rows_view(self):
        c, L = self.cfg, self.cfg.num_mla_layers
        if self.host_arena is None:
            return None
        return self.host_arena.view(c.host_blocks, L, c.page_tokens, self.R)
