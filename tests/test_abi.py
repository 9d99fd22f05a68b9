"""The C-ABI library loads and exports every symbol include/hs.h declares;
host-only entry points (no GPU work) behave as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def hs():
    from sparse_mla_kv_fp8_gb300 import build
    build.build()
    from sparse_mla_kv_fp8_gb300 import hs as mod
    return mod


def _declared_functions():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(hs_\w+)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_every_declared_symbol_is_exported(hs):
    names = _declared_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(hs.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(hs):
    assert hs.hs_abi_version() >= 100
    for s in range(9):
        assert b"unknown" not in hs.hs_status_string(s)
    assert b"unknown" in hs.hs_status_string(99)


def _cfg(hs, **kw):
    base = dict(max_requests=4, max_tokens=4096, top_k=256, num_spec=0, tail_tokens=512,
                num_mla_layers=1, mla_heads=16, idx_heads=4, idx_dim=32, gpu_blocks=100,
                host_blocks=100)
    base.update(kw)
    return hs.make_config(**base)


def test_required_bytes_is_host_arithmetic(hs):
    d, h = hs.required_bytes(_cfg(hs))
    assert d > 0 and h == 100 * 1 * 64 * 656
    d2, _ = hs.required_bytes(_cfg(hs, gpu_blocks=200))
    assert d2 - d >= 100 * 64 * 656  # the block pool grows by the extra blocks
    _, h3 = hs.required_bytes(_cfg(hs, row_fmt=hs.HS_ROW_F32_2304))
    assert h3 == 100 * 64 * 2304


@pytest.mark.parametrize("bad", [
    dict(max_requests=0), dict(top_k=0), dict(page_tokens=0), dict(mla_heads=12),
    dict(hot_rows=100),                 # not a multiple of the page
    dict(hot_rows=128),                 # below top_k
    dict(num_spec=3, top_k=4096),       # union too large for one CTA
    dict(idx_dim=20),                   # E4M3 keys need 16-byte rows
    dict(row_fmt=7), dict(idx_fmt=9), dict(gpu_blocks=-1),
    dict(gpu_blocks=1 << 25),           # 2^31 device rows: ids are int32
    dict(gpu_blocks=(1 << 24) + 1, num_mla_layers=256),  # > 2^32 row units
])
def test_required_bytes_rejects_bad_configs(hs, bad):
    c = _cfg(hs, **bad)
    d, h = ctypes.c_size_t(), ctypes.c_size_t()
    assert hs.hs_pool_required_bytes(ctypes.byref(c), ctypes.byref(d), ctypes.byref(h)) == hs.HS_ERR_INVALID_ARG


def test_hot_rows_default_follows_capacity_rule(hs):
    """Default hot buffer = (num_spec + 2) * top_k rows ("Ce qu'il faut en
    retenir"): 2K without MTP, 5K with MTP3."""
    for ns, mult in ((0, 2), (3, 5)):
        c = _cfg(hs, num_spec=ns, top_k=256)
        d_default, _ = hs.required_bytes(c)
        c2 = _cfg(hs, num_spec=ns, top_k=256, hot_rows=mult * 256)
        d_explicit, _ = hs.required_bytes(c2)
        assert d_default == d_explicit


def test_create_rejects_small_arena_without_gpu(hs):
    c = _cfg(hs)
    h = ctypes.c_void_p()
    # arena-size and argument checks happen before any CUDA call
    assert hs.hs_pool_create(ctypes.byref(c), ctypes.c_void_p(16), 10, None, 0,
                             ctypes.byref(h)) == hs.HS_ERR_ARENA_TOO_SMALL
    assert hs.hs_pool_create(ctypes.byref(c), None, 1 << 40, None, 1 << 40,
                             ctypes.byref(h)) == hs.HS_ERR_INVALID_ARG
    assert hs.hs_pool_create(None, None, 0, None, 0, ctypes.byref(h)) == hs.HS_ERR_INVALID_ARG


def test_null_pool_calls_are_rejected(hs):
    assert hs.hs_request_open(None, 0, 0) == hs.HS_ERR_INVALID_ARG
    assert hs.hs_resolve(None, None, 1, 1, None, None) == hs.HS_ERR_INVALID_ARG
    assert hs.hs_step(None, None, None) == hs.HS_ERR_INVALID_ARG
    assert hs.hs_pool_free_gpu_blocks(None) == -1


def test_binding_rejects_host_and_strided_tensors_for_device_arguments(hs):
    """The binding's marshalling: a "dev" argument must be a contiguous CUDA
    tensor, checked before any call reaches the library (no GPU needed: a CPU
    tensor is refused outright)."""
    import torch
    with pytest.raises(ValueError, match="CUDA tensor"):
        hs._dev(torch.zeros(4), "q")
    with pytest.raises(ValueError, match="contiguous"):
        hs._ptr(torch.zeros(4, 4).t(), "rows")
    assert hs._dev(None) is None and hs._ptr(None) is None
    t = torch.zeros(8)
    assert hs._ptr(t).value == t.data_ptr()
