"""Host-side checks of the C ABI that need no GPU: the library builds for sm_103a,
loads, exports every entry point include/kv4.h declares, and rejects bad
arguments before touching the device."""
import ctypes as C
import os
import re

import pytest

from int8_hybrid_paged_gb300 import build as kbuild
from int8_hybrid_paged_gb300 import kv4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kv4.load()


def declared_entry_points():
    text = open(os.path.join(ROOT, "include", "kv4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv4_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert "kv4_decode_attention" in names and "kv4_append" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(kv4.EXPORTED)


def test_status_strings(lib):
    for code in range(0, -7, -1):
        assert kv4.kv4_status_string(code) != "unknown status"
    assert kv4.kv4_status_string(-99) == "unknown status"


def _cfg(**kw):
    base = dict(num_kv_heads=8, head_dim=128, page_size=16, sink=16, window=128, num_pages=64,
                max_slots=4, max_batch=4, max_q_heads=32, max_work_items=0, format=0)
    base.update(kw)
    return kv4.kv4_cache_config(*[base[f] for f, _ in kv4.kv4_cache_config._fields_])


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), -2),
    (dict(page_size=32), -2),
    (dict(sink=200, window=100), -2),
    (dict(sink=5, window=128), -2),      # protected weights per page: s, w multiples of 16
    (dict(sink=16, window=40), -2),
    (dict(max_q_heads=36), -1),          # not a multiple of H_kv
    (dict(max_q_heads=64), -2),          # group of 8
    (dict(num_kv_heads=0), -1),
    (dict(num_pages=0), -1),
    (dict(sink=-1), -1),
    (dict(format=4), -1),                # unknown cache format
    (dict(format=-1), -1),               # unknown cache format
    (dict(format=2), -1),                # NVFP4 has no protected region
    (dict(format=3), -1),                # MXFP4 has no protected region
    (dict(format=1), -1),                # the 8-bit format has no protected region
    (dict(format=1, sink=0, window=4), -1),
])
def test_create_rejects_bad_configs_before_the_device(lib, kw, status):
    h = C.c_void_p()
    cfg = _cfg(**kw)
    assert lib.kv4_cache_create(C.byref(cfg), C.byref(h)) == status
    assert not h.value


def test_null_handles_are_rejected(lib):
    assert lib.kv4_cache_create(None, None) == -1
    assert lib.kv4_cache_free(None) == 0
    assert lib.kv4_append(None, None, None, None, None, None, None, 1, 1, 1, None) == -1
    assert lib.kv4_decode_attention(None, None, 32, None, None, None, 1, 1, 0.1, None, None,
                                    None) == -1
    assert lib.kv4_get_device_error(None, None, 0) == -1
