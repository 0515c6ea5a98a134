"""Host-side checks of the C ABI that need no GPU: exports, validation, status codes, fault injection."""

import ctypes
import os
import re

import pytest

from bit_kv_cache_write_gb300 import oscar as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            names += re.findall(r"OSCAR_API\s+[\w\s\*]+?\b(oscar_\w+)\s*\(", text)
    return names


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    for n in ("oscar_create", "oscar_destroy", "oscar_calibrate_upload", "oscar_write_tokens",
              "oscar_demote_recent", "oscar_decode", "oscar_decode_workspace_size"):
        assert n in names


def test_library_loads_and_exports_every_declared_symbol(liboscar):
    for name in declared_symbols():
        assert hasattr(liboscar, name), name
        assert ctypes.cast(getattr(liboscar, name), ctypes.c_void_p).value


def test_status_strings(liboscar):
    for st in range(-7, 1):
        assert O.oscar_status_string(st) not in ("", "unknown status")
    assert O.oscar_status_string(-99) == "unknown status"


def _cfg(**over):
    c = dict(n_layers=1, n_q_heads=4, n_kv_heads=2, head_dim=64, group=32, page_size=16, sink=64, recent=256,
             sm_scale=0.0, debug_bounds=0)
    c.update(over)
    return O.oscar_config_t(**c)


@pytest.mark.parametrize("over,status", [
    (dict(head_dim=96), -2), (dict(group=16), -2), (dict(group=128, head_dim=64), -2),
    (dict(page_size=32), -2), (dict(n_q_heads=6, n_kv_heads=4), -2), (dict(n_q_heads=32, n_kv_heads=2), -2),
    (dict(sink=400, recent=256), -2), (dict(n_layers=0), -1), (dict(n_kv_heads=0), -1),
])
def test_create_rejects_bad_config_before_touching_the_device(liboscar, over, status):
    ctx = ctypes.c_void_p()
    st = liboscar.oscar_create(ctypes.byref(_cfg(**over)), ctypes.byref(ctx))
    assert st == status
    assert ctx.value is None
    assert O.oscar_last_error()


def test_null_arguments(liboscar):
    assert liboscar.oscar_create(None, None) == -1
    assert liboscar.oscar_write_tokens(None, 0, None, None, None, 0, None, 0, None) == -1
    assert liboscar.oscar_demote_recent(None, 0, None, 0, None, None, 0, None, 0, None) == -1
    assert liboscar.oscar_calibrate_upload(None, 0, None, None, None, None, None) == -1
    assert liboscar.oscar_decode(None, 0, None, None, 0, None, 0, None, 0, None, 0, None, 0, None,
                                 None, None, 0, 1, None) == -1
    assert liboscar.oscar_decode_workspace_size(None, 1, 100) == 0
    assert liboscar.oscar_int2_page_bytes(None) == 0
    assert liboscar.oscar_debug_error(None, None, None) == -1
    liboscar.oscar_destroy(None)


def test_injected_allocation_failure(liboscar, monkeypatch):
    monkeypatch.setenv("OSCAR_FAULT", "alloc")
    ctx = ctypes.c_void_p()
    assert liboscar.oscar_create(ctypes.byref(_cfg()), ctypes.byref(ctx)) == -6
    assert "injected" in O.oscar_last_error()


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(O, "_lib", None)
    monkeypatch.setattr(O, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="liboscar.so not found"):
        O.lib()


def test_valid_config_without_a_gpu_reports_a_cuda_error(liboscar):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    ctx = ctypes.c_void_p()
    assert liboscar.oscar_create(ctypes.byref(_cfg()), ctypes.byref(ctx)) == -4
    assert ctx.value is None
