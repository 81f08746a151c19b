"""The C-ABI library loads and exports every entry point include/dattn.h
declares; its host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    text = open(os.path.join(ROOT, "include", "dattn.h")).read()
    return sorted(set(re.findall(r"DATTN_API\s+[\w\s\*]+?\b(dattn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for n in ("dattn_create", "dattn_append_kv", "dattn_decode", "dattn_verify", "dattn_destroy",
              "dattn_get_error", "dattn_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import decode_attention_kv_dattn_gb300 as d
    lib = ctypes.CDLL(d.LIB_PATH)
    for n in declared_entry_points():
        assert hasattr(lib, n), f"{n} declared in dattn.h but not exported"
    assert set(d.EXPORTS) == set(declared_entry_points())


def test_error_strings_and_null_arguments():
    import decode_attention_kv_dattn_gb300 as d
    assert d.error_string(d.OK) == "ok"
    assert "exceeds" in d.error_string(d.EXCEEDS)
    # rejected before any CUDA call
    assert d.lib.dattn_create(None, 0, None) == d.EINVAL
    cfg = d.Config(8, 3, 256, 1, 0, 0, 0, None)  # 8 % 3 != 0
    h = ctypes.c_void_p()
    assert d.lib.dattn_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == d.EINVAL
    assert d.lib.dattn_decode(None, 0, None, None, None) == d.EINVAL
    assert d.lib.dattn_get_error(None, None) == d.EINVAL
    d.lib.dattn_destroy(None)
