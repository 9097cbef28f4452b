"""The C ABI library builds for sm_103a, loads, and exports every entry point
that include/la.h declares (no GPU needed; no compute calls)."""
import ctypes
import os
import re

from conftest import ROOT
from helpers import ensure_built


def declared_entry_points():
    with open(os.path.join(ROOT, "include", "la.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for n in ("la_create", "la_prefill", "la_step", "la_generate", "la_destroy", "la_stats",
              "la_export_state", "la_import_state", "la_debug_logits", "la_gemm_bf16", "la_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol():
    ensure_built()
    from exact_decoding_gb300 import LIB_PATH, load_library
    lib = load_library()
    for name in declared_entry_points():
        assert hasattr(lib, name), name
    raw = ctypes.CDLL(LIB_PATH)
    assert raw.la_strerror  # plain dlsym works too


def test_error_strings_without_gpu():
    ensure_built()
    from exact_decoding_gb300 import la_strerror
    assert la_strerror(0) == "ok"
    assert la_strerror(-3) == "capacity exceeded"
    assert la_strerror(-5) == "device wait timed out"


def test_create_rejects_bad_options_without_touching_the_gpu():
    """Argument validation happens on the host before any CUDA call."""
    ensure_built()
    import exact_decoding_gb300.la as L
    lib = L.load_library()
    d = L.la_model_dims(2, 256, 4, 4, 96, 688, 1024, 1e-5, 1e4, L.LA_F32)   # head_dim 96: unsupported
    w = L.la_weights()
    o = L.la_opts(3, 4, 4, 256, 0, 0, 0.0, 0, None, 0)
    h = ctypes.c_void_p()
    assert lib.la_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(o), ctypes.byref(h)) == -7
    d.head_dim = 64
    assert lib.la_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(o), ctypes.byref(h)) == -1  # null weights
    p = ctypes.c_void_p(16)
    arr = (ctypes.c_void_p * 2)(16, 16)
    pp = ctypes.cast(arr, L._PP)
    w = L.la_weights(p, p, p, pp, pp, pp, pp, pp, pp, pp, pp, pp)
    o.N = 1
    assert lib.la_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(o), ctypes.byref(h)) == -1
    o.N, o.G = 3, 40
    assert lib.la_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(o), ctypes.byref(h)) == -1
    assert b"G 0..32" in lib.la_last_error()
    o.G, o.pool_policy = 4, 3
    assert lib.la_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(o), ctypes.byref(h)) == -1
    assert b"pool_policy" in lib.la_last_error()
