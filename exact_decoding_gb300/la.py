"""ctypes binding of include/la.h (argument marshalling only).

Each `la_*` function here calls the C entry point of the same name; errors
become `LaError`.  `Decoder` is a convenience owner: it uploads a weight dict
(from `synth`) to the device with torch and keeps those tensors alive for the
handle's lifetime.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libla.so")

LA_F32, LA_BF16 = 0, 1
LA_POOL_FIFO, LA_POOL_LRU, LA_POOL_LFU = 0, 1, 2
_lib = None


class LaError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where}: {msg} (code {code})")
        self.code = code


class la_model_dims(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_base", ctypes.c_float),
                ("dtype", ctypes.c_int32)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class la_weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("attn_norm", _PP), ("wq", _PP), ("wk", _PP), ("wv", _PP), ("wo", _PP), ("ffn_norm", _PP),
                ("w_gate", _PP), ("w_up", _PP), ("w_down", _PP)]


class la_opts(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int32), ("W", ctypes.c_int32), ("G", ctypes.c_int32), ("max_seq", ctypes.c_int32),
                ("prompt_as_reference", ctypes.c_int32), ("pool_cap", ctypes.c_int32),
                ("temperature", ctypes.c_float), ("seed", ctypes.c_uint64), ("cuda_stream", ctypes.c_void_p),
                ("profile", ctypes.c_int32), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float),
                ("pool_policy", ctypes.c_int32)]


class la_stats_t(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("generated", ctypes.c_int64), ("last_accept", ctypes.c_int32),
                ("last_candidates", ctypes.c_int32), ("prefix_len", ctypes.c_int32), ("rows", ctypes.c_int32),
                ("gemm_ms", ctypes.c_double), ("gemm_bytes", ctypes.c_double), ("gemm_launches", ctypes.c_int64),
                ("attn_ms", ctypes.c_double), ("attn_bytes", ctypes.c_double), ("attn_launches", ctypes.c_int64),
                ("kernel_launches", ctypes.c_int64), ("elem_ms", ctypes.c_double), ("spec_ms", ctypes.c_double),
                ("h2d_bytes", ctypes.c_int64), ("d2h_bytes", ctypes.c_int64)]


_I32P = ctypes.POINTER(ctypes.c_int32)
LA_ERR_CAPACITY = -3   # include/la.h


class la_state_t(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int32), ("tokens_cap", ctypes.c_int32), ("tokens", _I32P),
                ("window", _I32P), ("n_records", ctypes.c_int32), ("records_cap", ctypes.c_int32),
                ("records", _I32P), ("uses", _I32P)]


def load_library():
    """Load libla.so; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m exact_decoding_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    H = ctypes.c_void_p
    lib.la_create.argtypes = [ctypes.POINTER(la_model_dims), ctypes.POINTER(la_weights), ctypes.POINTER(la_opts),
                              ctypes.POINTER(H)]
    lib.la_prefill.argtypes = [H, _I32P, ctypes.c_int32, _I32P]
    lib.la_step.argtypes = [H, _I32P, _I32P]
    lib.la_ar_step.argtypes = [H, _I32P]
    lib.la_generate.argtypes = [H, _I32P, ctypes.c_int32, ctypes.c_int32, _I32P, _I32P, _I32P]
    lib.la_stats.argtypes = [H, ctypes.POINTER(la_stats_t)]
    lib.la_export_state.argtypes = [H, ctypes.POINTER(la_state_t)]
    lib.la_import_state.argtypes = [H, ctypes.POINTER(la_state_t)]
    lib.la_debug_logits.argtypes = [H, ctypes.c_void_p, _I32P, _I32P]
    lib.la_gemm_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    lib.la_gemm_bf16_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
    lib.la_gemm_status.argtypes = [ctypes.c_void_p]
    lib.la_selftest_timeout.argtypes = [H, ctypes.c_int64, ctypes.c_void_p]
    lib.la_step_tables.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _I32P,
                                   ctypes.POINTER(ctypes.c_uint32), _I32P, ctypes.c_int32, _I32P, _I32P]
    lib.la_gemm_schedule.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _I32P,
                                     ctypes.c_int32, _I32P, _I32P, _I32P, _I32P]
    lib.la_destroy.argtypes = [H]
    lib.la_destroy.restype = None
    lib.la_strerror.argtypes = [ctypes.c_int]
    lib.la_strerror.restype = ctypes.c_char_p
    lib.la_last_error.argtypes = []
    lib.la_last_error.restype = ctypes.c_char_p
    for name in ("la_create", "la_prefill", "la_step", "la_ar_step", "la_generate", "la_stats", "la_export_state",
                 "la_import_state", "la_debug_logits", "la_gemm_bf16", "la_gemm_bf16_noalloc", "la_gemm_status",
                 "la_selftest_timeout", "la_gemm_schedule", "la_step_tables"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def la_strerror(code: int) -> str:
    return load_library().la_strerror(code).decode()


def _check(rc: int, where: str):
    if rc != 0:
        lib = load_library()
        raise LaError(rc, where, lib.la_last_error().decode() or lib.la_strerror(rc).decode())


def _i32(a: np.ndarray):
    return a.ctypes.data_as(_I32P)


# ---------------------------------------------------------------------------- entry points
def la_create(dims: la_model_dims, weights: la_weights, opts: la_opts) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(load_library().la_create(ctypes.byref(dims), ctypes.byref(weights), ctypes.byref(opts),
                                    ctypes.byref(h)), "la_create")
    return h


def la_prefill(h, prompt) -> int:
    p = np.ascontiguousarray(prompt, dtype=np.int32)
    first = np.zeros(1, dtype=np.int32)
    _check(load_library().la_prefill(h, _i32(p), len(p), _i32(first)), "la_prefill")
    return int(first[0])


def la_step(h, N: int) -> List[int]:
    out = np.zeros(max(N, 8), dtype=np.int32)
    n = np.zeros(1, dtype=np.int32)
    _check(load_library().la_step(h, _i32(out), _i32(n)), "la_step")
    return out[: int(n[0])].tolist()


def la_ar_step(h) -> int:
    tok = np.zeros(1, dtype=np.int32)
    _check(load_library().la_ar_step(h, _i32(tok)), "la_ar_step")
    return int(tok[0])


def la_generate(h, prompt, max_new: int) -> Tuple[List[int], int]:
    p = np.ascontiguousarray(prompt, dtype=np.int32)
    out = np.zeros(max_new, dtype=np.int32)
    n = np.zeros(1, dtype=np.int32)
    steps = np.zeros(1, dtype=np.int32)
    _check(load_library().la_generate(h, _i32(p), len(p), max_new, _i32(out), _i32(n), _i32(steps)),
           "la_generate")
    return out[: int(n[0])].tolist(), int(steps[0])


def la_stats(h) -> dict:
    s = la_stats_t()
    _check(load_library().la_stats(h, ctypes.byref(s)), "la_stats")
    return {f: getattr(s, f) for f, _ in la_stats_t._fields_}


def la_export_state(h, N: int, W: int, tokens_cap: int = 1 << 16, records_cap: int = 1 << 16) -> dict:
    toks = np.zeros(tokens_cap, dtype=np.int32)
    win = np.zeros((N - 1) * W, dtype=np.int32)
    recs = np.zeros(records_cap * N, dtype=np.int32)
    uses = np.zeros(records_cap, dtype=np.int32)
    st = la_state_t(0, tokens_cap, _i32(toks), _i32(win), 0, records_cap, _i32(recs), _i32(uses))
    _check(load_library().la_export_state(h, ctypes.byref(st)), "la_export_state")
    r = recs[: st.n_records * N].reshape(st.n_records, N)
    return {"tokens": toks[: st.n_tokens].tolist(), "window": win.reshape(N - 1, W).copy(),
            "records": [(int(x[0]), tuple(int(t) for t in x[1:])) for x in r],
            "uses": uses[: st.n_records].tolist()}


def la_import_state(h, N: int, W: int, tokens, window, records, uses=None) -> None:
    toks = np.ascontiguousarray(tokens, dtype=np.int32)
    win = np.ascontiguousarray(np.asarray(window).reshape(-1), dtype=np.int32)
    recs = np.ascontiguousarray(np.array([[k, *s] for k, s in records], dtype=np.int32).reshape(-1, N))
    u = None if uses is None else np.ascontiguousarray(uses, dtype=np.int32)
    st = la_state_t(len(toks), len(toks), _i32(toks), _i32(win), len(recs), len(recs), _i32(recs),
                    _i32(u) if u is not None else None)
    _check(load_library().la_import_state(h, ctypes.byref(st)), "la_import_state")


def la_debug_logits(h) -> np.ndarray:
    rows = np.zeros(1, dtype=np.int32)
    vocab = np.zeros(1, dtype=np.int32)
    lib = load_library()
    _check(lib.la_debug_logits(h, None, _i32(rows), _i32(vocab)), "la_debug_logits")
    out = np.zeros((int(rows[0]), int(vocab[0])), dtype=np.float32)
    _check(lib.la_debug_logits(h, out.ctypes.data, _i32(rows), _i32(vocab)), "la_debug_logits")
    return out


def la_gemm_bf16(x_ptr: int, w_ptr: int, y_ptr: int, rows: int, out: int, k: int, splits: int = 1,
                 workspace_ptr: Optional[int] = None, stream: Optional[int] = None) -> None:
    _check(load_library().la_gemm_bf16(x_ptr, w_ptr, y_ptr, rows, out, k, splits, workspace_ptr, stream),
           "la_gemm_bf16")


def la_gemm_bf16_noalloc(x_ptr: int, w_ptr: int, y_ptr: int, rows: int, out: int, k: int, splits: int = 1,
                         stream: Optional[int] = None) -> None:
    """la_gemm_bf16 without a caller workspace: for callers that cannot allocate
    device memory at call time.  The split-K partials live in a fixed device
    array inside the library (LA_NOALLOC_SCRATCH_FLOATS floats); overlapping
    calls race on it."""
    _check(load_library().la_gemm_bf16_noalloc(x_ptr, w_ptr, y_ptr, rows, out, k, splits, stream),
           "la_gemm_bf16_noalloc")


NOALLOC_SCRATCH_FLOATS = 4 * 1024 * 1024


def la_gemm_status(stream: Optional[int] = None) -> None:
    """Raise LaError(-5) if a bounded wait inside an earlier la_gemm_bf16 /
    la_gemm_bf16_noalloc kernel on this device gave up; clears the status."""
    _check(load_library().la_gemm_status(stream), "la_gemm_status")


def la_selftest_timeout(h, limit_ns: int, stream: Optional[int] = None) -> None:
    """Launch the bounded-wait self-test kernel (its wait gives up after
    limit_ns and sets a timeout bit in h's error word, or with h None in the
    standalone GEMMs' words)."""
    _check(load_library().la_selftest_timeout(h, limit_ns, stream), "la_selftest_timeout")


def la_step_tables(N: int, W: int, G: int):
    """The static tables of a step's rows, from the library's host code:
    (depth [M], visibility words [M][8] as uint32, used rows [U]) as numpy
    arrays.  No GPU is touched."""
    import numpy as np
    lib = load_library()
    depth = np.zeros(256, dtype=np.int32)
    vis = np.zeros((256, 8), dtype=np.uint32)
    used = np.zeros(256, dtype=np.int32)
    m = np.zeros(1, dtype=np.int32)
    u = np.zeros(1, dtype=np.int32)
    rc = lib.la_step_tables(N, W, G, depth.ctypes.data_as(_I32P), vis.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)),
                            used.ctypes.data_as(_I32P), 256, m.ctypes.data_as(_I32P), u.ctypes.data_as(_I32P))
    _check(rc, "la_step_tables")
    return depth[:m[0]].copy(), vis[:m[0]].copy(), used[:u[0]].copy()


def la_gemm_schedule(tiles: int, n_kb: int, ctas: int, whole_first: bool):
    """The projection GEMMs' work split, from the library's host code: returns
    (segments [n][4] of (tile, kb0, kb1, plane), cta_first [ctas_used + 1],
    planes per tile [tiles]) as int32 numpy arrays.  No GPU is touched."""
    import numpy as np
    lib = load_library()
    cap = tiles + ctas + 16                      # a run adds at most one segment per tile boundary
    while True:
        segs = np.zeros((cap, 4), dtype=np.int32)
        first = np.zeros(ctas + 1, dtype=np.int32)
        used = np.zeros(1, dtype=np.int32)
        nseg = np.zeros(1, dtype=np.int32)
        planes = np.zeros(tiles, dtype=np.int32)
        ptr = lambda a: a.ctypes.data_as(_I32P)
        rc = lib.la_gemm_schedule(tiles, n_kb, ctas, int(bool(whole_first)), ptr(segs), cap, ptr(nseg), ptr(first),
                                  ptr(used), ptr(planes))
        if rc == LA_ERR_CAPACITY:
            cap *= 2
            continue
        _check(rc, "la_gemm_schedule")
        return segs[:nseg[0]].copy(), first[:used[0] + 1].copy(), planes


def la_destroy(h) -> None:
    if h:
        load_library().la_destroy(h)


# ---------------------------------------------------------------------------- owners
class DeviceWeights:
    """Device copies (torch tensors) of a weight dict in the synth.model_weights
    layout, and the la_weights / la_model_dims structs that point at them."""

    def __init__(self, weights: dict, device="cuda"):
        import torch
        dims = weights["dims"]
        self.dims = dims
        self._keep = []

        def up(a):
            if a.dtype == np.uint16:
                t = torch.from_numpy(a.view(np.int16)).to(device)
            else:
                t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)
            self._keep.append(t)
            return t.data_ptr()

        def arr(ptrs):
            a = (ctypes.c_void_p * len(ptrs))(*ptrs)
            self._keep.append(a)
            return ctypes.cast(a, _PP)

        names = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")
        per = {k: [] for k in names}
        for lw in weights["layers"]:
            for k in names:
                per[k].append(up(lw[k]))
        self.struct = la_weights(up(weights["embed"]), up(weights["final_norm"]), up(weights["lm_head"]),
                                 *[arr(per[k]) for k in names])
        self.dims_struct = la_model_dims(dims.n_layers, dims.d_model, dims.n_heads, dims.n_kv_heads, dims.head_dim,
                                         dims.ffn, dims.vocab, dims.rms_eps, dims.rope_base,
                                         LA_BF16 if dims.dtype == "bf16" else LA_F32)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self._keep if hasattr(t, "numel"))


class Decoder:
    """A la_handle over DeviceWeights (or a host weight dict, uploaded here)."""

    def __init__(self, weights, N: int, W: int, G: int, max_seq: int, temperature: float = 0.0,
                 seed: int = 0, prompt_as_reference: bool = False, pool_cap: int = 0, stream=None, device="cuda",
                 profile: bool = False, top_k: int = 0, top_p: float = 1.0, pool_policy: str = "fifo"):
        self.weights = weights if isinstance(weights, DeviceWeights) else DeviceWeights(weights, device)
        self.dims, self.N, self.W, self.G = self.weights.dims, N, W, G
        self.stream = stream
        sp = stream.cuda_stream if stream is not None else None
        policies = {"fifo": LA_POOL_FIFO, "lru": LA_POOL_LRU, "lfu": LA_POOL_LFU}
        if pool_policy not in policies:
            raise ValueError(f"pool_policy must be 'fifo', 'lru' or 'lfu', not {pool_policy!r}")
        o = la_opts(N, W, G, max_seq, int(prompt_as_reference), pool_cap, temperature, seed, sp, int(profile),
                    top_k, top_p, policies[pool_policy])
        self.h = la_create(self.weights.dims_struct, self.weights.struct, o)

    def prefill(self, prompt) -> int:
        return la_prefill(self.h, prompt)

    def step(self) -> List[int]:
        return la_step(self.h, self.N)

    def ar_step(self) -> int:
        return la_ar_step(self.h)

    def generate(self, prompt, max_new: int):
        return la_generate(self.h, prompt, max_new)

    def stats(self) -> dict:
        return la_stats(self.h)

    def export_state(self) -> dict:
        return la_export_state(self.h, self.N, self.W)

    def import_state(self, tokens, window, records, uses=None) -> None:
        la_import_state(self.h, self.N, self.W, tokens, window, records, uses)

    def debug_logits(self) -> np.ndarray:
        return la_debug_logits(self.h)

    def close(self):
        if getattr(self, "h", None):
            la_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
