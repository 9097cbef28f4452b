"""Seeded synthetic inputs for the lookahead-decoding step.

This module generates inputs only: the workload configurations, random model
weights N(0, 0.02) and uniform prompts.  It holds none of the decoding
arithmetic, so the CPU oracle and the CUDA path can both draw from it without
sharing any of the method.

Weights: one Philox4x32-10 stream per tensor (key = seed, counter = element
pair index and tensor index), Box-Muller in double precision, rounded to fp32
and, for bf16 models, to bfloat16 by round-to-nearest-even.  Norm gains are 1.
Tensor order (stream index): embed, then per layer [attn_norm, wq, wk, wv, wo,
ffn_norm, w_gate, w_up, w_down], then final_norm, lm_head.  All matrices are
row-major [out][in].
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
from typing import Dict, List, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_gen.so")
_lib = None

PROMPT_STREAM = 0x50000000


def build_generator(force: bool = False) -> str:
    """Compile gen.c into a shared library next to it (plain C, OpenMP)."""
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, src, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build_generator())
        _lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_double,
                                          ctypes.c_void_p, ctypes.c_int64]
        _lib.synth_normal_bf16.argtypes = _lib.synth_normal_f32.argtypes
        _lib.synth_uniform_tokens.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32,
                                              ctypes.c_void_p, ctypes.c_int64]
        _lib.synth_philox4x32_10.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return _lib


@dataclasses.dataclass(frozen=True)
class ModelDims:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-5
    rope_base: float = 10000.0
    dtype: str = "bf16"  # "f32" or "bf16"

    def n_params(self) -> int:
        d, hd = self.d_model, self.head_dim
        per_layer = (2 * d + d * self.n_heads * hd * 2 + d * self.n_kv_heads * hd * 2
                     + 3 * d * self.ffn)
        return self.n_layers * per_layer + 2 * self.vocab * d + d


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dims: ModelDims
    prompt_len: int
    N: int
    W: int
    G: int
    new_tokens: int
    temperature: float = 0.0
    prompt_as_reference: bool = False
    prompt_chunk: int = 0          # >0: prompt is one random chunk of this length repeated
    seed: int = 0

    @property
    def M(self) -> int:
        """Rows in one step: 1 + (W + G)(N - 1)."""
        return 1 + (self.W + self.G) * (self.N - 1)

    @property
    def max_seq(self) -> int:
        return self.prompt_len + self.new_tokens + self.M + 2 * self.N + 8


TINY = ModelDims(2, 256, 4, 4, 64, 688, 1024, dtype="f32")
LLAMA7B = ModelDims(32, 4096, 32, 32, 128, 11008, 32000)
CODELLAMA13B = ModelDims(40, 5120, 40, 40, 128, 13824, 32016)
LLAMA70B = ModelDims(80, 8192, 64, 8, 128, 28672, 32000)

WORKLOADS: Dict[str, Workload] = {
    "tiny-fp32-greedy": Workload("tiny-fp32-greedy", TINY, 32, 3, 4, 4, 64),
    "llama7b-bf16-greedy": Workload("llama7b-bf16-greedy", LLAMA7B, 256, 5, 15, 15, 256),
    "llama7b-bf16-sampling": Workload("llama7b-bf16-sampling", LLAMA7B, 512, 5, 7, 7, 256,
                                      temperature=1.0, prompt_as_reference=True, prompt_chunk=64),
    "codellama13b-bf16-greedy": Workload("codellama13b-bf16-greedy", CODELLAMA13B, 2048, 5, 10, 10, 512),
    "llama70b-bf16-greedy": Workload("llama70b-bf16-greedy", LLAMA70B, 512, 5, 5, 5, 128),
    # 7B layer shapes with 2 layers (about 1.3 GB of weights): small enough
    # for full-counter kernel profiles, same per-launch GEMM/attention shapes.
    "llama7b-2layer-bf16-greedy": Workload("llama7b-2layer-bf16-greedy", dataclasses.replace(LLAMA7B, n_layers=2),
                                           256, 5, 15, 15, 256),
}


def philox4x32_10(ctr, key) -> List[int]:
    """The generator's raw block function (for known-answer tests)."""
    lib = _load()
    c = (ctypes.c_uint32 * 4)(*ctr)
    k = (ctypes.c_uint32 * 2)(*key)
    o = (ctypes.c_uint32 * 4)()
    lib.synth_philox4x32_10(c, k, o)
    return list(o)


def normal(shape, seed: int, stream: int, std: float = 0.02, dtype: str = "f32") -> np.ndarray:
    """N(0, std) array; dtype "f32" -> float32, "bf16" -> uint16 bfloat16 bits."""
    lib = _load()
    n = int(np.prod(shape))
    if dtype == "f32":
        out = np.empty(shape, dtype=np.float32)
        lib.synth_normal_f32(seed, stream, std, out.ctypes.data, n)
    elif dtype == "bf16":
        out = np.empty(shape, dtype=np.uint16)
        lib.synth_normal_bf16(seed, stream, std, out.ctypes.data, n)
    else:
        raise ValueError(dtype)
    return out


def ones(shape, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ones(shape, dtype=np.float32)
    return np.full(shape, 0x3F80, dtype=np.uint16)  # bfloat16 1.0


def uniform_tokens(n: int, vocab: int, seed: int, stream: int = PROMPT_STREAM) -> np.ndarray:
    lib = _load()
    out = np.empty(n, dtype=np.int32)
    lib.synth_uniform_tokens(seed, stream, vocab, out.ctypes.data, n)
    return out


def model_weights(dims: ModelDims, seed: int = 0, std: float = 0.02,
                  layers: Optional[List[int]] = None, lm_head_std: Optional[float] = None) -> dict:
    """All weights of a LLaMA-style decoder.  `layers` limits which layers are
    materialised (the others are None) for callers that stream layer by layer.
    `lm_head_std` (default `std`) draws the lm_head with another spread: the
    final hidden row has RMS 1, so the logits' spread is lm_head_std *
    sqrt(d_model); small test models use it to get 7B-like logit spreads."""
    dt = dims.dtype
    d, hd, L = dims.d_model, dims.head_dim, dims.n_layers
    w = {"dims": dims, "embed": normal((dims.vocab, d), seed, 0, std, dt), "layers": []}
    for l in range(L):
        if layers is not None and l not in layers:
            w["layers"].append(None)
            continue
        w["layers"].append(layer_weights(dims, l, seed, std))
    w["final_norm"] = ones((d,), dt)
    w["lm_head"] = normal((dims.vocab, d), seed, 2 + 9 * L, std if lm_head_std is None else lm_head_std, dt)
    return w


def layer_weights(dims: ModelDims, l: int, seed: int = 0, std: float = 0.02) -> dict:
    dt = dims.dtype
    d, hd = dims.d_model, dims.head_dim
    b = 1 + 9 * l
    return {
        "attn_norm": ones((d,), dt),
        "wq": normal((dims.n_heads * hd, d), seed, b + 1, std, dt),
        "wk": normal((dims.n_kv_heads * hd, d), seed, b + 2, std, dt),
        "wv": normal((dims.n_kv_heads * hd, d), seed, b + 3, std, dt),
        "wo": normal((d, dims.n_heads * hd), seed, b + 4, std, dt),
        "ffn_norm": ones((d,), dt),
        "w_gate": normal((dims.ffn, d), seed, b + 6, std, dt),
        "w_up": normal((dims.ffn, d), seed, b + 7, std, dt),
        "w_down": normal((d, dims.ffn), seed, b + 8, std, dt),
    }


class LazyLayers:
    """Per-layer weight dicts generated on access (the same values as
    model_weights), so models larger than host memory can be streamed to the
    device or through the CPU oracle one layer at a time."""

    def __init__(self, dims: ModelDims, seed: int = 0, std: float = 0.02):
        self.dims, self.seed, self.std = dims, seed, std

    def __len__(self):
        return self.dims.n_layers

    def __getitem__(self, l):
        if l < 0 or l >= self.dims.n_layers:
            raise IndexError(l)
        return layer_weights(self.dims, l, self.seed, self.std)

    def __iter__(self):
        return (self[l] for l in range(len(self)))


def lazy_model_weights(dims: ModelDims, seed: int = 0, std: float = 0.02) -> dict:
    """model_weights with the layers generated on access (LazyLayers)."""
    return {"dims": dims, "embed": normal((dims.vocab, dims.d_model), seed, 0, std, dims.dtype),
            "layers": LazyLayers(dims, seed, std), "final_norm": ones((dims.d_model,), dims.dtype),
            "lm_head": normal((dims.vocab, dims.d_model), seed, 2 + 9 * dims.n_layers, std, dims.dtype)}


def prompt(wl: Workload) -> np.ndarray:
    """The workload's prompt: uniform ids, or one uniform chunk repeated."""
    V = wl.dims.vocab
    if wl.prompt_chunk:
        chunk = uniform_tokens(wl.prompt_chunk, V, wl.seed)
        reps = -(-wl.prompt_len // wl.prompt_chunk)
        return np.tile(chunk, reps)[: wl.prompt_len].copy()
    return uniform_tokens(wl.prompt_len, V, wl.seed)


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits (uint16) to float32."""
    return (a.astype(np.uint32) << 16).view(np.float32)
