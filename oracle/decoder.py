"""LLaMA-style decoder forward, written out plainly in numpy (oracle side).

The pages run the method on LLaMA-2 / CodeLlama (paper-graph-ui page, section
5, "Experimental setup"); the decoder itself is the textbook one:

  h = E[token]
  per layer:  x = rmsnorm(h) * g_attn
              q, k, v = Wq x, Wk x, Wv x;  rotate q, k by the row's position
              a = softmax over the row's visible keys of (q . k / sqrt(hd)) v
              h = h + Wo a
              x = rmsnorm(h) * g_ffn
              h = h + Wd (silu(Wg x) * (Wu x))
  logits = Wlm (rmsnorm(h) * g_final)

Readings where the pages are silent: rotary embedding in the rotate-half form
(pairs i, i + hd/2; angle = position * base**(-2i/hd)); query head i reads
key/value head floor(i * n_kv / n_h); RMSNorm eps from the model dims.

Which keys a row sees is an explicit boolean matrix built by the caller
(`lookahead.py` builds the lookahead mask); nothing here knows about it.
"""
from __future__ import annotations

import numpy as np


def as_float(a, dtype=np.float64):
    """Weights arrive as float32 or as bfloat16 bits (uint16): widen exactly."""
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << 16).view(np.float32)
    return np.asarray(a, dtype=dtype)


def rmsnorm(x, g, eps):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def silu(x):
    return x / (1.0 + np.exp(-x))


def rope(x, positions, base):
    """x: [n, heads, hd]; rotate pairs (i, i + hd/2) by positions * base**(-2i/hd)."""
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = base ** (-(2.0 * np.arange(half, dtype=np.float64)) / hd)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    c = np.cos(ang)[:, None, :].astype(x.dtype)
    s = np.sin(ang)[:, None, :].astype(x.dtype)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def attention(q, k, v, visible):
    """q: [n, n_h, hd]; k, v: [n_keys, n_kv, hd]; visible: [n, n_keys] bool."""
    n, n_h, hd = q.shape
    n_kv = k.shape[1]
    out = np.empty((n, n_h, hd), dtype=q.dtype)
    for h in range(n_h):
        kvh = (h * n_kv) // n_h
        s = q[:, h, :] @ k[:, kvh, :].T / np.sqrt(hd)
        s = np.where(visible, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, kvh, :]
    return out.reshape(n, n_h * hd)


def forward(weights, tokens, positions, visible, cache=None, dtype=np.float64, logit_rows=None):
    """Run the decoder over `tokens` (new rows) given an optional KV cache.

    weights   -- dict from synth.model_weights (weights["layers"][l] indexable)
    tokens    -- [n] token ids of the new rows
    positions -- [n] absolute positions of the new rows
    visible   -- [n, n_cache + n] bool: keys are the cached rows, then the new rows
    cache     -- list over layers of (K [n_cache, n_kv, hd], V) or None
    logit_rows-- which new rows need logits (default all)
    Returns (logits [len(logit_rows), vocab], new_cache) where new_cache holds
    this call's K/V rows per layer (rotated K), not concatenated with `cache`.
    """
    dims = weights["dims"]
    n = len(tokens)
    hd, n_h, n_kv = dims.head_dim, dims.n_heads, dims.n_kv_heads
    eps = dims.rms_eps
    h = as_float(weights["embed"][np.asarray(tokens)], dtype)
    new_cache = []
    for l in range(dims.n_layers):
        lw = weights["layers"][l]
        x = rmsnorm(h, as_float(lw["attn_norm"], dtype), eps)
        q = (x @ as_float(lw["wq"], dtype).T).reshape(n, n_h, hd)
        k = (x @ as_float(lw["wk"], dtype).T).reshape(n, n_kv, hd)
        v = (x @ as_float(lw["wv"], dtype).T).reshape(n, n_kv, hd)
        q = rope(q, positions, dims.rope_base)
        k = rope(k, positions, dims.rope_base)
        new_cache.append((k, v))
        if cache is not None and len(cache[l][0]):
            K = np.concatenate([cache[l][0].astype(dtype), k], axis=0)
            V = np.concatenate([cache[l][1].astype(dtype), v], axis=0)
        else:
            K, V = k, v
        a = attention(q, K, V, visible)
        h = h + a @ as_float(lw["wo"], dtype).T
        x = rmsnorm(h, as_float(lw["ffn_norm"], dtype), eps)
        gate = x @ as_float(lw["w_gate"], dtype).T
        up = x @ as_float(lw["w_up"], dtype).T
        h = h + (silu(gate) * up) @ as_float(lw["w_down"], dtype).T
    if logit_rows is None:
        logit_rows = np.arange(n)
    xf = rmsnorm(h[np.asarray(logit_rows)], as_float(weights["final_norm"], dtype), eps)
    logits = xf @ as_float(weights["lm_head"], dtype).T
    return logits, new_cache


def causal_mask(n_cache, n):
    """Row i of the new block sees every cached key and new rows 0..i."""
    vis = np.zeros((n, n_cache + n), dtype=bool)
    vis[:, :n_cache] = True
    vis[:, n_cache:] = np.tril(np.ones((n, n), dtype=bool))
    return vis


def concat_cache(a, b):
    if a is None:
        return [(k.copy(), v.copy()) for k, v in b]
    return [(np.concatenate([ka, kb]), np.concatenate([va, vb])) for (ka, va), (kb, vb) in zip(a, b)]
