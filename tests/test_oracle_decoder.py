"""Pins of the oracle's decoder forward against closed forms, library
routines and invariants (not against itself)."""
import numpy as np
import pytest
import torch

import synth
from oracle import decoder, lookahead as la


def test_rmsnorm_closed_form():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(5, 64)) * 3.0
    y = decoder.rmsnorm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-12)
    np.testing.assert_allclose(decoder.rmsnorm(7.5 * x, np.ones(64), 0.0), y, rtol=1e-12)
    g = rng.normal(size=64)
    np.testing.assert_allclose(decoder.rmsnorm(x, g, 0.0), y * g, rtol=1e-12)


def test_silu_matches_library():
    x = np.linspace(-20, 20, 401)
    np.testing.assert_allclose(decoder.silu(x), torch.nn.functional.silu(torch.from_numpy(x)).numpy(),
                               rtol=1e-13, atol=1e-300)


def test_rope_is_complex_rotation():
    """Rotate-half pairs (i, i+hd/2) = multiplying x_i + 1j*x_{i+hd/2} by exp(1j*p*base^(-2i/hd))."""
    rng = np.random.default_rng(2)
    hd, base = 16, 10000.0
    x = rng.normal(size=(6, 3, hd))
    pos = np.array([0, 1, 5, 17, 300, 2047])
    y = decoder.rope(x, pos, base)
    z = x[..., : hd // 2] + 1j * x[..., hd // 2:]
    theta = np.array([base ** (-2.0 * i / hd) for i in range(hd // 2)])
    zr = z * np.exp(1j * pos[:, None, None] * theta[None, None, :])
    np.testing.assert_allclose(y[..., : hd // 2], zr.real, atol=1e-12)
    np.testing.assert_allclose(y[..., hd // 2:], zr.imag, atol=1e-12)
    np.testing.assert_allclose(decoder.rope(x, np.zeros(6), base), x)   # position 0 is identity


def test_rope_relative_positions():
    rng = np.random.default_rng(3)
    q, k = rng.normal(size=(1, 1, 32)), rng.normal(size=(1, 1, 32))
    d1 = np.sum(decoder.rope(q, [40], 1e4) * decoder.rope(k, [33], 1e4))
    d2 = np.sum(decoder.rope(q, [1007], 1e4) * decoder.rope(k, [1000], 1e4))
    assert abs(d1 - d2) < 1e-10


@pytest.mark.parametrize("n_h,n_kv", [(4, 4), (8, 2)])
def test_attention_matches_library(n_h, n_kv):
    rng = np.random.default_rng(4)
    n, nk, hd = 7, 11, 16
    q = rng.normal(size=(n, n_h, hd))
    k = rng.normal(size=(nk, n_kv, hd))
    v = rng.normal(size=(nk, n_kv, hd))
    vis = rng.random((n, nk)) < 0.6
    vis[:, 0] = True
    out = decoder.attention(q, k, v, vis)
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(n_h // n_kv, dim=0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(n_h // n_kv, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(vis))
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).reshape(n, n_h * hd).numpy(), atol=1e-12)


def test_incremental_equals_full_forward(tiny):
    """Row-by-row decoding with a KV cache == one causal pass over the sequence."""
    wl, w, p = tiny
    toks = list(p[:12])
    full, _ = decoder.forward(w, toks, np.arange(12), decoder.causal_mask(0, 12))
    _, cache = decoder.forward(w, toks[:5], np.arange(5), decoder.causal_mask(0, 5))
    for i in range(5, 12):
        lg, kv = decoder.forward(w, [toks[i]], np.array([i]), np.ones((1, i + 1), bool), cache=cache)
        np.testing.assert_allclose(lg[0], full[i], atol=1e-12)
        cache = decoder.concat_cache(cache, kv)


def test_tree_rows_equal_their_linear_paths(tiny):
    """Each step row, under the lookahead mask, computes exactly what a plain
    causal pass computes over prefix + its ancestor chain + itself at the
    same positions (this pins the mask together with the positions)."""
    wl, w, p = tiny
    N, W, G = 4, 3, 2
    rows = la.step_rows(N, W, G)
    P = 10
    rng = np.random.default_rng(5)
    toks = rng.integers(0, wl.dims.vocab, size=len(rows))
    prefix = list(p[:P])
    _, cache = decoder.forward(w, prefix, np.arange(P), decoder.causal_mask(0, P))
    pos = np.array([P + r.depth for r in rows])
    vis = np.concatenate([np.ones((len(rows), P), bool), la.step_mask(N, W, G)], axis=1)
    step_logits, _ = decoder.forward(w, toks, pos, vis, cache=cache)
    for r in range(len(rows)):
        chain = list(reversed(la.ancestors(rows, r))) + [r]
        seq = prefix + [int(toks[c]) for c in chain]
        cpos = list(range(P)) + [P + rows[c].depth for c in chain]
        assert cpos == list(range(P + len(chain))), "a path's positions must be consecutive"
        lin, _ = decoder.forward(w, seq, np.array(cpos), decoder.causal_mask(0, len(seq)),
                                 logit_rows=[len(seq) - 1])
        np.testing.assert_allclose(step_logits[r], lin[0], atol=1e-11)


def test_bf16_widening_is_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x4049, 0x3C23], dtype=np.uint16)
    np.testing.assert_array_equal(decoder.as_float(bits), [1.0, -1.0, 0.0, 3.140625, 1.2734375 * 2.0 ** -7])
