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


# ---------------------------------------------------------------------------
# Hand-worked one-layer decoders (d = 4).  Each case zeroes or fixes weights
# so that the logits have a closed form worked out below with scalars; a
# wiring mistake in the oracle (SiLU on the wrong projection, a norm moved or
# skipped, the lm_head reading the raw residual, the FFN norm reading the
# pre-attention residual) changes the numbers.
# ---------------------------------------------------------------------------
import math


def _silu(z):
    return z / (1.0 + math.exp(-z))


def _one_layer(**over):
    dims = synth.ModelDims(1, 4, 1, 1, 4, 2, 3, rms_eps=0.0, dtype="f32")
    z4, z24, z42 = np.zeros((4, 4)), np.zeros((2, 4)), np.zeros((4, 2))
    layer = {"attn_norm": np.ones(4), "wq": z4, "wk": z4, "wv": z4, "wo": z4, "ffn_norm": np.ones(4),
             "w_gate": z24, "w_up": z24, "w_down": z42}
    w = {"dims": dims, "embed": np.zeros((3, 4)), "layers": [layer], "final_norm": np.ones(4),
         "lm_head": np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0], [1.0, 1.0, 1.0, 1.0]])}
    for k, v in over.items():
        (layer if k in layer else w)[k] = np.asarray(v, dtype=np.float64)
    return w


def _logits(w, token, position=0):
    lg, _ = decoder.forward(w, [token], np.array([position]), np.ones((1, 1), bool))
    return lg[0]


def _rms_normed(v, g=(1.0, 1.0, 1.0, 1.0)):
    r = math.sqrt(sum(x * x for x in v) / len(v))
    return [x / r * gi for x, gi in zip(v, g)]


def test_hand_worked_lm_head_reads_the_final_normed_residual():
    # No layer contribution: h = E[t] = (3, 4, 0, 0); rms 2.5 -> (1.2, 1.6, 0, 0);
    # final gain (2, 1, 1, 1) -> (2.4, 1.6, 0, 0); lm_head rows e0, e1, 1.
    w = _one_layer(embed=[[3.0, 4, 0, 0], [30.0, 40, 0, 0], [0, 0, 0, 1.0]], final_norm=[2.0, 1, 1, 1])
    np.testing.assert_allclose(_logits(w, 0), [2.4, 1.6, 4.0], rtol=1e-14)
    np.testing.assert_allclose(_logits(w, 1), [2.4, 1.6, 4.0], rtol=1e-14)   # scale-free: the norm is applied


def test_hand_worked_silu_goes_through_the_gate_projection():
    # Attention zero.  E[0] = (2, 0, 0, 0) has rms 1, so the FFN input is
    # (2, 0, 0, 0): gate = 1 * 2 = 2, up = 0.5 * 2 = 1, silu(2) * 1 goes to
    # h[1] through w_down[1][0] = 1.  Swapping gate and up would give silu(1) * 2.
    w = _one_layer(embed=[[2.0, 0, 0, 0], [0, 0, 0, 1.0], [0, 0, 1.0, 0]],
                   w_gate=[[1.0, 0, 0, 0], [0, 0, 0, 0]], w_up=[[0.5, 0, 0, 0], [0, 0, 0, 0]],
                   w_down=[[0, 0], [1.0, 0], [0, 0], [0, 0]])
    h = [2.0, _silu(2.0) * 1.0, 0.0, 0.0]
    x = _rms_normed(h)
    np.testing.assert_allclose(_logits(w, 0), [x[0], x[1], sum(x)], rtol=1e-13)
    assert abs(_silu(2.0) - _silu(1.0) * 2.0) > 0.25   # the swap is visible


def test_hand_worked_strongly_negative_gate_closes_the_ffn():
    # gate = -50 on the FFN input: silu(-50) * up is below 1e-20 whatever up is.
    w = _one_layer(embed=[[2.0, 0, 0, 0], [0, 0, 0, 1.0], [0, 0, 1.0, 0]],
                   w_gate=[[-25.0, 0, 0, 0], [0, 0, 0, 0]], w_up=[[7.0, 0, 0, 0], [0, 0, 0, 0]],
                   w_down=[[0, 0], [1.0, 0], [0, 0], [0, 0]])
    np.testing.assert_allclose(_logits(w, 0), [2.0, 0.0, 2.0], atol=1e-18)


def test_hand_worked_norm_gains_sit_where_the_decoder_puts_them():
    # The FFN gain (0.5, 1, 1, 1) halves the FFN input: gate 1, up 0.5,
    # h[1] = silu(1) * 0.5.  The attention gain (7, ...) changes nothing,
    # because attention is zero; swapping the two gains would change h[1].
    w = _one_layer(embed=[[2.0, 0, 0, 0], [0, 0, 0, 1.0], [0, 0, 1.0, 0]], attn_norm=[7.0, 7, 7, 7],
                   ffn_norm=[0.5, 1, 1, 1],
                   w_gate=[[1.0, 0, 0, 0], [0, 0, 0, 0]], w_up=[[0.5, 0, 0, 0], [0, 0, 0, 0]],
                   w_down=[[0, 0], [1.0, 0], [0, 0], [0, 0]])
    x = _rms_normed([2.0, _silu(1.0) * 0.5, 0.0, 0.0])
    np.testing.assert_allclose(_logits(w, 0), [x[0], x[1], sum(x)], rtol=1e-13)


def test_hand_worked_ffn_norm_reads_the_residual_after_attention():
    # One row at position 5 sees only itself: softmax weight 1, so the
    # attention output is v = Wv x_attn whatever the rotation does to q and k.
    # E[0] = (2, 2, 0, 0): rms 2^0.5, x_attn = (2^0.5, 2^0.5, 0, 0) with gain 1.
    # Wv = I, and Wo moves component 0 to component 2: h1 = (2, 2, 2^0.5, 0).
    # The FFN input is
    # rmsnorm(h1); gate row (1, 0, 0, 0), up row (0, 0, 1, 0), w_down[3][0] = 1:
    # h2[3] = silu(n0) * n2 with n = rmsnorm(h1).  Reading E[0] instead of h1
    # would give n2 = 0 and h2[3] = 0.
    wo = np.zeros((4, 4))
    wo[2, 0] = 1.0
    w = _one_layer(embed=[[2.0, 2.0, 0, 0], [0, 0, 0, 1.0], [0, 0, 1.0, 0]], wq=np.eye(4), wk=np.eye(4),
                   wv=np.eye(4), wo=wo, w_gate=[[1.0, 0, 0, 0], [0, 0, 0, 0]],
                   w_up=[[0, 0, 1.0, 0], [0, 0, 0, 0]], w_down=[[0, 0], [0, 0], [0, 0], [1.0, 0]])
    w["lm_head"] = np.array([[1.0, 0, 0, 0], [0, 0, 1.0, 0], [0, 0, 0, 1.0]])
    h1 = [2.0, 2.0, math.sqrt(2.0), 0.0]
    n = _rms_normed(h1)
    h2 = h1[:3] + [_silu(n[0]) * n[2]]
    x = _rms_normed(h2)
    np.testing.assert_allclose(_logits(w, 0, position=5), [x[0], x[2], x[3]], rtol=1e-13)
    assert x[3] > 0.1


def test_softmax_temperature_hand_worked():
    # logits ln(1, 4, 16): T = 1 gives (1, 4, 16) / 21; T = 2 gives (1, 2, 4) / 7.
    lg = np.log(np.array([1.0, 4.0, 16.0]))
    np.testing.assert_allclose(la.softmax(lg, 1.0), np.array([1, 4, 16]) / 21.0, rtol=1e-14)
    np.testing.assert_allclose(la.softmax(lg, 2.0), np.array([1, 2, 4]) / 7.0, rtol=1e-14)
    np.testing.assert_allclose(la.softmax(lg + 1000.0, 2.0), np.array([1, 2, 4]) / 7.0, rtol=1e-12)
