"""Lookahead step on the GPU vs the oracle, tiny fp32 decoder (2 layers,
d 256, 4 heads x 64, FFN 688, vocab 1024): end-to-end streams, step-level
teacher-forced parity (accepted tokens, new window, pool, logits <= 1e-4),
edge configurations and error paths."""
import numpy as np
import pytest

import synth
from helpers import MARGIN_F32 as MARGIN, ar_with_margins, compare_stream, ensure_built, teacher_forced, top2_margin
from oracle import lookahead as la

pytestmark = pytest.mark.gpu

LOGIT_TOL_F32 = 1e-4


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    import exact_decoding_gb300 as e
    return e


@pytest.fixture(scope="module")
def tiny_model():
    wl = synth.WORKLOADS["tiny-fp32-greedy"]
    return wl, synth.model_weights(wl.dims, wl.seed), synth.prompt(wl)


def make(lib, w, N, W, G, max_seq=256, **kw):
    return lib.Decoder(w, N, W, G, max_seq, **kw)


def test_prefill_first_token_and_logits(lib, tiny_model):
    from oracle import decoder
    wl, w, p = tiny_model
    dec = make(lib, w, 3, 4, 4)
    y1 = dec.prefill(p)
    ref, _ = decoder.forward(w, list(p), np.arange(len(p)), decoder.causal_mask(0, len(p)), logit_rows=[len(p) - 1])
    g = dec.debug_logits()
    assert g.shape == (1, wl.dims.vocab)
    assert np.max(np.abs(g[0] - ref[0])) <= LOGIT_TOL_F32
    assert y1 == la.argmax_lowest(ref[0]) or top2_margin(ref[0]) <= MARGIN
    dec.close()


@pytest.mark.parametrize("N,W,G,par", [(3, 4, 4, False), (2, 3, 2, False), (5, 3, 0, False), (4, 2, 5, True),
                                       (3, 1, 1, False), (8, 2, 3, False)])
def test_generate_equals_autoregressive(lib, tiny_model, N, W, G, par):
    wl, w, p = tiny_model
    ar, margins = ar_with_margins(w, p, wl.new_tokens)
    dec = make(lib, w, N, W, G, prompt_as_reference=par)
    out, steps = dec.generate(p, wl.new_tokens)
    assert len(out) == wl.new_tokens
    upto = compare_stream(out, ar, margins, MARGIN)
    assert upto >= 16, f"first low-margin decision at {upto}"
    st = dec.stats()
    assert st["steps"] == steps and st["generated"] >= wl.new_tokens
    dec.close()


def _teacher_forced(lib, w, p, N, W, G, steps, par=False, pool_policy=la.FIFO, pool_cap=0):
    return teacher_forced(lib, w, p, N, W, G, steps, MARGIN, LOGIT_TOL_F32, par=par, pool_policy=pool_policy,
                          pool_cap=pool_cap, max_seq=256)


def test_step_teacher_forced_greedy(lib, tiny_model):
    wl, w, p = tiny_model
    t = _teacher_forced(lib, w, p, 3, 4, 4, steps=12)
    print(t)
    assert t.steps == 12 and t.accept_compared >= 10 and t.columns_compared >= 40


def test_step_teacher_forced_repetitive_prompt(lib, tiny_model):
    """A repeated prompt with prompt-as-reference makes candidates hit (A > 1)."""
    wl, w, _ = tiny_model
    p = np.tile(synth.uniform_tokens(8, wl.dims.vocab, seed=9), 5)
    t = _teacher_forced(lib, w, p, 4, 3, 4, steps=10, par=True)
    print(t)
    assert t.steps == 10 and t.accept_compared >= 8 and t.accept_compared_multi >= 1


@pytest.mark.parametrize("N,W,G,cap", [(4, 3, 4, 0), (4, 3, 2, 5), (3, 4, 3, 3)])
def test_step_teacher_forced_lru_pool(lib, tiny_model, N, W, G, cap):
    """LRU pool: candidates most recent first, the winner and repeated
    harvests move to the most recent end; the pool after every step equals
    the oracle's replay, and some steps do accept a candidate."""
    wl, w, _ = tiny_model
    p = np.tile(synth.uniform_tokens(6, wl.dims.vocab, seed=4), 6)
    t = _teacher_forced(lib, w, p, N, W, G, steps=12, par=True, pool_policy=la.LRU, pool_cap=cap)
    print(t)
    assert t.steps == 12 and t.hits >= 1 and t.accept_compared >= 9 and t.accept_compared_multi >= 1


def test_generate_lru_pool_equals_autoregressive(lib, tiny_model):
    wl, w, _ = tiny_model
    p = np.tile(synth.uniform_tokens(6, wl.dims.vocab, seed=4), 6)
    ar, margins = ar_with_margins(w, p, wl.new_tokens)
    dec = make(lib, w, 4, 3, 2, prompt_as_reference=True, pool_policy=la.LRU, pool_cap=5)
    out, steps = dec.generate(p, wl.new_tokens)
    upto = compare_stream(out, ar, margins, MARGIN)
    assert upto >= 16, f"first low-margin decision at {upto}"
    assert steps < wl.new_tokens - 1     # some steps accepted more than one token
    dec.close()


@pytest.mark.parametrize("N,W,G,cap", [(4, 3, 4, 0), (4, 3, 2, 2), (3, 4, 3, 3)])
def test_step_teacher_forced_lfu_pool(lib, tiny_model, N, W, G, cap):
    """LFU pool (reading R16): use counts beside the device ring, each key's
    list ordered by (uses, time); after every step the pool and the counts
    equal the oracle's replay, and candidates hit.  These shapes end with a
    pool that differs from the LRU pool's on the same run."""
    wl, w, _ = tiny_model
    p = np.tile(synth.uniform_tokens(6, wl.dims.vocab, seed=4), 6)
    t = _teacher_forced(lib, w, p, N, W, G, steps=14, par=True, pool_policy=la.LFU, pool_cap=cap)
    print(t)
    assert t.steps == 14 and t.hits >= 2 and t.accept_compared >= 11 and t.accept_compared_multi >= 2


def test_generate_lfu_pool_equals_autoregressive(lib, tiny_model):
    wl, w, _ = tiny_model
    p = np.tile(synth.uniform_tokens(6, wl.dims.vocab, seed=4), 6)
    ar, margins = ar_with_margins(w, p, wl.new_tokens)
    dec = make(lib, w, 4, 3, 2, prompt_as_reference=True, pool_policy=la.LFU, pool_cap=2)
    out, steps = dec.generate(p, wl.new_tokens)
    upto = compare_stream(out, ar, margins, MARGIN)
    assert upto >= 16, f"first low-margin decision at {upto}"
    assert steps < wl.new_tokens - 1
    dec.close()


def test_lfu_state_with_counts_resumes_identically(lib, tiny_model):
    """An LFU snapshot carries the use counts; a fresh handle that imports it
    continues exactly like the handle that kept stepping (tokens, pool and
    counts)."""
    wl, w, _ = tiny_model
    p = np.tile(synth.uniform_tokens(6, wl.dims.vocab, seed=4), 6)
    a = make(lib, w, 3, 4, 3, prompt_as_reference=True, pool_policy=la.LFU, pool_cap=3)
    a.prefill(p)
    for _ in range(8):
        a.step()
    s = a.export_state()
    assert max(s["uses"]) >= 2
    b = make(lib, w, 3, 4, 3, prompt_as_reference=True, pool_policy=la.LFU, pool_cap=3)
    b.import_state(s["tokens"], s["window"], s["records"], s["uses"])
    assert b.export_state()["uses"] == s["uses"]
    for _ in range(6):
        assert a.step() == b.step()
    sa, sb = a.export_state(), b.export_state()
    assert sa["records"] == sb["records"] and sa["uses"] == sb["uses"]
    a.close()
    b.close()


def test_step_teacher_forced_sampling(lib, tiny_model):
    """Algorithm 4: same Philox draws on both sides; decisions within 1e-3 of
    a threshold may differ (fp32 vs fp64), everything else must match."""
    wl, w, _ = tiny_model
    p = np.tile(synth.uniform_tokens(8, wl.dims.vocab, seed=9), 5)
    N, W, G = 4, 3, 4
    dec = make(lib, w, N, W, G, temperature=1.0, seed=1234, prompt_as_reference=True)
    dec.prefill(p)
    orc = la.Lookahead(w, N, W, G, temperature=1.0, seed=1234, prompt_as_reference=True, keep_logits=True)
    exact = 0
    for t in range(10):
        s0 = dec.export_state()
        orc.load_state(s0["tokens"], s0["window"], s0["records"])
        acc_ref = orc.step()
        trace = orc.history[-1].trace
        acc = dec.step()
        if acc == acc_ref:
            exact += 1
            continue
        # find the first differing decision: it must be a near-tie
        k = next(i for i in range(min(len(acc), len(acc_ref))) if acc[i] != acc_ref[i]) \
            if any(a != b for a, b in zip(acc, acc_ref)) else min(len(acc), len(acc_ref))
        near = [d for d in trace if abs(d.value) <= 1e-3]
        assert near, f"step {t}: gpu {acc} vs oracle {acc_ref} with no near-threshold decision"
    assert exact >= 8
    dec.close()


def test_import_state_resumes_identically(lib, tiny_model):
    wl, w, p = tiny_model
    a = make(lib, w, 3, 4, 4)
    a.prefill(p)
    for _ in range(5):
        a.step()
    s = a.export_state()
    b = make(lib, w, 3, 4, 4)
    b.import_state(s["tokens"], s["window"], s["records"])
    for _ in range(6):
        assert a.step() == b.step()
    assert a.export_state()["records"] == b.export_state()["records"]
    a.close()
    b.close()


def test_runs_are_bitwise_deterministic(lib, tiny_model):
    wl, w, p = tiny_model
    outs = []
    for _ in range(2):
        dec = make(lib, w, 4, 4, 4, prompt_as_reference=True)
        outs.append((dec.generate(p, 40), dec.debug_logits().tobytes()))
        dec.close()
    assert outs[0] == outs[1]


def test_error_paths(lib, tiny_model):
    wl, w, p = tiny_model
    dec = make(lib, w, 3, 4, 4, max_seq=64)
    with pytest.raises(lib.LaError) as e:
        dec.step()
    assert e.value.code == -6            # step before prefill
    with pytest.raises(lib.LaError) as e:
        dec.prefill([1, 2])              # shorter than N
    assert e.value.code == -1
    with pytest.raises(lib.LaError) as e:
        dec.prefill(list(p) + [5000])    # token out of range
    assert e.value.code == -1
    dec.prefill(p)
    with pytest.raises(lib.LaError) as e:
        for _ in range(64):
            dec.step()
    assert e.value.code == -3            # max_seq reached, reported before any launch
    dec.close()


def test_ar_step_equals_oracle_autoregressive(lib, tiny_model):
    """la_ar_step (the plain autoregressive baseline) reproduces the oracle's
    greedy AR stream, and interleaving it with lookahead steps keeps the
    stream on the same greedy trajectory."""
    wl, w, p = tiny_model
    ar, margins = ar_with_margins(w, p, 40)
    dec = make(lib, w, 3, 4, 4)
    out = [dec.prefill(p)]
    for _ in range(20):
        out.append(dec.ar_step())
    while len(out) < 40:
        out.extend(dec.step())
    for _ in range(3):
        out.append(dec.ar_step())
    out = out[:40]
    upto = compare_stream(out, ar, margins, MARGIN)
    assert upto >= 16, f"first low-margin decision at {upto}"
    dec.close()


def test_sampling_top_k1_equals_greedy(lib, tiny_model):
    """top_k = 1 keeps one token per distribution: lookahead sampling at T = 1
    on the GPU reproduces the greedy autoregressive stream."""
    wl, w, p = tiny_model
    ar, margins = ar_with_margins(w, p, 40)
    dec = make(lib, w, 3, 4, 4, temperature=1.0, seed=77, top_k=1)
    out, _ = dec.generate(p, 40)
    upto = compare_stream(out, ar, margins, MARGIN)
    assert upto >= 16, f"first low-margin decision at {upto}"
    dec.close()


def _keep_sets_safe(orc_logits_rows, T, top_k, top_p, eps=1e-4):
    """True when no top-k / top-p boundary of these rows lies within eps (in
    logit for top-k, in renormalised mass for top-p) of a flip, so fp32 and
    fp64 must keep the same tokens."""
    for l in orc_logits_rows:
        l = np.asarray(l, dtype=np.float64)
        order = sorted(range(len(l)), key=lambda v: (-l[v], v))
        if 0 < top_k < len(l) and l[order[top_k - 1]] - l[order[top_k]] <= eps:
            return False
        if 0 < top_p < 1:
            kept = order[:top_k] if 0 < top_k < len(l) else order
            q = np.exp((l[kept] - l[kept[0]]) / T)
            c = np.cumsum(q) / q.sum()
            if np.min(np.abs(c - top_p)) <= eps:
                return False
    return True


@pytest.mark.parametrize("top_k,top_p", [(8, 1.0), (0, 0.9), (6, 0.8)])
def test_step_teacher_forced_sampling_top_k_top_p(lib, tiny_model, top_k, top_p):
    """Algorithm 4 on top-k / top-p filtered distributions: same Philox draws
    on both sides; a step may differ only where a draw sits within 1e-3 of
    its threshold or a filter boundary within 1e-4 of a flip."""
    wl, w, _ = tiny_model
    p = np.tile(synth.uniform_tokens(8, wl.dims.vocab, seed=19), 5)
    N, W, G = 4, 3, 4
    T = 0.7
    dec = make(lib, w, N, W, G, temperature=T, seed=4321, prompt_as_reference=True, top_k=top_k, top_p=top_p)
    dec.prefill(p)
    orc = la.Lookahead(w, N, W, G, temperature=T, seed=4321, prompt_as_reference=True, keep_logits=True,
                       top_k=top_k, top_p=top_p)
    exact = 0
    for t in range(10):
        s0 = dec.export_state()
        orc.load_state(s0["tokens"], s0["window"], s0["records"])
        acc_ref = orc.step()
        rec = orc.history[-1]
        acc = dec.step()
        if acc == acc_ref:
            exact += 1
            continue
        near = [d for d in rec.trace if abs(d.value) <= 1e-3]
        rows = [rec.logits[0]] + [rec.logits[1 + W + i] for i in range(G * (N - 1))]
        assert near or not _keep_sets_safe(rows, T, top_k, top_p), \
            f"step {t}: gpu {acc} vs oracle {acc_ref} with no near-threshold decision"
    assert exact >= 7
    dec.close()
