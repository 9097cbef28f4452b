"""bf16 path (tcgen05 GEMMs, tensor-core lookahead attention) vs the oracle on
small bf16 decoders: teacher-forced steps, logits within 2e-2, tokens exact
where the oracle's margin exceeds 0.05, pool exact.  Shapes cover head dim 64
and 128, grouped-query attention, several prefix chunks and prefill chunks."""
import dataclasses

import numpy as np
import pytest

import synth
from helpers import MARGIN, ensure_built, top2_margin
from oracle import lookahead as la

pytestmark = pytest.mark.gpu
LOGIT_TOL_BF16 = 2e-2

SMALL = {
    "mha-hd64": synth.ModelDims(2, 256, 4, 4, 64, 688, 1024, dtype="bf16"),
    "gqa-hd128": synth.ModelDims(2, 512, 8, 2, 128, 1024, 2048, dtype="bf16"),
    "mha-hd128-3l": synth.ModelDims(3, 512, 4, 4, 128, 1376, 1536, dtype="bf16"),
}


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    import exact_decoding_gb300 as e
    return e


def run_teacher_forced(lib, w, prompt, N, W, G, steps, par=False, max_seq=1024):
    dec = lib.Decoder(w, N, W, G, max_seq, prompt_as_reference=par)
    dec.prefill(prompt)
    orc = la.Lookahead(w, N, W, G, prompt_as_reference=par, keep_logits=True)
    worst = 0.0
    for t in range(steps):
        s0 = dec.export_state()
        orc.load_state(s0["tokens"], s0["window"], s0["records"])
        acc_ref = orc.step()
        rec = orc.history[-1]
        acc = dec.step()
        logits = dec.debug_logits()
        err = float(np.max(np.abs(logits - rec.logits)))
        worst = max(worst, err)
        assert err <= LOGIT_TOL_BF16, f"step {t}: logits max-abs {err}"
        decisive = [0] + [1 + W + i for i in range(G * (N - 1))]
        if not any(top2_margin(rec.logits[i]) <= MARGIN for i in decisive):
            assert acc == acc_ref, f"step {t}"
        s1 = dec.export_state()
        for j in range(W):
            lr = rec.logits[1 + j]
            gnew = int(s1["window"][N - 2, j])
            if top2_margin(lr) > MARGIN:
                assert gnew == rec.new[j], f"step {t} column {j}"
        pool = la.Pool.from_records(orc.pool.cap, s0["records"])
        for key, suf in la.harvest(np.asarray(s0["window"]), [int(x) for x in s1["window"][N - 2]]):
            pool.insert(key, suf)
        assert pool.records() == s1["records"]
        assert s1["tokens"] == s0["tokens"] + acc
    dec.close()
    return worst


@pytest.mark.parametrize("name", list(SMALL))
def test_bf16_small_models_teacher_forced(lib, name):
    dims = SMALL[name]
    w = synth.model_weights(dims, seed=3)
    p = synth.uniform_tokens(40, dims.vocab, seed=4)
    run_teacher_forced(lib, w, p, N=4, W=5, G=3, steps=4)


def test_bf16_long_prompt_spans_chunks(lib):
    """300-token prompt: three prefill chunks, three prefix attention chunks."""
    dims = SMALL["gqa-hd128"]
    w = synth.model_weights(dims, seed=5)
    p = synth.uniform_tokens(300, dims.vocab, seed=6)
    run_teacher_forced(lib, w, p, N=5, W=7, G=7, steps=3)


def test_bf16_repetitive_prompt_accepts(lib):
    dims = SMALL["mha-hd64"]
    w = synth.model_weights(dims, seed=7)
    p = np.tile(synth.uniform_tokens(12, dims.vocab, seed=8), 6)
    run_teacher_forced(lib, w, p, N=4, W=4, G=4, steps=6, par=True)


def test_bf16_wide_step_rows(lib):
    """M = 1 + (15 + 15) * 4 = 121 rows (the 7B step's shape) on a small model."""
    dims = SMALL["mha-hd128-3l"]
    w = synth.model_weights(dims, seed=9)
    p = synth.uniform_tokens(64, dims.vocab, seed=10)
    run_teacher_forced(lib, w, p, N=5, W=15, G=15, steps=2)


def test_graph_replay_matches_direct_launches(lib):
    """Steps after the first replay a captured CUDA graph; a profiled decoder
    launches every kernel directly.  Both run the same kernels with the same
    arguments, so tokens and logits must agree bit for bit."""
    dims = SMALL["gqa-hd128"]
    w = synth.model_weights(dims, 11)
    prompt = synth.uniform_tokens(40, dims.vocab, 11, 5)
    outs = []
    for profile in (False, True):
        dec = lib.Decoder(w, 4, 5, 4, 512, profile=profile)
        dec.prefill(prompt)
        toks, logits = [], []
        for _ in range(6):
            toks.append(list(dec.step()))
            logits.append(dec.debug_logits().copy())
        dec.close()
        outs.append((toks, logits))
    assert outs[0][0] == outs[1][0]
    for a, b in zip(outs[0][1], outs[1][1]):
        assert np.array_equal(a, b)


def test_ar_step_bf16_matches_oracle(lib):
    """la_ar_step on a bf16 decoder: each step's logits within 2e-2 of the
    oracle's last-row logits, tokens equal where the margin exceeds 0.05."""
    from oracle import decoder
    dims = SMALL["gqa-hd128"]
    w = synth.model_weights(dims, 13)
    p = [int(t) for t in synth.uniform_tokens(40, dims.vocab, 13, 7)]
    dec = lib.Decoder(w, 4, 5, 4, 256)
    toks = list(p) + [dec.prefill(p)]
    for _ in range(6):
        y = dec.ar_step()
        ref, _ = decoder.forward(w, toks, np.arange(len(toks)), decoder.causal_mask(0, len(toks)),
                                 logit_rows=[len(toks) - 1])
        err = float(np.max(np.abs(dec.debug_logits()[0] - ref[0])))
        assert err <= LOGIT_TOL_BF16, f"logits max-abs {err}"
        if top2_margin(ref[0]) > MARGIN:
            assert y == la.argmax_lowest(ref[0])
        toks.append(y)
    dec.close()
