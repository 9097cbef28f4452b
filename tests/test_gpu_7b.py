"""Full-size parity on the LLaMA-2-7B-shaped bf16 workload (32 layers, d 4096,
32 x 128 heads, FFN 11008, vocab 32000, 256-token prompt, N=5 W=15 G=15): the
GPU step that bench.py times vs the fp64 oracle, on one teacher-forced step.
Logits of all 76 used rows within 2e-2; tokens exact where the oracle margin
exceeds 0.05; pool exact.  Takes about a minute of host time (oracle)."""
import time

import numpy as np
import pytest

import synth
from helpers import MARGIN, ensure_built, top2_margin
from oracle import decoder, lookahead as la

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
LOGIT_TOL_BF16 = 2e-2


def test_7b_step_matches_oracle():
    ensure_built()
    import exact_decoding_gb300 as e
    wl = synth.WORKLOADS["llama7b-bf16-greedy"]
    w = synth.model_weights(wl.dims, wl.seed)
    prompt = synth.prompt(wl)
    dec = e.Decoder(w, wl.N, wl.W, wl.G, wl.max_seq)
    y1 = dec.prefill(prompt)
    pre = dec.debug_logits()[0]
    dec.step()
    s0 = dec.export_state()
    acc = dec.step()
    logits = dec.debug_logits()
    s1 = dec.export_state()
    dec.close()

    t = time.time()
    orc = la.Lookahead(w, wl.N, wl.W, wl.G, keep_logits=True)
    orc.load_state(s0["tokens"], s0["window"], s0["records"])
    acc_ref = orc.step()
    rec = orc.history[-1]
    print(f"oracle step: {time.time() - t:.1f} s")
    err = float(np.max(np.abs(logits - rec.logits)))
    print(f"7B step logits max-abs error {err:.4g} over {logits.shape}")
    assert err <= LOGIT_TOL_BF16
    decisive = [0] + [1 + wl.W + i for i in range(wl.G * (wl.N - 1))]
    if not any(top2_margin(rec.logits[i]) <= MARGIN for i in decisive):
        assert acc == acc_ref
    for j in range(wl.W):
        if top2_margin(rec.logits[1 + j]) > MARGIN:
            assert int(s1["window"][wl.N - 2, j]) == rec.new[j]
    pool = la.Pool.from_records(orc.pool.cap, s0["records"])
    for key, suf in la.harvest(np.asarray(s0["window"]), [int(x) for x in s1["window"][wl.N - 2]]):
        pool.insert(key, suf)
    assert pool.records() == s1["records"]
    # prefill's last-row logits against the oracle's prefix pass
    P = len(prompt)
    ref_pre, _ = decoder.forward(w, list(prompt), np.arange(P), decoder.causal_mask(0, P), logit_rows=[P - 1])
    assert float(np.max(np.abs(pre - ref_pre[0]))) <= LOGIT_TOL_BF16
    if top2_margin(ref_pre[0]) > MARGIN:
        assert y1 == la.argmax_lowest(ref_pre[0])
