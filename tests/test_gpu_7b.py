"""Full-size parity on the LLaMA-2-7B-shaped bf16 workload (32 layers, d 4096,
32 x 128 heads, FFN 11008, vocab 32000, 256-token prompt, N=5 W=15 G=15): the
GPU step that bench.py times vs the fp64 oracle, teacher-forced.  Logits of
all 76 used rows within 2e-2; the accepted tokens exact whenever every row
the oracle's verification read has a top-1/top-2 margin above 0.05 (the test
steps until one such step has been compared, at most three); new lookahead
tokens exact per column under the same rule; pool exact.  About a minute of
host time per oracle step."""
import time

import numpy as np
import pytest

import synth
from helpers import MARGIN, Tally, check_step, ensure_built, top2_margin
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
    tally = Tally()
    orc = la.Lookahead(w, wl.N, wl.W, wl.G, keep_logits=True)
    for t in range(3):
        s0 = dec.export_state()
        acc = dec.step()
        logits = dec.debug_logits()
        s1 = dec.export_state()
        t0 = time.time()
        orc.load_state(s0["tokens"], s0["window"], s0["records"])
        acc_ref = orc.step()
        print(f"oracle step: {time.time() - t0:.1f} s")
        check_step(orc.history[-1], acc, acc_ref, logits, s0, s1, wl.N, wl.W, MARGIN, LOGIT_TOL_BF16, orc.pool.cap,
                   la.FIFO, tally, where=f"7B step {t + 2}")
        print(tally)
        if tally.accept_compared:
            break
    dec.close()
    assert tally.accept_compared >= 1, tally
    assert 2 * tally.columns_compared >= tally.columns, tally
    # prefill's last-row logits against the oracle's prefix pass
    P = len(prompt)
    ref_pre, _ = decoder.forward(w, list(prompt), np.arange(P), decoder.causal_mask(0, P), logit_rows=[P - 1])
    assert float(np.max(np.abs(pre - ref_pre[0]))) <= LOGIT_TOL_BF16
    if top2_margin(ref_pre[0]) > MARGIN:
        assert y1 == la.argmax_lowest(ref_pre[0])
