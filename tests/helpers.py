"""Shared test helpers: margin rule, library build, oracle runners."""
import numpy as np

# Token decisions must match exactly wherever the oracle's top-1 / top-2 logit
# margin exceeds this.  bf16 models: 0.05.  fp32 models: twice the 1e-4 logit
# tolerance, a stricter rule (the GPU and the oracle differ by ~1e-6 there).
MARGIN = 0.05
MARGIN_F32 = 2e-4


def top2_margin(row: np.ndarray) -> float:
    part = np.partition(np.asarray(row, dtype=np.float64), -2)
    return float(part[-1] - part[-2])


def ensure_built():
    import synth
    from exact_decoding_gb300 import build
    synth.build_generator()
    build.build()


def ar_with_margins(weights, prompt, max_new, dtype=np.float64):
    """Greedy AR tokens and the top-1/top-2 margin of each decision (oracle)."""
    from oracle import decoder, lookahead as la
    prompt = [int(t) for t in prompt]
    s = len(prompt)
    logits, cache = decoder.forward(weights, prompt, np.arange(s), decoder.causal_mask(0, s), dtype=dtype,
                                    logit_rows=[s - 1])
    out, margins = [la.argmax_lowest(logits[0])], [top2_margin(logits[0])]
    while len(out) < max_new:
        P = s + len(out) - 1
        logits, kv = decoder.forward(weights, [out[-1]], np.array([P]), np.ones((1, P + 1), bool), cache=cache,
                                     dtype=dtype)
        cache = decoder.concat_cache(cache, kv)
        out.append(la.argmax_lowest(logits[0]))
        margins.append(top2_margin(logits[0]))
    return out, margins


def compare_stream(gpu, ref, margins, margin=MARGIN):
    """Tokens must agree up to the first oracle decision with margin <= `margin`."""
    for i, (a, b) in enumerate(zip(gpu, ref)):
        if margins[i] <= margin:
            return i
        assert a == b, f"token {i}: gpu {a} vs oracle {b} (oracle margin {margins[i]:.4f})"
    return len(ref)


class Tally:
    """What a teacher-forced run actually compared, so tests can assert floors."""

    def __init__(self):
        self.steps = 0
        self.accept_compared = 0        # steps whose accepted tokens were compared exactly
        self.accept_compared_multi = 0  # ... of which accepted more than one token (A > 1)
        self.columns = 0                # lookahead columns checked
        self.columns_compared = 0       # ... whose new token was compared exactly
        self.hits = 0                   # steps with a winning candidate (GPU side)
        self.worst = 0.0                # largest logits max-abs error

    def __repr__(self):
        return (f"Tally(steps={self.steps}, accept_compared={self.accept_compared}, "
                f"accept_compared_multi={self.accept_compared_multi}, columns={self.columns_compared}/"
                f"{self.columns}, hits={self.hits}, worst={self.worst:.3g})")


def check_step(rec, acc, acc_ref, logits, s0, s1, N, W, margin, tol, pool_cap, policy, tally, where="",
               greedy=True, uses0=None, uses1=None):
    """Compare one GPU step with the oracle's step from the same state.

    rec       -- the oracle's StepRecord (keep_logits=True)
    acc       -- GPU accepted tokens; acc_ref the oracle's
    logits    -- GPU used-row logits
    s0, s1    -- GPU states exported before and after the step
    Checks: logits within tol; accepted tokens equal whenever every row the
    oracle's verification read (rec.decisive) has a top-1/top-2 margin above
    `margin` (greedy); new lookahead tokens equal per column under the same
    rule, else the GPU's token within `margin` of the oracle's max; the pool
    equals the oracle's replay of the GPU's own decisions; tokens appended.
    """
    from oracle import lookahead as la
    err = float(np.max(np.abs(logits - rec.logits)))
    tally.worst = max(tally.worst, err)
    assert err <= tol, f"{where}: logits max-abs {err}"
    tally.steps += 1
    if greedy:
        if all(top2_margin(rec.logits[i]) > margin for i in rec.decisive):
            assert acc == acc_ref, f"{where}: gpu {acc} vs oracle {acc_ref}"
            tally.accept_compared += 1
            tally.accept_compared_multi += len(acc) > 1
    else:
        # Sampling (reading R13): the decisions may differ only at a draw that
        # sits within 1e-3 of its threshold.  At a 32000-token vocabulary the
        # final inverse-CDF draw always lies that close to a token edge, so a
        # step counts as compared when the GPU and the oracle agree on it.
        if acc == acc_ref:
            tally.accept_compared += 1
            tally.accept_compared_multi += len(acc) > 1
        else:
            assert any(abs(d.value) <= 1e-3 for d in rec.trace), \
                f"{where}: gpu {acc} vs oracle {acc_ref} with no near-threshold decision"
    for j in range(W):
        lr = rec.logits[1 + j]
        gnew = int(s1["window"][N - 2, j])
        tally.columns += 1
        if top2_margin(lr) > margin:
            assert gnew == rec.new[j], f"{where} column {j}"
            tally.columns_compared += 1
        else:
            assert lr[gnew] >= lr.max() - margin, f"{where} column {j}: token off the near-tie"
    # Pool: replay the GPU's own decisions on the state it started from: the
    # winner (first candidate, in the oracle's lookup order, whose prefix is
    # the accepted candidate tokens) is used, then the harvest goes in.
    pool = la.Pool.from_records(pool_cap, s0["records"], policy, uses0)
    a = len(acc) - 1
    win = next((c for c, cand in enumerate(rec.cands) if a > 0 and list(cand[:a]) == acc[:a]), -1)
    if win >= 0:
        pool.use(s0["tokens"][-1], rec.cands[win])
        tally.hits += 1
    for key, suf in la.harvest(np.asarray(s0["window"]), [int(x) for x in s1["window"][N - 2]]):
        pool.insert(key, suf)
    assert pool.records() == s1["records"], f"{where}: pool"
    if uses1 is not None:
        assert pool.use_counts() == list(uses1), f"{where}: pool use counts"
    assert s1["tokens"] == s0["tokens"] + list(acc), f"{where}: committed tokens"


def teacher_forced(lib, w, prompt, N, W, G, steps, margin, tol, temperature=0.0, seed=0, par=False,
                   pool_policy="fifo", pool_cap=0, max_seq=1024, **kw):
    """Run `steps` GPU steps; before each, the oracle loads the GPU's exported
    state and runs the same step; check_step compares them.  Returns a Tally."""
    from oracle import lookahead as la
    dec = lib.Decoder(w, N, W, G, max_seq, temperature=temperature, seed=seed, prompt_as_reference=par,
                      pool_policy=pool_policy, pool_cap=pool_cap, **kw)
    dec.prefill(prompt)
    orc = la.Lookahead(w, N, W, G, temperature=temperature, seed=seed, prompt_as_reference=par, keep_logits=True,
                       pool_policy=pool_policy, pool_cap=pool_cap)
    tally = Tally()
    lfu = pool_policy == la.LFU
    for t in range(steps):
        s0 = dec.export_state()
        orc.load_state(s0["tokens"], s0["window"], s0["records"], s0.get("uses") if lfu else None)
        acc_ref = orc.step()
        rec = orc.history[-1]
        acc = dec.step()
        logits = dec.debug_logits()
        s1 = dec.export_state()
        check_step(rec, acc, acc_ref, logits, s0, s1, N, W, margin, tol, orc.pool.cap, pool_policy, tally,
                   where=f"step {t}", greedy=temperature == 0.0,
                   uses0=s0.get("uses") if lfu else None, uses1=s1.get("uses") if lfu else None)
    dec.close()
    return tally
