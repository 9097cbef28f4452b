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
