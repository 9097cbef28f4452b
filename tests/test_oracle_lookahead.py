"""Pins of the oracle's lookahead method: the mask against brute force, the
pages' worked examples and tables, Algorithm 3 cases, the lossless
invariant, pool replay, KV recompute and the progress bound."""
import json
import os
from fractions import Fraction
from itertools import product

import numpy as np
import pytest

import synth
from oracle import decoder, lookahead as la, philox

from conftest import GOLDEN


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("N,W,G", [(2, 1, 0), (2, 3, 2), (3, 4, 4), (4, 5, 2), (5, 15, 15), (5, 5, 5)])
def test_mask_closed_form_equals_brute_force(N, W, G):
    rows = la.step_rows(N, W, G)
    mask = la.step_mask(N, W, G)
    for r in range(len(rows)):
        brute = set(la.ancestors(rows, r)) | {r}
        assert set(np.nonzero(mask[r])[0]) == brute


@pytest.mark.parametrize("N,W,G", [(3, 4, 4), (4, 5, 2), (5, 7, 7)])
def test_mask_structure(N, W, G):
    """Causal in position, no edges between the branches or between two
    candidates, lookahead rows see their column history and the oldest
    level's left context."""
    rows = la.step_rows(N, W, G)
    mask = la.step_mask(N, W, G)
    for r, s in product(range(len(rows)), repeat=2):
        if not mask[r, s] or r == s:
            continue
        assert rows[s].depth < rows[r].depth
        if s != 0:
            assert rows[r].kind == rows[s].kind
            if rows[r].kind == "cand":
                assert rows[r].a == rows[s].a
    for k in range(N - 1):
        for j in range(W):
            r = la.look_row(N, W, k, j)
            seen = {(rows[s].a, rows[s].b) for s in np.nonzero(mask[r])[0] if rows[s].kind == "look"}
            want = {(kk, j) for kk in range(k + 1)} | {(0, jj) for jj in range(j)}
            assert seen == want


def test_table4_extra_tokens():
    for case in _load("table4_rows.json")["cases"]:
        rows = la.step_rows(case["N"], case["W"], case["G"])
        assert len(rows) - 1 == case["extra"]


def test_fig1_ngram_is_a_diagonal():
    g = _load("fig1_ngram.json")
    N, W = g["N"], g["W"]
    rows = la.step_rows(N, W, g["G"])
    window = np.zeros((N - 1, W), dtype=np.int64)
    for k in range(N - 1):
        for j in range(W):
            depth = rows[la.look_row(N, W, k, j)].depth
            window[k, j] = 100 * (k + 1) + depth
    new = [100 * N + rows[la.look_row(N, W, N - 2, j)].depth + 1 for j in range(W)]
    grams = [(key,) + suf for key, suf in la.harvest(window, new)]
    assert tuple(g["example_ngram"]) in grams


def test_alg3_golden_cases():
    for case in _load("alg3_cases.json")["cases"]:
        cands = [tuple(c) for c in case["cands"]]
        acc, win = la.greedy_verify(cands, case["row0"], lambda c, m: case["cand"][c][m - 1])
        assert acc == case["accepted"], case["name"]
        assert win == case["winner"], case["name"]
        assert 1 <= len(acc) <= case["N"]


def test_pool_fifo_and_dedup():
    p = la.Pool(cap=3)
    p.insert(7, (1, 2))
    p.insert(7, (3, 4))
    p.insert(7, (1, 2))            # present: no-op, order unchanged
    assert p.lookup(7, 10) == [(1, 2), (3, 4)]
    p.insert(7, (5, 6))
    p.insert(7, (8, 9))            # over capacity: oldest (1, 2) leaves
    assert p.lookup(7, 10) == [(3, 4), (5, 6), (8, 9)]
    assert p.lookup(7, 2) == [(3, 4), (5, 6)]
    p.insert(1, (0, 0))
    assert p.records() == [(1, (0, 0)), (7, (3, 4)), (7, (5, 6)), (7, (8, 9))]
    assert p.lookup(99, 4) == []


def test_pool_lru_hand_example():
    """Reading R15 worked by hand: a repeated harvest and a use move an entry
    to the most recent end; a full list drops its least recently used entry;
    lookup is most recent first."""
    p = la.Pool(cap=3, policy=la.LRU)
    p.insert(7, (1, 2))
    p.insert(7, (3, 4))
    p.insert(7, (5, 6))
    p.insert(7, (1, 2))            # met again: (1, 2) becomes the most recent
    assert p.records() == [(7, (3, 4)), (7, (5, 6)), (7, (1, 2))]
    p.insert(7, (8, 9))            # full: the least recently used (3, 4) leaves
    assert p.lookup(7, 10) == [(8, 9), (1, 2), (5, 6)]
    assert p.lookup(7, 2) == [(8, 9), (1, 2)]
    p.use(7, (5, 6))
    assert p.lookup(7, 10) == [(5, 6), (8, 9), (1, 2)]
    p.insert(7, (0, 1))            # now (1, 2) is the least recently used
    assert p.lookup(7, 10) == [(0, 1), (5, 6), (8, 9)]
    # the same operations under FIFO: neither the repeat nor the use reorders
    f = la.Pool(cap=3)
    for suf in [(1, 2), (3, 4), (5, 6), (1, 2), (8, 9)]:
        f.insert(7, suf)
    f.use(7, (5, 6))
    f.insert(7, (0, 1))
    assert f.lookup(7, 10) == [(5, 6), (8, 9), (0, 1)]


class _StampLRU:
    """LRU written another way: every entry carries the time of its last
    use; the list is the entries by ascending time, and a full key drops the
    entry with the smallest time."""

    def __init__(self, cap):
        self.cap, self.t, self.stamp = cap, 0, {}

    def touch(self, key, suf):
        self.t += 1
        ent = self.stamp.setdefault(key, {})
        if suf not in ent and len(ent) == self.cap:
            del ent[min(ent, key=ent.get)]
        ent[suf] = self.t

    def records(self):
        return [(k, s) for k in sorted(self.stamp) for s in sorted(self.stamp[k], key=self.stamp[k].get)]


@pytest.mark.parametrize("cap,seed", [(1, 0), (2, 1), (3, 2), (5, 3)])
def test_pool_lru_equals_timestamp_model(cap, seed):
    rng = np.random.default_rng(seed)
    p, ref = la.Pool(cap, la.LRU), _StampLRU(cap)
    for _ in range(400):
        key, suf = int(rng.integers(0, 3)), (int(rng.integers(0, 4)), int(rng.integers(0, 3)))
        if rng.random() < 0.3 and p.lists.get(key):
            suf = p.lists[key][int(rng.integers(0, len(p.lists[key])))]
            p.use(key, suf)
        else:
            p.insert(key, suf)
        ref.touch(key, suf)
        assert p.records() == ref.records()
    for key in range(3):
        assert p.lookup(key, 2) == [s for k, s in reversed(ref.records()) if k == key][:2]


@pytest.mark.parametrize("N,W,G,cap", [(4, 3, 4, 0), (3, 4, 2, 3), (5, 2, 3, 2)])
def test_lru_pool_lossless_and_replay(tiny, N, W, G, cap):
    """With the LRU pool greedy lookahead still equals greedy autoregressive
    decoding, and the pool after the run equals the timestamp model fed the
    prompt's n-grams, then per step the winner's use and the harvest."""
    wl, w, _ = tiny
    chunk = synth.uniform_tokens(6, wl.dims.vocab, seed=4)
    p = np.tile(chunk, 5)
    ar = la.generate_ar(w, p, 40)
    o = la.Lookahead(w, N, W, G, prompt_as_reference=True, pool_cap=cap, pool_policy=la.LRU)
    out, _ = o.generate(p, 40)
    assert out == ar
    ref = _StampLRU(o.pool.cap)
    for i in range(len(p) - N + 1):
        ref.touch(int(p[i]), tuple(int(t) for t in p[i + 1:i + N]))
    used = 0
    for rec in o.history:
        assert rec.cands == [s for k, s in reversed(ref.records()) if k == rec.o][:G]
        if rec.winner >= 0:
            ref.touch(rec.o, rec.cands[rec.winner])
            used += 1
        for j in range(W):
            ref.touch(int(rec.window_before[0, j]),
                      tuple(int(rec.window_before[k, j]) for k in range(1, N - 1)) + (rec.new[j],))
    assert used > 0
    assert o.pool.records() == ref.records()


def test_pool_lfu_hand_example():
    """Reading R16 worked by hand: uses raise an entry's count; a full list
    drops the entry with the fewest uses (the oldest among equals) before the
    new one enters; lookup is most used first."""
    p = la.Pool(cap=3, policy=la.LFU)
    p.insert(7, (1, 2))
    p.insert(7, (3, 4))
    p.insert(7, (5, 6))
    p.insert(7, (1, 2))            # met again: (1, 2) has 1 use
    p.use(7, (3, 4))
    p.use(7, (3, 4))               # (3, 4) has 2 uses
    assert p.records() == [(7, (5, 6)), (7, (1, 2)), (7, (3, 4))]
    assert p.use_counts() == [0, 1, 2]
    p.insert(7, (8, 9))            # full: (5, 6) (no uses) leaves, (8, 9) enters with none
    assert p.lookup(7, 10) == [(3, 4), (1, 2), (8, 9)]
    p.insert(7, (0, 1))            # (8, 9) is now the least used: it leaves at once
    assert p.lookup(7, 10) == [(3, 4), (1, 2), (0, 1)]
    p.use(7, (0, 1))               # one use each for (0, 1) and (1, 2); (0, 1) more recent
    assert p.lookup(7, 2) == [(3, 4), (0, 1)]
    p.insert(7, (2, 2))            # (1, 2): 1 use, older than (0, 1)
    assert p.records() == [(7, (2, 2)), (7, (0, 1)), (7, (3, 4))]
    assert p.use_counts() == [0, 1, 2]


class _StampLFU:
    """LFU written another way: every entry carries (uses, time of last use
    or entry); a full key drops the entry with the smallest pair, found by a
    search, and the list is the entries by ascending pair."""

    def __init__(self, cap):
        self.cap, self.t, self.ent = cap, 0, {}

    def touch(self, key, suf):
        self.t += 1
        ent = self.ent.setdefault(key, {})
        if suf in ent:
            ent[suf] = (ent[suf][0] + 1, self.t)
            return
        if len(ent) == self.cap:
            del ent[min(ent, key=ent.get)]
        ent[suf] = (0, self.t)

    def records(self):
        return [(k, s) for k in sorted(self.ent) for s in sorted(self.ent[k], key=self.ent[k].get)]

    def uses(self):
        return [self.ent[k][s][0] for k, s in self.records()]


@pytest.mark.parametrize("cap,seed", [(1, 0), (2, 1), (3, 2), (5, 3)])
def test_pool_lfu_equals_search_model(cap, seed):
    rng = np.random.default_rng(seed)
    p, ref = la.Pool(cap, la.LFU), _StampLFU(cap)
    for _ in range(400):
        key, suf = int(rng.integers(0, 3)), (int(rng.integers(0, 4)), int(rng.integers(0, 3)))
        if rng.random() < 0.3 and p.lists.get(key):
            suf = p.lists[key][int(rng.integers(0, len(p.lists[key])))]
            p.use(key, suf)
        else:
            p.insert(key, suf)
        ref.touch(key, suf)
        assert p.records() == ref.records()
        assert p.use_counts() == ref.uses()
    # a snapshot (records in eviction order with their counts) rebuilds the same pool
    q = la.Pool.from_records(cap, p.records(), la.LFU, p.use_counts())
    assert q.records() == p.records() and q.use_counts() == p.use_counts()
    for key in range(3):
        assert q.lookup(key, 2) == p.lookup(key, 2)


def test_pool_policies_agree_at_cap_one():
    """With one suffix per key every policy keeps the last suffix seen."""
    rng = np.random.default_rng(5)
    pools = [la.Pool(1, pol) for pol in (la.FIFO, la.LRU, la.LFU)]
    for _ in range(300):
        key, suf = int(rng.integers(0, 4)), (int(rng.integers(0, 3)),)
        for p in pools:
            p.insert(key, suf)
        assert pools[0].records() == pools[1].records() == pools[2].records()


@pytest.mark.parametrize("N,W,G,cap", [(4, 3, 4, 0), (4, 3, 2, 5), (3, 4, 3, 3)])
def test_lfu_pool_lossless_and_replay(tiny, N, W, G, cap):
    """With the LFU pool greedy lookahead still equals greedy autoregressive
    decoding, and the pool after the run equals the search model fed the
    prompt's n-grams, then per step the winner's use and the harvest."""
    wl, w, _ = tiny
    chunk = synth.uniform_tokens(6, wl.dims.vocab, seed=4)
    p = np.tile(chunk, 5)
    ar = la.generate_ar(w, p, 40)
    o = la.Lookahead(w, N, W, G, prompt_as_reference=True, pool_cap=cap, pool_policy=la.LFU)
    out, _ = o.generate(p, 40)
    assert out == ar
    ref = _StampLFU(o.pool.cap)
    for i in range(len(p) - N + 1):
        ref.touch(int(p[i]), tuple(int(t) for t in p[i + 1:i + N]))
    used = 0
    for rec in o.history:
        assert rec.cands == [s for k, s in reversed(ref.records()) if k == rec.o][:G]
        if rec.winner >= 0:
            ref.touch(rec.o, rec.cands[rec.winner])
            used += 1
        for j in range(W):
            ref.touch(int(rec.window_before[0, j]),
                      tuple(int(rec.window_before[k, j]) for k in range(1, N - 1)) + (rec.new[j],))
    assert used > 0
    assert o.pool.records() == ref.records() and o.pool.use_counts() == ref.uses()


@pytest.mark.parametrize("N,W,G,par", [(3, 4, 4, False), (2, 3, 3, False), (4, 2, 5, False),
                                       (5, 3, 0, False), (3, 1, 2, True), (4, 4, 4, True)])
def test_lossless_vs_autoregressive(tiny, N, W, G, par):
    """Greedy lookahead output == greedy autoregressive output (fp64)."""
    wl, w, p = tiny
    ar = la.generate_ar(w, p, 48)
    o = la.Lookahead(w, N, W, G, prompt_as_reference=par)
    out, steps = o.generate(p, 48)
    assert out == ar
    acc_lens = [len(r.accepted) for r in o.history]
    assert all(1 <= a <= N for a in acc_lens)
    assert 1 + sum(acc_lens) == len(o.tokens) - len(p)
    if G == 0:
        assert steps == 47


def test_lossless_repetitive_prompt(tiny):
    """A repeated prompt with prompt-as-reference: candidates get accepted."""
    wl, w, _ = tiny
    chunk = synth.uniform_tokens(8, wl.dims.vocab, seed=9)
    p = np.tile(chunk, 5)
    ar = la.generate_ar(w, p, 40)
    o = la.Lookahead(w, 4, 3, 4, prompt_as_reference=True)
    out, steps = o.generate(p, 40)
    assert out == ar


def test_pool_replay_from_window_trajectory(tiny):
    """The pool after each step equals the n-grams read off the logged window
    trajectory (plus the prompt's, when seeded), replayed in order."""
    wl, w, p = tiny
    N, W, G = 4, 3, 3
    o = la.Lookahead(w, N, W, G, prompt_as_reference=True, pool_cap=2)
    o.prefill(p)
    for _ in range(12):
        o.step()
    grams = [(int(p[i]), tuple(int(t) for t in p[i + 1:i + N])) for i in range(len(p) - N + 1)]
    for t, rec in enumerate(o.history):
        # the window a step starts from is the previous window slid by the previous new tokens
        if t:
            prev = o.history[t - 1]
            np.testing.assert_array_equal(rec.window_before[:-1], prev.window_before[1:])
            np.testing.assert_array_equal(rec.window_before[-1], prev.new)
        for j in range(W):
            grams.append((int(rec.window_before[0, j]),
                          tuple(int(rec.window_before[k, j]) for k in range(1, N - 1)) + (rec.new[j],)))
    lists = {}
    for key, suf in grams:
        lst = lists.setdefault(key, [])
        if suf not in lst:
            lst.append(suf)
            del lst[:-2]
    assert sorted((k, s) for k, v in lists.items() for s in v) == sorted(o.pool.records())
    assert [(k, s) for k in sorted(lists) for s in lists[k]] == o.pool.records()


def test_kv_after_steps_equals_fresh_prefill(tiny):
    wl, w, p = tiny
    o = la.Lookahead(w, 3, 4, 4)
    o.prefill(p)
    for _ in range(6):
        o.step()
    P = o.P
    _, fresh = decoder.forward(w, o.tokens[:P], np.arange(P), decoder.causal_mask(0, P))
    for (k1, v1), (k2, v2) in zip(o.cache, fresh):
        np.testing.assert_allclose(k1, k2, atol=1e-12)
        np.testing.assert_allclose(v1, v2, atol=1e-12)


def test_window_init_and_splitmix():
    g = _load("splitmix64.json")
    x, outs = g["seed"], []
    for _ in range(2):
        outs.append(str(la.splitmix64(x)))
        x = (x + 0x9E3779B97F4A7C15) % 2 ** 64
    assert outs == g["outputs"]
    prompt = list(range(100, 137))
    V = la.init_window(prompt, 4, 5, seed=3)
    assert V.shape == (3, 5)
    for k in range(3):
        for j in range(5):
            assert V[k, j] == prompt[la.splitmix64(3 ^ (k * 5 + j)) % len(prompt)]


def test_philox_known_answers():
    for case in _load("philox_kat.json")["cases"]:
        out = philox.philox4x32_10([int(c, 16) for c in case["ctr"]], [int(c, 16) for c in case["key"]])
        assert out == [int(c, 16) for c in case["out"]]
        # and the input generator's C implementation
        assert synth.philox4x32_10([int(c, 16) for c in case["ctr"]], [int(c, 16) for c in case["key"]]) == out


def test_inverse_cdf_exact_frequencies():
    w = np.array([0.1, 0.0, 0.2, 0.3, 0.4])
    counts = np.zeros(5, int)
    for k in range(1000):
        counts[la.inverse_cdf(w, (k + 0.5) / 1000)] += 1
    assert counts.tolist() == [100, 0, 200, 300, 400]


def _exact_rejection_chain(p, tokens):
    """Probability of each output token for one depth of Algorithm 4, by
    exact enumeration over accept/reject outcomes (rational arithmetic)."""
    out = {x: Fraction(0) for x in range(len(p))}

    def rec(dist, i, prob, rejected):
        while i < len(tokens) and tokens[i] in rejected:
            i += 1
        if i == len(tokens):
            tot = sum(dist)
            for x in range(len(dist)):
                out[x] += prob * dist[x] / tot
            return
        x = tokens[i]
        px = dist[x] / sum(dist)
        out[x] += prob * px
        nd = list(dist)
        nd[x] = Fraction(0)
        rec(nd, i + 1, prob * (1 - px), rejected | {x})

    rec([Fraction(v) for v in p], 0, Fraction(1), frozenset())
    return out


@pytest.mark.parametrize("tokens", [[0], [3, 1], [2, 2, 5], [1, 4, 6, 7, 0]])
def test_sampling_rule_preserves_distribution_exactly(tokens):
    """Appendix B's claim for one depth: with greedy (one-hot) drafts the
    output token is distributed exactly as the model's distribution."""
    p = [Fraction(k, 36) for k in (1, 2, 3, 4, 5, 6, 7, 8)]
    got = _exact_rejection_chain(p, tokens)
    assert all(got[x] == p[x] for x in range(8))


def test_sampling_verify_joint_distribution_monte_carlo():
    """The oracle's Algorithm 4 over two depths: first two output tokens are
    distributed as p(x1) q_x1(x2), by a chi-square test over seeds."""
    V = 4
    p = np.array([0.1, 0.2, 0.3, 0.4])
    q = np.array([[0.25, 0.25, 0.25, 0.25], [0.7, 0.1, 0.1, 0.1], [0.05, 0.05, 0.1, 0.8], [0.3, 0.3, 0.2, 0.2]])
    cands = [(2, 3), (3, 0), (2, 1)]
    counts = np.zeros((V, V))
    n = 20000
    for seed in range(n):
        acc, _ = la.sampling_verify(cands, p, lambda c, m: q[cands[c][0]], P=5, seed=seed, N=3)
        if len(acc) >= 2:
            counts[acc[0], acc[1]] += 1
        else:
            # stopped after one token: the next token would come from q[x1] in the following step
            x1 = acc[0]
            x2 = la.inverse_cdf(q[x1], philox.uniform(seed + 10 ** 6, 0, 0))
            counts[x1, x2] += 1
    expect = n * p[:, None] * q
    chi2 = np.sum((counts - expect) ** 2 / expect)
    assert chi2 < 45.0, chi2   # 15 dof: p < 1e-4 false-alarm rate


def test_sampling_progress_bounds(tiny):
    wl, w, p = tiny
    o = la.Lookahead(w, 3, 4, 4, temperature=1.0, seed=11, prompt_as_reference=True)
    out, steps = o.generate(np.tile(p[:8], 4), 32)
    assert len(out) == 32
    for rec in o.history:
        assert 1 <= len(rec.accepted) <= 3


# ---------------------------------------------------------------- top-k / top-p (reading R14)
def test_filter_top_hand_examples():
    """Hand-worked cases on binary fractions: ranking by probability with ties
    to the lower id, top-k keeps the first k, top-p keeps the prefix whose
    mass first reaches p (crossing token included), top-p acts on the
    renormalised top-k set."""
    d = np.array([0.125, 0.375, 0.25, 0.125, 0.125])   # ranked ids: 1, 2, 0, 3, 4
    keep = lambda out: [v for v in range(len(out)) if out[v] > 0]
    assert keep(la.filter_top(d, 1)) == [1]
    assert keep(la.filter_top(d, 3)) == [0, 1, 2]                 # tie 0/3/4 at 0.125: id 0
    assert keep(la.filter_top(d, 4)) == [0, 1, 2, 3]
    assert keep(la.filter_top(d, 0, 0.375)) == [1]                # reaches p exactly
    assert keep(la.filter_top(d, 0, 0.376)) == [1, 2]             # crossing token kept
    assert keep(la.filter_top(d, 0, 0.75)) == [0, 1, 2]
    assert keep(la.filter_top(d, 0, 0.76)) == [0, 1, 2, 3]
    assert keep(la.filter_top(d, 2, 0.61)) == [1, 2]              # renormalised top-2: 0.6, 0.4
    assert keep(la.filter_top(d, 2, 0.59)) == [1]
    assert np.array_equal(la.filter_top(d, 0, 1.0), d)
    assert np.array_equal(la.filter_top(d, 5, 1.0), d)


@pytest.mark.parametrize("top_k,top_p,tokens", [(3, 1.0, [4, 7, 2]), (0, 0.5, [7, 6, 0]), (5, 0.8, [1, 7, 6, 5])])
def test_sampling_rule_preserves_filtered_distribution_exactly(top_k, top_p, tokens):
    """With top-k / top-p the rejection chain runs on the filtered
    distribution, so the output follows that distribution exactly."""
    p = [Fraction(k, 36) for k in (1, 2, 3, 4, 5, 6, 7, 8)]
    f = la.filter_top(np.array([float(x) for x in p]), top_k, top_p)
    pf = [p[v] if f[v] > 0 else Fraction(0) for v in range(8)]
    tot = sum(pf)
    got = _exact_rejection_chain(pf, tokens)
    assert all(got[x] == pf[x] / tot for x in range(8))


def test_top_k1_sampling_equals_greedy(tiny):
    """top_k = 1 leaves one token per row: lookahead sampling at T = 1 must
    reproduce greedy autoregressive decoding token for token."""
    wl, w, p = tiny
    ref = la.generate_ar(w, p, 20)
    o = la.Lookahead(w, 3, 4, 4, temperature=1.0, seed=5, top_k=1)
    out, _ = o.generate(p, 20)
    assert out == ref


def test_verification_reads_the_rows_of_the_matching_candidate(tiny):
    """A pool candidate equal to the model's greedy continuation is accepted
    whole (A = N, Algorithm 3 with every token matching), the step's tokens
    equal plain greedy decoding, and the rows the verification reads are row
    0 and that candidate's N-1 rows (a non-matching candidate ahead of it is
    read at depth 1 only through row 0)."""
    wl, w, p = tiny
    N, W, G = 4, 2, 3
    prompt = [int(t) for t in p[:20]]
    ar = la.generate_ar(w, prompt, N + 1)
    o = ar[0]
    good = tuple(ar[1:N])                              # the N-1 tokens greedy decoding emits after o
    bad = tuple((t + 1) % wl.dims.vocab for t in good)
    orc = la.Lookahead(w, N, W, G, keep_logits=True)
    window = la.init_window(prompt, N, W, 0)
    orc.load_state(prompt + [o], window, [(o, bad), (o, good)])
    acc = orc.step()
    rec = orc.history[-1]
    assert acc == ar[1:N + 1]
    assert rec.winner == 1
    used = la.used_rows(N, W, G)
    assert rec.decisive == [0] + [used.index(la.cand_row(N, W, 1, m)) for m in range(1, N)]
