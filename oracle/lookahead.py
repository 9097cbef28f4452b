"""Lookahead decoding, written out plainly (oracle side).

Source: "Break the Sequential Dependency of LLM Inference Using Lookahead
Decoding" (arXiv 2402.02057), paper-graph-ui summary, section 3.4:
  * "The Lookahead Branch" -- the 2D window (W columns x N-1 past Jacobi
    levels), the per-column generation rule, n-gram harvesting, the slide;
  * "The Verification Branch" -- candidate selection by first token, greedy
    verification (Algorithm 3), sampling verification (Algorithm 4), greedy
    drafting in the lookahead branch;
  * "Integrated Forward Pass" -- one forward pass under the custom mask
    (Figure 2b), the n-gram pool as first-token -> list of suffixes.
Autoregressive greedy decoding (section 3.4, "The autoregressive system") is
the reference the method must reproduce exactly (lossless).

Readings taken where the pages are open:
  R1 Step rows.  Row 0 is the last committed token o at position P (the
     prefix [0, P) is cached).  Lookahead row (k, j), level k in [0, N-2],
     column j in [0, W-1], holds window token V[k][j] at position P+1+j+k.
     Candidate row (c, m), m in [1, N-1], holds suffix token m of candidate c
     at position P+m.  Row order: 0, then (k, j) at 1 + k*W + j, then (c, m)
     at 1 + (N-1)*W + c*(N-1) + (m-1).  Always G candidate slots; slots past
     the g found are padding (token 0) and are ignored.
  R2 Mask.  Each row has one parent: (0, j) -> (0, j-1), (0, 0) -> row 0,
     (k>=1, j) -> (k-1, j), (c, 1) -> row 0, (c, m) -> (c, m-1).  A row sees
     the cached prefix, itself and its ancestors; so a lookahead row sees its
     column's lower levels and the oldest level's earlier columns, and a
     candidate row sees its own n-gram's earlier tokens, never another branch.
  R3 Candidates are looked up (oldest first, at most G) before the forward
     pass, from the pool as it stood after the previous step.
  R4 Greedy verification picks, among candidates, the longest prefix that
     matches the model's argmax chain (lowest candidate index on ties) and
     appends the argmax after it: 1 <= A <= N tokens per step.
  R5 Harvest after verification: for each column j ascending, key V[0][j],
     suffix (V[1][j], ..., V[N-2][j], new_j), new_j = argmax of row (N-2, j).
  R6 Pool: per key a FIFO list of distinct suffixes, capacity `pool_cap`
     (default G); re-inserting a present suffix is a no-op; the oldest is
     dropped when full.
  R7 Window slides by one level every step whatever A is: V[k] <- V[k+1],
     V[N-2] <- new.  Initial window: V[k][j] = prompt[splitmix64(seed ^
     (k*W + j)) mod s].
  R8 Prompt-as-reference: after prefill insert (prompt[i], prompt[i+1..i+N-1])
     for i = 0..s-N ascending.
  R9 Argmax ties go to the lowest token id.
  R10 Sampling (Algorithm 4): rows' distributions softmax(logits / T); the
     lookahead branch stays argmax; candidates are tried in index order,
     skipping tokens already rejected at the same depth; a draw r accepts x
     when r <= dist(x), otherwise dist(x) <- 0 and dist is renormalised; if
     none is accepted, or after N-1 accepted tokens, one token is drawn from
     dist by inverse CDF (smallest id whose ascending cumulative mass exceeds
     u * total).  Draw index counts draws at the same position.
  R14 Top-k / top-p (the pages name them for sampling without an order or a
     tie rule): temperature first, then top-k, then top-p on the renormalised
     top-k distribution.  Tokens are ranked by probability, ties to the lower
     id; top-k keeps the first k; top-p keeps the shortest ranked prefix whose
     mass reaches p (the token that crosses p included).  Algorithm 4 then
     runs on the filtered distributions unchanged, so its output follows the
     filtered distribution exactly.
  R15 LRU pool (section 7, "Follow-Up Research This Work Enables", names
     LRU next to FIFO as an eviction policy the paper leaves open).  Each
     key's list is kept least recently used first.  An entry is used when a
     step accepts at least one of its tokens as the winning candidate, or
     when the harvest meets it again; a use moves it to the most recent
     end.  The winner's use is recorded after verification and before the
     harvest.  A new suffix is appended at the most recent end, and when
     the list is full the least recently used entry is dropped.  Lookup
     returns the G most recently used entries, most recent first.  Under
     FIFO (R6) neither a use nor a repeated harvest changes the order.
  R16 LFU pool (the same passage names frequency-based eviction).  The uses
     are R15's.  Each entry carries a use count (0 when it enters) and the
     time of its last use or entry; each key's list is ordered by (count,
     time) ascending.  A new suffix into a full list first drops the head
     (fewest uses, the oldest among equals), then enters.  Lookup returns
     the G entries at the tail end, highest (count, time) first.  The counts
     are part of the pool's state, so a snapshot carries them.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from . import decoder, philox

MASK64 = (1 << 64) - 1


# --------------------------------------------------------------------------
# Step rows and the attention mask (Figure 2b; reading R1, R2)
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Row:
    kind: str          # "root", "look", "cand"
    a: int             # look: level k; cand: candidate c
    b: int             # look: column j; cand: depth m (1..N-1)
    parent: int        # row index of the parent, -1 for root
    depth: int         # position offset from P


def step_rows(N: int, W: int, G: int) -> List[Row]:
    rows = [Row("root", 0, 0, -1, 0)]
    for k in range(N - 1):
        for j in range(W):
            if k == 0:
                parent = 0 if j == 0 else 1 + (j - 1)
            else:
                parent = 1 + (k - 1) * W + j
            rows.append(Row("look", k, j, parent, 1 + j + k))
    base = 1 + (N - 1) * W
    for c in range(G):
        for m in range(1, N):
            parent = 0 if m == 1 else base + c * (N - 1) + (m - 2)
            rows.append(Row("cand", c, m, parent, m))
    assert len(rows) == 1 + (W + G) * (N - 1)
    return rows


def look_row(N, W, k, j):
    return 1 + k * W + j


def cand_row(N, W, c, m):
    return 1 + (N - 1) * W + c * (N - 1) + (m - 1)


def used_rows(N: int, W: int, G: int) -> List[int]:
    """Rows whose logits the step reads: row 0, the top level, all candidates."""
    return [0] + [look_row(N, W, N - 2, j) for j in range(W)] + \
           [cand_row(N, W, c, m) for c in range(G) for m in range(1, N)]


def ancestors(rows: Sequence[Row], r: int) -> List[int]:
    """Brute force: walk the parent pointers."""
    out = []
    p = rows[r].parent
    while p >= 0:
        out.append(p)
        p = rows[p].parent
    return out


def sees(rows: Sequence[Row], r: int, s: int) -> bool:
    """Closed-form visibility of step row s from step row r (reading R2)."""
    if s == r or s == 0:
        return True
    A, B = rows[r], rows[s]
    if A.kind == "look" and B.kind == "look":
        return (B.b == A.b and B.a < A.a) or (B.a == 0 and B.b < A.b)
    if A.kind == "cand" and B.kind == "cand":
        return B.a == A.a and B.b < A.b
    return False


def step_mask(N: int, W: int, G: int) -> np.ndarray:
    """[M, M] visibility among step rows, built from the closed-form rule."""
    rows = step_rows(N, W, G)
    M = len(rows)
    return np.array([[sees(rows, r, s) for s in range(M)] for r in range(M)], dtype=bool)


# --------------------------------------------------------------------------
# n-gram pool (reading R6)
# --------------------------------------------------------------------------

FIFO, LRU, LFU = "fifo", "lru", "lfu"


class Pool:
    """First token -> list of distinct (N-1)-token suffixes, in eviction
    order (the next to be dropped first): oldest first under FIFO (R6),
    least recently used first under LRU (R15), fewest uses first under LFU
    (R16)."""

    def __init__(self, cap: int, policy: str = FIFO):
        assert policy in (FIFO, LRU, LFU)
        assert cap >= 1, "a key's list holds at least one suffix"
        self.cap = cap
        self.policy = policy
        self.lists: Dict[int, List[Tuple[int, ...]]] = {}
        self.clock = 0                                            # LFU: event counter
        self.meta: Dict[Tuple[int, Tuple[int, ...]], List[int]] = {}   # LFU: (key, suffix) -> [count, time]

    def _lfu_order(self, key: int) -> None:
        self.lists[key].sort(key=lambda s: tuple(self.meta[(key, s)]))

    def insert(self, key: int, suffix: Sequence[int], uses: int = 0) -> None:
        key, suffix = int(key), tuple(int(t) for t in suffix)
        lst = self.lists.setdefault(key, [])
        if suffix in lst:
            self.use(key, suffix)
            return
        if self.policy == LFU:
            self.clock += 1
            if len(lst) == self.cap:
                del self.meta[(key, lst.pop(0))]
            lst.append(suffix)
            self.meta[(key, suffix)] = [uses, self.clock]
            self._lfu_order(key)
            return
        lst.append(suffix)
        if len(lst) > self.cap:
            lst.pop(0)

    def use(self, key: int, suffix: Sequence[int]) -> None:
        """LRU: move a present suffix to the most recent end.  LFU: count the
        use and re-order.  FIFO: no-op."""
        key, suffix = int(key), tuple(int(t) for t in suffix)
        lst = self.lists[key]
        if self.policy == LRU:
            lst.remove(suffix)
            lst.append(suffix)
        elif self.policy == LFU:
            self.clock += 1
            m = self.meta[(key, suffix)]
            m[0] += 1
            m[1] = self.clock
            self._lfu_order(key)

    def lookup(self, key: int, G: int) -> List[Tuple[int, ...]]:
        lst = list(self.lists.get(int(key), []))
        if self.policy in (LRU, LFU):
            lst.reverse()
        return lst[:G]

    def records(self) -> List[Tuple[int, Tuple[int, ...]]]:
        """Canonical form: keys ascending, each key's suffixes in eviction order."""
        return [(k, s) for k in sorted(self.lists) for s in self.lists[k]]

    def use_counts(self) -> List[int]:
        """LFU: the use count of each entry of records(), in the same order."""
        return [self.meta[(k, s)][0] for k, s in self.records()]

    def copy(self) -> "Pool":
        p = Pool(self.cap, self.policy)
        p.lists = {k: list(v) for k, v in self.lists.items()}
        p.clock = self.clock
        p.meta = {k: list(v) for k, v in self.meta.items()}
        return p

    @staticmethod
    def from_records(cap: int, records, policy: str = FIFO, uses=None) -> "Pool":
        """Rebuild a pool from records in eviction order (LFU: with their use
        counts; entry times follow the record order, which keeps it)."""
        p = Pool(cap, policy)
        for i, (k, s) in enumerate(records):
            p.insert(k, s, uses[i] if uses is not None else 0)
        return p


# --------------------------------------------------------------------------
# Window: init, harvest, slide (readings R5, R7, R8)
# --------------------------------------------------------------------------

def splitmix64(x: int) -> int:
    """splitmix64 finaliser (Steele, Lea, Flood, OOPSLA 2014)."""
    x = (x + 0x9E3779B97F4A7C15) & MASK64
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & MASK64
    return x ^ (x >> 31)


def init_window(prompt: Sequence[int], N: int, W: int, seed: int) -> np.ndarray:
    s = len(prompt)
    V = np.zeros((N - 1, W), dtype=np.int64)
    for k in range(N - 1):
        for j in range(W):
            V[k, j] = prompt[splitmix64((seed ^ (k * W + j)) & MASK64) % s]
    return V


def harvest(window: np.ndarray, new: Sequence[int]) -> List[Tuple[int, Tuple[int, ...]]]:
    """Column j's n-gram: key V[0][j], suffix (V[1][j], ..., V[N-2][j], new_j)."""
    Nm1, W = window.shape
    out = []
    for j in range(W):
        suffix = tuple(int(window[k, j]) for k in range(1, Nm1)) + (int(new[j]),)
        out.append((int(window[0, j]), suffix))
    return out


def shift(window: np.ndarray, new: Sequence[int]) -> np.ndarray:
    out = np.empty_like(window)
    out[:-1] = window[1:]
    out[-1] = np.asarray(new)
    return out


def prompt_ngrams(prompt: Sequence[int], N: int):
    return [(int(prompt[i]), tuple(int(t) for t in prompt[i + 1:i + N])) for i in range(len(prompt) - N + 1)]


# --------------------------------------------------------------------------
# Verification (Algorithms 3 and 4; readings R4, R9, R10)
# --------------------------------------------------------------------------

def argmax_lowest(logits: np.ndarray) -> int:
    """Argmax with ties to the lowest id (np.argmax returns the first max)."""
    return int(np.argmax(logits))


def greedy_verify(cands: Sequence[Sequence[int]], tau0: int, cand_argmax) -> Tuple[List[int], int]:
    """Algorithm 3.  tau0 = argmax of row 0; cand_argmax(c, m) = argmax of row
    (c, m).  Returns (accepted tokens, winning candidate or -1)."""
    g = len(cands)
    survivors = list(range(g))
    acc: List[int] = []
    target = tau0                  # argmax distribution at the current depth
    depth = 1
    while True:
        nxt = [c for c in survivors if depth <= len(cands[c]) and cands[c][depth - 1] == target]
        if not nxt:
            acc.append(target)     # no candidate matches: take the model's token, stop
            break
        acc.append(target)         # matched candidate token == argmax
        survivors = nxt
        if depth == len(cands[survivors[0]]):
            acc.append(cand_argmax(survivors[0], depth))  # all N-1 matched: bonus token
            break
        target = cand_argmax(survivors[0], depth)
        depth += 1
    winner = survivors[0] if len(acc) > 1 else -1
    return acc, winner


def inverse_cdf(weights: np.ndarray, u: float) -> int:
    """Smallest id whose ascending cumulative weight exceeds u * total."""
    c = np.cumsum(weights)
    return int(np.searchsorted(c, u * c[-1], side="right"))


@dataclasses.dataclass
class SampleDecision:
    position: int
    kind: str              # "accept" (r vs dist(x)) or "draw" (inverse CDF)
    token: int
    value: float           # r - dist(x) for accept tests; distance of u*total to the nearest CDF edge for draws


def sampling_verify(cands, dist_row0: np.ndarray, cand_dist, P: int, seed: int, N: int,
                    trace: Optional[List[SampleDecision]] = None) -> Tuple[List[int], int]:
    """Algorithm 4 with greedy drafts (reading R10).  dist_row0 is softmax of
    row 0; cand_dist(c, m) the softmax of row (c, m).  Draws come from Philox
    keyed by seed at counter (position, draw index)."""
    g = len(cands)
    survivors = list(range(g))
    dist = np.array(dist_row0, dtype=np.float64)
    acc: List[int] = []
    depth = 1
    while True:
        pos = P + depth
        nd = 0
        accepted = None
        if depth <= N - 1 and survivors:
            rejected = set()
            for c in survivors:
                x = int(cands[c][depth - 1])
                if x in rejected:
                    continue
                r = philox.uniform(seed, pos, nd)
                nd += 1
                px = dist[x] / dist.sum()
                if trace is not None:
                    trace.append(SampleDecision(pos, "accept", x, r - px))
                if r <= px:
                    accepted = x
                    break
                dist[x] = 0.0
                dist = dist / dist.sum()
                rejected.add(x)
        if accepted is not None:
            acc.append(accepted)
            survivors = [c for c in survivors if int(cands[c][depth - 1]) == accepted]
            dist = np.array(cand_dist(survivors[0], depth), dtype=np.float64)
            depth += 1
            continue
        u = philox.uniform(seed, pos, nd)
        x = inverse_cdf(dist, u)
        if trace is not None:
            c = np.cumsum(dist)
            t = u * c[-1]
            lo = c[x - 1] if x > 0 else 0.0
            trace.append(SampleDecision(pos, "draw", x, min(t - lo, c[x] - t) / c[-1]))
        acc.append(x)
        break
    winner = survivors[0] if len(acc) > 1 else -1
    return acc, winner


def softmax(logits: np.ndarray, T: float) -> np.ndarray:
    z = logits / T
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def filter_top(dist: np.ndarray, top_k: int = 0, top_p: float = 1.0) -> np.ndarray:
    """Reading R14: zero every token outside the top-k, then outside the
    top-p prefix of what is left; ranking by probability, ties to the lower
    id.  top_k <= 0 or >= V and top_p >= 1 leave the distribution whole."""
    p = np.array(dist, dtype=np.float64)
    order = sorted(range(len(p)), key=lambda v: (-p[v], v))
    keep = list(order)
    if 0 < top_k < len(p):
        keep = keep[:top_k]
    if top_p < 1.0:
        mass = np.array([p[v] for v in keep])
        cum = np.cumsum(mass) / mass.sum()
        n = int(np.searchsorted(cum, top_p, side="left")) + 1   # first prefix with cum >= top_p
        keep = keep[:min(n, len(keep))]
    out = np.zeros_like(p)
    out[keep] = p[keep]
    return out


# --------------------------------------------------------------------------
# Generation (autoregressive reference and lookahead)
# --------------------------------------------------------------------------

def generate_ar(weights, prompt: Sequence[int], max_new: int, dtype=np.float64) -> List[int]:
    """Greedy autoregressive decoding, one forward per token (the lossless reference)."""
    prompt = [int(t) for t in prompt]
    s = len(prompt)
    logits, cache = decoder.forward(weights, prompt, np.arange(s), decoder.causal_mask(0, s),
                                    dtype=dtype, logit_rows=[s - 1])
    out = [argmax_lowest(logits[0])]
    while len(out) < max_new:
        P = s + len(out) - 1
        logits, kv = decoder.forward(weights, [out[-1]], np.array([P]), np.ones((1, P + 1), bool),
                                     cache=cache, dtype=dtype)
        cache = decoder.concat_cache(cache, kv)
        out.append(argmax_lowest(logits[0]))
    return out


@dataclasses.dataclass
class StepRecord:
    P: int                       # prefix length before the step
    o: int                       # last committed token before the step
    cands: List[Tuple[int, ...]]
    accepted: List[int]
    winner: int
    new: List[int]               # new lookahead tokens (argmax of the top level)
    window_before: np.ndarray
    logits: Optional[np.ndarray] = None   # used-row logits [U, V]
    trace: Optional[List[SampleDecision]] = None
    decisive: Optional[List[int]] = None   # used-row indices whose argmax / distribution verification read


class Lookahead:
    """Lookahead decoding state and steps (oracle)."""

    def __init__(self, weights, N: int, W: int, G: int, temperature: float = 0.0, seed: int = 0,
                 prompt_as_reference: bool = False, pool_cap: int = 0, dtype=np.float64,
                 keep_logits: bool = False, top_k: int = 0, top_p: float = 1.0, pool_policy: str = FIFO):
        assert N >= 2 and W >= 1 and G >= 0
        self.w, self.N, self.W, self.G = weights, N, W, G
        self.T, self.seed = temperature, seed
        self.top_k, self.top_p = top_k, top_p
        self.par = prompt_as_reference
        self.dtype = dtype
        self.keep_logits = keep_logits
        self.pool = Pool(pool_cap if pool_cap > 0 else max(G, 1), pool_policy)
        self.rows = step_rows(N, W, G)
        self.used = used_rows(N, W, G)
        self.mask = step_mask(N, W, G)
        self.tokens: List[int] = []    # committed tokens: prompt, outputs; the last is o
        self.cache = None
        self.window = None
        self.history: List[StepRecord] = []

    def dist(self, logits: np.ndarray) -> np.ndarray:
        """A row's sampling distribution: softmax at T, then top-k / top-p (R14)."""
        return filter_top(softmax(logits, self.T), self.top_k, self.top_p)

    # state ------------------------------------------------------------
    @property
    def P(self) -> int:
        return len(self.tokens) - 1

    def prefill(self, prompt: Sequence[int]) -> int:
        prompt = [int(t) for t in prompt]
        s = len(prompt)
        logits, self.cache = decoder.forward(self.w, prompt, np.arange(s), decoder.causal_mask(0, s),
                                             dtype=self.dtype, logit_rows=[s - 1])
        if self.T > 0:
            y1 = inverse_cdf(self.dist(logits[0]), philox.uniform(self.seed, s, 0))
        else:
            y1 = argmax_lowest(logits[0])
        self.tokens = prompt + [y1]
        self.window = init_window(prompt, self.N, self.W, self.seed)
        if self.par:
            for key, suf in prompt_ngrams(prompt, self.N):
                self.pool.insert(key, suf)
        return y1

    def load_state(self, tokens: Sequence[int], window: np.ndarray, pool_records, pool_uses=None) -> None:
        """Start from a given committed sequence, window and pool (LFU: with
        the entries' use counts); the prefix KV is recomputed from the tokens."""
        self.tokens = [int(t) for t in tokens]
        P = self.P
        _, self.cache = decoder.forward(self.w, self.tokens[:P], np.arange(P), decoder.causal_mask(0, P),
                                        dtype=self.dtype, logit_rows=[P - 1])
        self.window = np.array(window, dtype=np.int64).reshape(self.N - 1, self.W)
        self.pool = Pool.from_records(self.pool.cap, pool_records, self.pool.policy, pool_uses)

    # one step -----------------------------------------------------------
    def step_inputs(self):
        """Tokens, positions and visibility of the step rows (R1-R3)."""
        N, W, G = self.N, self.W, self.G
        P, o = self.P, self.tokens[-1]
        cands = self.pool.lookup(o, G)
        toks = np.zeros(len(self.rows), dtype=np.int64)
        toks[0] = o
        for k in range(N - 1):
            for j in range(W):
                toks[look_row(N, W, k, j)] = self.window[k, j]
        for c, cand in enumerate(cands):
            for m in range(1, N):
                toks[cand_row(N, W, c, m)] = cand[m - 1]
        pos = np.array([P + r.depth for r in self.rows])
        vis = np.concatenate([np.ones((len(self.rows), P), bool), self.mask], axis=1)
        return cands, toks, pos, vis

    def step(self) -> List[int]:
        N, W, G = self.N, self.W, self.G
        P, o = self.P, self.tokens[-1]
        cands, toks, pos, vis = self.step_inputs()
        logits, kv = decoder.forward(self.w, toks, pos, vis, cache=self.cache, dtype=self.dtype,
                                     logit_rows=self.used)
        lrow = {r: logits[i] for i, r in enumerate(self.used)}
        new = [argmax_lowest(lrow[look_row(N, W, N - 2, j)]) for j in range(W)]
        trace = None
        # Bookkeeping for parity checks: which rows' logits the verification
        # reads (row 0, then the row of each candidate position it consults).
        read = [0]

        def row_of(c, m):
            read.append(self.used.index(cand_row(N, W, c, m)))
            return lrow[cand_row(N, W, c, m)]

        if self.T > 0:
            trace = []
            acc, winner = sampling_verify(
                cands, self.dist(lrow[0]), lambda c, m: self.dist(row_of(c, m)), P, self.seed, N, trace)
        else:
            acc, winner = greedy_verify(cands, argmax_lowest(lrow[0]), lambda c, m: argmax_lowest(row_of(c, m)))
        A = len(acc)
        assert 1 <= A <= N
        # KV of the accepted rows: row 0 and the winner's first A-1 rows.
        keep = [0] + [cand_row(N, W, winner, m) for m in range(1, A)]
        self.cache = decoder.concat_cache(self.cache, [(k[keep], v[keep]) for k, v in kv])
        rec = StepRecord(P, o, cands, acc, winner, new, self.window.copy(),
                         logits if self.keep_logits else None, trace, read)
        if winner >= 0:
            self.pool.use(o, cands[winner])
        for key, suf in harvest(self.window, new):
            self.pool.insert(key, suf)
        self.window = shift(self.window, new)
        self.tokens.extend(acc)
        self.history.append(rec)
        return acc

    def generate(self, prompt: Sequence[int], max_new: int) -> Tuple[List[int], int]:
        out = [self.prefill(prompt)]
        steps = 0
        while len(out) < max_new:
            out.extend(self.step())
            steps += 1
        return out[:max_new], steps
