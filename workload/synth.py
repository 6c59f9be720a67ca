"""Seeded synthetic workloads for the verify-and-graft step of tree speculative decoding.

What this module is
-------------------
It draws random numbers and shapes them into the inputs that one verify-and-graft
step consumes:

* a draft tree per request (parent array in topological order, draft tokens, and
  the cumulative path score s(v) = product of edge probabilities from the root to v,
  as in the EAGLE-style tree grammar of "TreeGraft 精读" §三);
* the prune budget (a keep count, or a confidence threshold for the batched static
  tree of the Graft write-up §四);
* a retrieval template (template parent, successor rank) and the number of slots
  to refill (Graft write-up §二, the 8/24/40 + 52/36/20 split of 60 slots);
* the successor table (vocab x k, the write-up's "adjacency matrix"), initialised
  from a seeded bigram table or from a seeded repetitive token stream (a stand-in
  for the warm-up of Graft write-up §六);
* Q, K, V of one attention layer (K/V cache with the tree's rows already appended);
* target logits with a planted peak per node (a stand-in for the target model).

It holds none of the step's own arithmetic: no pruning, grafting, masking,
attention, top-k, path walk or table update. The CUDA path and the oracle both
consume exactly the arrays produced here; the drafter that grows the input tree
is upstream of the step and lives here only as an input generator.

All randomness comes from numpy's PCG64 seeded through SeedSequence, one child
stream per component, so every array is reproducible from (config, seed).
"""
from __future__ import annotations

import dataclasses
import heapq
from typing import Optional

import numpy as np

# ----------------------------------------------------------------------------------------
# bf16 encoding (data representation only)
# ----------------------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    lsb = (b >> 16) & np.uint32(1)
    # uint32 wrap-around only affects negative NaNs, which are replaced below
    r = ((b + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, np.uint16(0x7FC0), r)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Decode bfloat16 bits (uint16) to float32 exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------------------
# Draft-tree generators (upstream drafters; inputs of the step)
# ----------------------------------------------------------------------------------------


def _edge_probs(rng: np.random.Generator, V: int) -> np.ndarray:
    """A drafter's next-token distribution: softmax of N(0,1) logits, rounded to fp32."""
    z = rng.standard_normal(V, dtype=np.float32).astype(np.float64)
    z -= z.max()
    e = np.exp(z)
    return (e / e.sum()).astype(np.float32)


def _top_children(p: np.ndarray, m: int) -> np.ndarray:
    """The m most likely tokens of a drafter distribution (ties: lower token id)."""
    return np.argsort(-p, kind="stable")[:m]


def eagle_tree(rng: np.random.Generator, V: int, steps):
    """Grow a draft tree EAGLE-style.

    ``steps`` is a list of (W, m): at each step the top-W newest nodes by cumulative
    score form the frontier and each gets its top-m children (the first step expands
    the root only). Nodes are appended step by step, frontier in score order, children
    in probability order, so parent index < child index. Scores are fp32 products of
    fp32 edge probabilities, hence non-increasing from root to leaf.
    """
    parent = [-1]
    tokens = [int(rng.integers(V))]
    score = [np.float32(1.0)]
    newest = [0]
    for W, m in steps:
        frontier = sorted(newest, key=lambda v: (-float(score[v]), v))[:W]
        new = []
        for f in frontier:
            p = _edge_probs(rng, V)
            for t in _top_children(p, m):
                parent.append(f)
                tokens.append(int(t))
                score.append(np.float32(score[f] * p[t]))
                new.append(len(parent) - 1)
        newest = new
    return (np.asarray(parent, np.int32), np.asarray(tokens, np.int32),
            np.asarray(score, np.float32))


def static_tree_widths():
    """Expansion widths of a fixed 60-node static tree: 1 + 10 + 5*7 + 2*7 = 60."""
    return [(1, 10), (5, 7), (2, 7)]


def treegraft_tree(rng_small: np.random.Generator, rng_mid: np.random.Generator, V: int,
                   D: int = 5, W: int = 10, m: int = 10, schedule=(1, 0, 1, 0, 1),
                   n_max: int = 256):
    """Grow one shared tree with two drafters ("TreeGraft 精读" §四, Where/How).

    Small-drafter steps draw the frontier from the newest nodes; mid-drafter steps draw
    it from every node the mid drafter has not visited yet, then mark the pool visited.
    New children are attached without removing existing ones (non-destructive), so a
    node can gain children from both drafters. Growth stops at ``n_max`` nodes.
    """
    root = int(rng_small.integers(V))
    parent, tokens, score = [-1], [root], [np.float32(1.0)]
    newest, visited = [0], set()
    for k in range(D):
        if len(parent) >= n_max:
            break
        use_mid = bool(schedule[k])
        if use_mid:
            pool = [v for v in range(len(parent)) if v not in visited]
            visited.update(pool)
        else:
            pool = newest
        frontier = sorted(pool, key=lambda v: (-float(score[v]), v))[:W]
        new = []
        for f in frontier:
            p = _edge_probs(rng_mid if use_mid else rng_small, V)
            for t in _top_children(p, m):
                if len(parent) >= n_max:
                    break
                parent.append(f)
                tokens.append(int(t))
                score.append(np.float32(score[f] * p[t]))
                new.append(len(parent) - 1)
        newest = new
    return (np.asarray(parent, np.int32), np.asarray(tokens, np.int32),
            np.asarray(score, np.float32))


def dflash_chain(rng: np.random.Generator, V: int, L: int = 16):
    """One block draft of L tokens as a chain below the root (Graft write-up §七, DFlash).

    A block drafter proposes L tokens at once, each with its own confidence. The tokens
    are uniform draws; the confidence c_i of position i is a Beta(8, 2) draw scaled by
    (1 - 0.03 i), so later positions of the block are less sure on average. The node score
    is the fp32 running product of the confidences, non-increasing along the chain like
    the path scores of the tree drafters, so a score threshold keeps a prefix of the block.
    """
    tokens = rng.integers(0, V, size=L + 1).astype(np.int32)
    conf = (rng.beta(8.0, 2.0, size=L) * (1.0 - 0.03 * np.arange(L))).astype(np.float32)
    score = [np.float32(1.0)]
    for c in conf:
        score.append(np.float32(score[-1] * c))
    parent = np.arange(-1, L, dtype=np.int32)
    return parent, tokens, np.asarray(score, np.float32)


# ----------------------------------------------------------------------------------------
# Retrieval template (an input of the graft; its shape is a reading, see default_template)
# ----------------------------------------------------------------------------------------


def default_template(T: int, k: int = 8, max_depth: int = 8):
    """Asymmetric retrieval template of T nodes rooted at the current token.

    A template node is a path of successor ranks (r_1, ..., r_d). Nodes are chosen
    best-first by the integer weight prod(r_i + 2) (smaller first; ties by depth, then
    lexicographic rank path), with depth <= max_depth and ranks < k. Higher-ranked
    successors therefore get more children and deeper chains (Graft write-up §二,
    "asymmetric" template). Output is in selection order: every prefix of the template
    is ancestor-closed, so one template serves every refill size R <= T.
    Returns (tpar, trank): template parent index (-1 = the tree root) and rank.
    """
    if T <= 0:
        return np.zeros(0, np.int32), np.zeros(0, np.int32)
    heap = [(r + 2, 1, (r,)) for r in range(k)]
    heapq.heapify(heap)
    index, tpar, trank = {}, [], []
    while len(tpar) < T and heap:
        w, dep, path = heapq.heappop(heap)
        index[path] = len(tpar)
        tpar.append(index[path[:-1]] if dep > 1 else -1)
        trank.append(path[-1])
        if dep < max_depth:
            for r in range(k):
                heapq.heappush(heap, (w * (r + 2), dep + 1, path + (r,)))
    return np.asarray(tpar, np.int32), np.asarray(trank, np.int32)


# ----------------------------------------------------------------------------------------
# Successor-table initialisations (stand-ins for the warm-up of Graft write-up §六)
# ----------------------------------------------------------------------------------------


def bigram_table(rng: np.random.Generator, V: int, k: int) -> np.ndarray:
    """Seeded random bigram table: row t holds k distinct successor ids."""
    base = rng.integers(0, V, size=V, dtype=np.int64)
    step_max = max(2, V // (4 * k))
    steps = rng.integers(1, step_max, size=(V, k), dtype=np.int64)
    steps[:, 0] = 0
    offs = np.cumsum(steps, axis=1)
    return ((base[:, None] + offs) % V).astype(np.int32)


def repetitive_stream(rng: np.random.Generator, V: int, length: int, p_copy: float = 0.3,
                      ngram: int = 8, zipf_a: float = 1.2) -> np.ndarray:
    """Code-like token stream: with probability p_copy a position starts a copy of an
    earlier ``ngram``-gram, otherwise it emits one Zipf-distributed token."""
    perm = rng.permutation(V)
    out = np.empty(length + ngram, dtype=np.int64)
    n = 0
    fresh = perm[(rng.zipf(zipf_a, size=length) - 1) % V]
    fi = 0
    u = rng.random(length)
    starts = rng.random(length)
    ui = 0
    while n < length:
        if n >= 2 * ngram and u[ui] < p_copy:
            s = int(starts[ui] * (n - ngram))
            out[n:n + ngram] = out[s:s + ngram]
            n += ngram
        else:
            out[n] = fresh[fi]
            fi += 1
            n += 1
        ui += 1
    return out[:length]


def stream_table(rng: np.random.Generator, V: int, k: int, length: int = 1 << 20,
                 p_copy: float = 0.3, ngram: int = 8) -> np.ndarray:
    """Successor table counted from a seeded repetitive stream.

    Row t lists the k most frequent successors of t in the stream (ties: smaller id);
    rows with fewer than k observed successors are completed, in order, from a seeded
    random permutation of the vocabulary, skipping ids already in the row.
    """
    s = repetitive_stream(rng, V, length, p_copy, ngram)
    key = s[:-1] * V + s[1:]
    uniq, cnt = np.unique(key, return_counts=True)
    ta, tb = uniq // V, uniq % V
    order = np.lexsort((tb, -cnt, ta))
    ta, tb = ta[order], tb[order]
    first = np.searchsorted(ta, ta, side="left")
    rank = np.arange(len(ta)) - first
    sel = rank < k
    table = np.full((V, k), -1, dtype=np.int64)
    table[ta[sel], rank[sel]] = tb[sel]
    fill = rng.permutation(V)
    have = (table >= 0).sum(axis=1)
    empty = np.nonzero(have == 0)[0]
    table[empty] = fill[(empty[:, None] * k + np.arange(k)[None, :]) % V]
    for t in np.nonzero((have > 0) & (have < k))[0]:
        row = [int(x) for x in table[t, :have[t]]]
        j = int(t) * k
        while len(row) < k:
            c = int(fill[j % V])
            j += 1
            if c not in row:
                row.append(c)
        table[t] = row
    return table.astype(np.int32)


# ----------------------------------------------------------------------------------------
# Inputs of the n-gram drafter: a token history and the target's top-m cache of prefill
# ----------------------------------------------------------------------------------------


def topm_cache(rng: np.random.Generator, seq: np.ndarray, V: int, m: int,
               p_hit: float = 0.6):
    """A stand-in for the target's top-m cache of prefill over the history ``seq[:-1]``.

    Row i lists m token ids for position i+1 with float32 probabilities in descending
    order (a softmax of m N(0, 1.5^2) draws scaled by a mass in [0.5, 0.95]). With
    probability p_hit the true next token seq[i+1] sits at a uniform rank; the other ids
    are tokens of uniformly drawn stream positions (plausible alternatives, distributed
    like the stream itself).
    """
    L = len(seq) - 1
    ids = np.asarray(seq, np.int32)[rng.integers(0, L + 1, size=(L, m))]
    hit = rng.random(L) < p_hit
    rank = rng.integers(0, m, size=L)
    rows = np.nonzero(hit)[0]
    ids[rows, rank[rows]] = seq[1:][rows]
    z = rng.standard_normal((L, m)) * 1.5
    w = np.exp(z - z.max(axis=1, keepdims=True))
    probs = -np.sort(-(w / w.sum(axis=1, keepdims=True)), axis=1)
    mass = rng.uniform(0.5, 0.95, size=(L, 1))
    return ids, (probs * mass).astype(np.float32)


@dataclasses.dataclass
class DraftScenario:
    """Inputs of n-gram drafting steps for B requests (numpy, host memory)."""
    hist: np.ndarray       # int32 [B][L] committed tokens before the root
    hist_len: np.ndarray   # int32 [B]
    cache_id: np.ndarray   # int32 [B][L][m]
    cache_p: np.ndarray    # float32 [B][L][m]
    root: np.ndarray       # int32 [B] the current token (tree node 0)
    V: int
    m: int
    W: int
    q_max: int
    Nmax: int


def make_draft_scenario(B: int = 1, L: int = 32768, V: int = 151936, m: int = 10, W: int = 10,
                        q_max: int = 4, Nmax: int = 256, seed: int = 7) -> DraftScenario:
    """Code-like histories (the repetitive stream of the successor tables) with their
    top-m caches; the tree starts as the root alone (TreeGraft write-up §五: D = 5,
    W = 10, m = 10; growth capped at Nmax nodes before the prune)."""
    rngs = _rngs(seed, 2 * B)
    hist = np.zeros((B, L), np.int32)
    cid = np.zeros((B, L, m), np.int32)
    cp = np.zeros((B, L, m), np.float32)
    root = np.zeros(B, np.int32)
    for b in range(B):
        seq = repetitive_stream(rngs[2 * b], V, L + 1).astype(np.int32)
        hist[b], root[b] = seq[:L], seq[L]
        cid[b], cp[b] = topm_cache(rngs[2 * b + 1], seq, V, m)
    return DraftScenario(hist=hist, hist_len=np.full(B, L, np.int32), cache_id=cid, cache_p=cp,
                         root=root, V=V, m=m, W=W, q_max=q_max, Nmax=Nmax)


# ----------------------------------------------------------------------------------------
# Target stand-in: logits with a planted peak per node
# ----------------------------------------------------------------------------------------


def plant_logits(rng: np.random.Generator, parent: np.ndarray, tokens: np.ndarray, n: int,
                 N: int, V: int, p_accept: float, peak: float = 6.0) -> np.ndarray:
    """Synthetic target logits for one request's tree of n nodes (rows padded to N).

    Row v is N(0,1) noise plus ``peak`` on one token: with probability p_accept the
    token of v's first child (lowest index; for drafted nodes the most likely child),
    otherwise a uniform token. Padding rows (v >= n) are noise only.
    """
    out = rng.standard_normal((N, V), dtype=np.float32)
    first_child = {}
    for v in range(1, n):
        first_child.setdefault(int(parent[v]), v)
    u = rng.random(N)
    unif = rng.integers(0, V, size=N)
    for v in range(n):
        c = first_child.get(v)
        t = int(tokens[c]) if (c is not None and u[v] < p_accept) else int(unif[v])
        out[v, t] += np.float32(peak)
    return out


# ----------------------------------------------------------------------------------------
# Scenarios: the five workloads of the verify-and-graft step
# ----------------------------------------------------------------------------------------

CONFIGS = {
    1: dict(name="tiny-eagle411to63-fp32-h8kv8-P512-V32000", B=1, Hq=8, Hkv=8, d=128,
            dtype="f32", V=32000, k=8, P=512, tree="eagle", keep=63, R=0, N=63,
            p_accept=0.7, table="bigram"),
    2: dict(name="llama3.1-8b-h32kv8-P4096-V128256-stage1-24+36", B=1, Hq=32, Hkv=8,
            d=128, dtype="bf16", V=128256, k=8, P=4096, tree="eagle", keep=24, R=36,
            N=60, p_accept=0.6, table="bigram"),
    3: dict(name="qwen3-8b-h32kv8-P32768-V151936-root-8+52", B=1, Hq=32, Hkv=8, d=128,
            dtype="bf16", V=151936, k=8, P=32768, tree="eagle", keep=8, R=52, N=60,
            p_accept=0.5, table="stream"),
    4: dict(name="qwen3-32b-h64kv8-B16-P1024..8192-V151936-static60", B=16, Hq=64,
            Hkv=8, d=128, dtype="bf16", V=151936, k=8, P=(1024, 8192), tree="static60",
            keep=60, R=60, N=60, p_accept=0.6, table="stream"),
    5: dict(name="llama3-70b-h64kv8-P16384-V128256-treegraft256to63", B=1, Hq=64, Hkv=8,
            d=128, dtype="bf16", V=128256, k=8, P=16384, tree="treegraft", keep=63, R=0,
            N=63, p_accept=0.55, table="bigram"),
    # Graft-TAIL on a block draft: keep the confident prefix of a 16-token DFlash chain,
    # refill the freed slots with retrieved candidates hung from the prefix's last token
    6: dict(name="qwen3-8b-h32kv8-P4096-V151936-dflash16-tail", B=1, Hq=32, Hkv=8, d=128,
            dtype="bf16", V=151936, k=8, P=4096, tree="dflash", keep=17, R=17, N=17,
            p_accept=0.6, table="stream", anchor=-1),
}

EAGLE_STEPS = [(1, 10), (10, 10), (10, 10), (10, 10), (10, 10)]  # D=5, W=10, m=10


@dataclasses.dataclass
class Scenario:
    """All pre-step inputs of one verify-and-graft workload (numpy, host memory)."""
    cid: int
    name: str
    B: int
    Nin: int            # draft-tree nodes per request before the prune
    N: int              # slots per request after prune + graft (rows of Q / logits)
    V: int
    k: int
    Hq: int
    Hkv: int
    d: int
    dtype: str          # "f32" or "bf16" (Q/K/V storage)
    Lcap: int
    scale: float
    parent_in: np.ndarray   # int32 [B][Nin]
    tokens_in: np.ndarray   # int32 [B][Nin]
    score_in: np.ndarray    # float32 [B][Nin]
    keep: np.ndarray        # int32 [B]
    thresh: Optional[np.ndarray]  # float32 [B] or None
    tpar: np.ndarray        # int32 [T]
    trank: np.ndarray       # int32 [T]
    R: np.ndarray           # int32 [B]
    table: np.ndarray       # int32 [V][k]
    prefix_len: np.ndarray  # int32 [B]
    Q: np.ndarray           # [B][N][Hq][d]  float32 or uint16 (bf16 bits)
    K: np.ndarray           # [B][Hkv][Lcap][d]
    Vc: np.ndarray          # [B][Hkv][Lcap][d]
    p_accept: float
    seed: int
    anchor: Optional[np.ndarray] = None  # int32 [B] graft anchor (-1: last kept node) or None

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    def logits(self, parent: np.ndarray, tokens: np.ndarray, n_nodes: np.ndarray) -> np.ndarray:
        """Planted target logits [B][N][V] for the given final trees (deterministic)."""
        ss = np.random.SeedSequence([self.seed, 0x10617])
        rngs = [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(self.B)]
        return np.stack([plant_logits(rngs[b], parent[b], tokens[b], int(n_nodes[b]), self.N,
                                      self.V, self.p_accept) for b in range(self.B)])


def _rngs(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def make_scenario(cid: int, seed: Optional[int] = None, *, V: Optional[int] = None,
                  P=None, B: Optional[int] = None, stream_len: int = 1 << 20,
                  kv_fill: str = "zero", tree_scale: Optional[list] = None) -> Scenario:
    """Build the inputs of workload ``cid`` (1..5) with optional size overrides.

    ``V``/``P``/``B`` shrink the vocabulary, KV prefix and batch for quick tests while
    keeping the tree shapes and budgets. ``kv_fill`` fills cache rows past each request's
    valid length with zeros ("zero") or NaN ("nan", to check that they are never read).
    """
    c = dict(CONFIGS[cid])
    seed = cid if seed is None else seed
    V = c["V"] if V is None else V
    B = c["B"] if B is None else B
    P = c["P"] if P is None else P
    k, Hq, Hkv, d, N = c["k"], c["Hq"], c["Hkv"], c["d"], c["N"]
    r_tree, r_small, r_mid, r_tab, r_qkv, r_pre, r_thr = _rngs(seed, 7)

    # prefix lengths
    if isinstance(P, tuple):
        prefix = r_pre.integers(P[0], P[1] + 1, size=B).astype(np.int32)
    else:
        prefix = np.full(B, int(P), np.int32)

    # draft trees
    trees = []
    for _b in range(B):
        if c["tree"] == "eagle":
            trees.append(eagle_tree(r_tree, V, tree_scale or EAGLE_STEPS))
        elif c["tree"] == "static60":
            trees.append(eagle_tree(r_tree, V, tree_scale or static_tree_widths()))
        elif c["tree"] == "dflash":
            trees.append(dflash_chain(r_tree, V, c["N"] - 1))
        else:
            trees.append(treegraft_tree(r_small, r_mid, V))
    Nin = max(len(t[0]) for t in trees)
    parent_in = np.full((B, Nin), -1, np.int32)
    tokens_in = np.full((B, Nin), -1, np.int32)
    score_in = np.zeros((B, Nin), np.float32)
    for b, (pa, to, sc) in enumerate(trees):
        n = len(pa)
        parent_in[b, :n], tokens_in[b, :n], score_in[b, :n] = pa, to, sc
    if any(len(t[0]) != Nin for t in trees):
        raise ValueError("draft trees of one scenario must have equal node counts")

    keep = np.full(B, min(c["keep"], Nin), np.int32)
    thresh = None
    if c["tree"] in ("static60", "dflash"):
        # seeded confidence threshold: log-uniform between the smallest and largest
        # non-root score, at a seeded fraction q_b of that range
        thresh = np.zeros(B, np.float32)
        q = r_thr.uniform(0.2, 0.9, size=B)
        for b in range(B):
            s = score_in[b, 1:].astype(np.float64)
            lo, hi = np.log(s.min()), np.log(s.max())
            thresh[b] = np.float32(np.exp(lo + q[b] * (hi - lo)))

    tpar, trank = default_template(c["R"], k)
    R = np.full(B, c["R"], np.int32)

    if c["table"] == "bigram":
        table = bigram_table(r_tab, V, k)
    else:
        table = stream_table(r_tab, V, k, length=stream_len)

    Lcap = int(prefix.max()) + N
    Lcap = (Lcap + 63) // 64 * 64
    Q = r_qkv.standard_normal((B, N, Hq, d), dtype=np.float32)
    Kc = np.zeros((B, Hkv, Lcap, d), np.float32)
    Vc = np.zeros((B, Hkv, Lcap, d), np.float32)
    for b in range(B):
        L = int(prefix[b]) + N
        Kc[b, :, :L] = r_qkv.standard_normal((Hkv, L, d), dtype=np.float32)
        Vc[b, :, :L] = r_qkv.standard_normal((Hkv, L, d), dtype=np.float32)
        if kv_fill == "nan":
            Kc[b, :, L:] = np.nan
            Vc[b, :, L:] = np.nan
    if c["dtype"] == "bf16":
        Q, Kc, Vc = f32_to_bf16_bits(Q), f32_to_bf16_bits(Kc), f32_to_bf16_bits(Vc)

    return Scenario(cid=cid, name=c["name"], B=B, Nin=Nin, N=N, V=V, k=k, Hq=Hq, Hkv=Hkv,
                    d=d, dtype=c["dtype"], Lcap=Lcap, scale=float(np.float32(1.0 / np.sqrt(d))),
                    parent_in=parent_in, tokens_in=tokens_in, score_in=score_in, keep=keep,
                    thresh=thresh, tpar=tpar, trank=trank, R=R, table=table, prefix_len=prefix,
                    Q=Q, K=Kc, Vc=Vc, p_accept=c["p_accept"], seed=seed,
                    anchor=None if "anchor" not in c else np.full(B, c["anchor"], np.int32))
