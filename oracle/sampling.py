"""CPU oracle of tree verification at temperature T > 0 (test infrastructure).

Like the rest of ``oracle/``, this module is slow on purpose, shares no code with the CUDA
path and is imported only by the tests, the package smoke check and the benchmark's CPU
leg.

Sources (page title, then section):
  [TreeGraft] "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题",
              §三 (the pruned tree goes to tree-attention verification and rejection
              sampling; the output distribution must not change) and §七 (rejection
              sampling keeps the target's output distribution).
  Philox-4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2,
              3", SC 2011 (counter-based generator; round function and constants).
  Gumbel-max: sampling from softmax(s) as argmax_j (s_j + G_j) with G_j i.i.d. standard
              Gumbel, G = -log(-log U) for U uniform on (0, 1) (Gumbel 1954; e.g.
              Maddison, Tarlow, Minka 2014).
  Logarithm:  log m = 2 artanh((m - 1)/(m + 1)) = 2 (s + s^3/3 + s^5/5 + ...), s = (m-1)/(m+1)
              (Abramowitz & Stegun 4.1.27), after splitting off the binary exponent.

Readings where the pages are silent:
  * The tree's proposals are deterministic (top-m children of a drafter, retrieved
    successors), i.e. point masses. Rejection sampling of point-mass proposals tries the
    children of the accepted node u in index order; child c is accepted with the residual
    target probability of its token, a rejected token's mass is removed and the residual
    renormalised; if every child is rejected the bonus token is drawn from the residual.
    That is the same distribution as drawing ONE token y_u from the target's softmax at u
    and moving to the first child (lowest index) whose token is y_u, stopping with y_u as
    the bonus when no child carries it. The oracle and the kernels use the one-draw form.
  * The target distribution at node u is softmax(z_u / T) over the whole vocabulary.
  * The draw y_u is the Gumbel-max sample of row r = b * N + u: score_j = z_j * (1/T) +
    G_j in float32 (1/T rounded to float32 once), G_j = -log(-log U_j), U_j the uniform
    ((x_j >> 9) + 0.5) * 2^-23 of a 32-bit word x_j = (A_j << 24) | (B_j >> 8). A_j is byte
    (j mod 16) (little-endian, word (j mod 16) div 4) of the Philox-4x32-10 block at counter
    (j div 16, r, step mod 2^32, step div 2^32); B_j is word (j mod 4) of the block at
    counter ((j div 4) + 2^31, r, step mod 2^32, step div 2^32); both with key
    (seed mod 2^32, seed div 2^32). The two counter ranges never meet (j < 2^30), so x_j
    is a uniform 32-bit word independent across j; its top byte alone tells whether U_j
    can be large, which lets a kernel skip the logarithms of almost every element;
    the largest score wins, ties to the smaller index; NaN ranks below -inf and +0.0
    equals -0.0 (the top-k order). Every float32 operation is one IEEE round to nearest,
    in the order written in ``log_f32`` and ``gumbel_scores``, so a float32 kernel that
    performs the same operations reaches the same integer decision.
  * The table update at T > 0 is the greedy one: the target's top-k of the unscaled
    logits at every verified node.
"""
from __future__ import annotations

import numpy as np

from .step import _check_tree, _children

# Philox-4x32 multipliers and Weyl key increments (Salmon et al. 2011, §5)
PHILOX_M0, PHILOX_M1 = 0xD2511F53, 0xCD9E8D57
PHILOX_W0, PHILOX_W1 = 0x9E3779B9, 0xBB67AE85
_M32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox-4x32-10 on arrays of counters (uint32 values in any integer dtype).

    Round: (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2 (64-bit products);
    c <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0); the key gains (W0, W1) before every
    round but the first. Returns four uint32 arrays.
    """
    c = [np.asarray(x, np.uint64) & _M32 for x in (c0, c1, c2, c3)]
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    for rnd in range(10):
        if rnd:
            k0 = np.uint64((int(k0) + PHILOX_W0) & 0xFFFFFFFF)
            k1 = np.uint64((int(k1) + PHILOX_W1) & 0xFFFFFFFF)
        p0 = np.uint64(PHILOX_M0) * c[0]
        p1 = np.uint64(PHILOX_M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _M32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _M32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return [x.astype(np.uint32) for x in c]


def uniform_f32(x):
    """The float32 uniform ((x >> 9) + 0.5) * 2^-23 of a 32-bit word: a multiple of 2^-24
    in [2^-24, 1 - 2^-24], exact in float32."""
    hi = (np.asarray(x, np.uint32) >> np.uint32(9)).astype(np.float32)
    return (hi + np.float32(0.5)) * np.float32(2.0 ** -23)


_F = np.float32
_SQRT2_MANT = 0x3504F3          # mantissa field of float32(sqrt 2)
_LN2 = _F(np.log(2.0))          # float32(ln 2)
_C3, _C5, _C7, _C9 = (_F(1) / _F(3), _F(1) / _F(5), _F(1) / _F(7), _F(1) / _F(9))


def log_f32(x):
    """Natural logarithm of positive normal float32 values, in float32 operations.

    x = 2^e * m with m in [sqrt(2)/2, sqrt(2)) (the mantissa field decides: above the
    field of sqrt(2) the value is halved and e raised by one); s = (m - 1) / (m + 1);
    log m = (s + s) * (1 + z/3 + z^2/5 + z^3/7 + z^4/9), z = s * s, the polynomial by
    Horner's rule from the 1/9 end; log x = e * ln2 + log m. Each operation rounds once.
    """
    x = np.asarray(x, np.float32)
    bits = x.view(np.uint32)
    mant = bits & np.uint32(0x7FFFFF)
    e = (bits >> np.uint32(23)).astype(np.int64) - 127
    big = mant > np.uint32(_SQRT2_MANT)
    mbits = np.where(big, mant | np.uint32(0x3F000000), mant | np.uint32(0x3F800000))
    e = e + big.astype(np.int64)
    m = mbits.astype(np.uint32).view(np.float32)
    f = m - _F(1)
    d = m + _F(1)
    s = f / d
    z = s * s
    p = _C9
    p = p * z + _C7
    p = p * z + _C5
    p = p * z + _C3
    p = p * z + _F(1)
    lm = (s + s) * p
    return e.astype(np.float32) * _LN2 + lm


def _byte_word(w, e):
    """Byte e (0..15) of a Philox block given as four word arrays, little-endian words."""
    return (w[e // 4] >> np.uint32(8 * (e % 4))) & np.uint32(0xFF)


def noise_words(V: int, rows, seed: int, step: int):
    """The 32-bit words x_j [R][V] of the rows ``rows`` (see the readings above)."""
    rows = np.asarray(rows, np.uint64)
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    s_lo, s_hi = step & 0xFFFFFFFF, (step >> 32) & 0xFFFFFFFF
    j = np.arange(V, dtype=np.int64)
    A16 = philox4x32_10(np.arange((V + 15) // 16, dtype=np.uint64)[None, :], rows[:, None],
                        s_lo, s_hi, *key)
    A = np.stack([_byte_word(A16, e) for e in range(16)], axis=-1).reshape(len(rows), -1)[:, :V]
    B4 = philox4x32_10(np.arange((V + 3) // 4, dtype=np.uint64)[None, :] + np.uint64(1 << 31),
                       rows[:, None], s_lo, s_hi, *key)
    B = np.stack(B4, axis=-1).reshape(len(rows), -1)[:, :V]
    assert A.shape[1] == B.shape[1] == j.size
    return (A << np.uint32(24)) | (B >> np.uint32(8))


def gumbel_scores(z, rows, temperature: float, seed: int, step: int):
    """Perturbed scores z * (1/T) + G of logit rows ``z`` [R][V] whose global row numbers
    are ``rows`` [R] (float32 [R][V])."""
    z = np.asarray(z, np.float32)
    R, V = z.shape
    inv_t = _F(1) / _F(temperature)
    rows = np.asarray(rows, np.uint64)
    out = np.empty((R, V), np.float32)
    chunk = max(1, (1 << 20) // max(V, 1))  # rows per batch
    for r0 in range(0, R, chunk):
        rr = rows[r0:r0 + chunk]
        u = uniform_f32(noise_words(V, rr, seed, step))
        g = -log_f32(-log_f32(u))
        with np.errstate(over="ignore"):  # z / T may overflow to +-inf, as in IEEE float32
            out[r0:r0 + len(rr)] = z[r0:r0 + len(rr)] * inv_t + g
    return out


def argmax_first(scores):
    """Index of the largest entry of each row: non-NaN before NaN, value descending
    (+0.0 equals -0.0), ties to the smaller index (0 for a row of NaN only)."""
    s = np.asarray(scores, np.float32)
    out = np.zeros(s.shape[0], np.int32)
    for i, row in enumerate(s):
        ok = ~np.isnan(row)
        if ok.any():
            m = row[ok].max()
            out[i] = np.flatnonzero(ok & (row == m))[0]
    return out


def vocab_sample(z, rows, temperature: float, seed: int, step: int):
    """One target draw per logit row ([TreeGraft] §三: sampling from the target's
    distribution at temperature T), by the Gumbel-max rule above. Returns int32 [R]."""
    return argmax_first(gumbel_scores(z, rows, temperature, seed, step))


def verify_sampled(tokens, parent, n: int, sample, prefix_len: int):
    """Tree verification at T > 0 of one request with one target draw per node.

    From the root: at the current node u the draw sample[u] is compared with u's
    children in index order; the first child carrying it becomes the current node; when
    none does the walk stops and sample[u] is the bonus token. Outputs as in greedy
    verification (path, committed tokens, KV commit indices).
    """
    _check_tree(parent, n)
    ch = _children(parent, n)
    path = [0]
    u = 0
    while True:
        nxt = next((c for c in ch[u] if int(tokens[c]) == int(sample[u])), None)
        if nxt is None:
            break
        u = nxt
        path.append(u)
    L = len(path) - 1
    out_tok = [int(tokens[path[j]]) for j in range(1, L + 1)] + [int(sample[u])]
    P = int(prefix_len)
    return dict(acc_len=L, path=path, out_tok=out_tok,
                kv_src=[P + p for p in path], kv_dst=[P + j for j in range(L + 1)])


def step_verify_sampled(tree, logits, table, prefix_len, k: int, temperature: float,
                        seed: int, step: int):
    """a5 + a6 + a7 at T > 0: per-node draws and the sampled walk, the top-k of every row
    and the greedy table update. Row r of the logits is request r // N, node r % N."""
    from .step import succ_update, vocab_topk
    B, N, V = logits.shape
    flat = np.asarray(logits, np.float32).reshape(B * N, V)
    sample = vocab_sample(flat, np.arange(B * N), temperature, seed, step).reshape(B, N)
    topk_id = np.zeros((B, N, k), np.int32)
    topk_val = np.zeros((B, N, k), np.float32)
    for b in range(B):
        for v in range(N):
            topk_id[b, v], topk_val[b, v] = vocab_topk(logits[b, v], k)
    out = dict(sample=sample, topk_id=topk_id, topk_val=topk_val,
               acc_len=np.zeros(B, np.int32), path=np.full((B, N), -1, np.int32),
               out_tok=np.full((B, N + 1), -1, np.int32), kv_src=np.full((B, N), -1, np.int32),
               kv_dst=np.full((B, N), -1, np.int32))
    for b in range(B):
        n = int(tree["n_nodes"][b])
        r = verify_sampled(tree["tokens"][b], tree["parent"][b], n, sample[b], prefix_len[b])
        L = r["acc_len"]
        out["acc_len"][b] = L
        out["path"][b, :L + 1] = r["path"]
        out["out_tok"][b, :L + 1] = r["out_tok"]
        out["kv_src"][b, :L + 1] = r["kv_src"]
        out["kv_dst"][b, :L + 1] = r["kv_dst"]
    out["table"] = succ_update(table, tree["tokens"], topk_id, tree["n_nodes"])
    return out
