"""One Token Recycling step, written out plainly (test infrastructure only).

Each function restates one part of the method in the pages' order; see the
package docstring for the sources.  Floating point that decides nothing
discrete (attention) is fp64; the top-K compares the logits exactly as given.
"""
from __future__ import annotations

import numpy as np

INIT_ZERO, INIT_RANDOM, INIT_INHERIT = 0, 1, 2
UPD_ALL, UPD_ACCEPTED = 0, 1

_MASK64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15


def mix64_stream(state, index):
    """Output ``index`` of a splitmix64 stream started at ``state``.

    splitmix64 as published by Steele, Lea and Flood (OOPSLA 2014): advance
    the state by the golden gamma, then apply the two xor-shift-multiply
    rounds and a final xor-shift.  Written with Python integers so it is
    independent of any array library.
    """
    z = (int(state) + (int(index) + 1) * _GAMMA) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def init_matrix(mode, V, K, seed=0, src=None, seq=0, dtype=np.int64):
    """Adjacency matrix M in V^{|V| x K} at the start of a request.

    hyper.ai summary, "Method": row i holds the K candidate successors of
    token i; the matrix is hot-started by inheriting one from earlier
    inference.  "Experiment": the ablation compares all-zero, random-vocab
    and inherited initialisation.  RANDOM draws entry (i, j) of sequence
    ``seq`` as output (seq*V + i)*K + j of a splitmix64 stream at ``seed``,
    modulo V (the pages fix no generator; this reading is listed).
    """
    if mode == INIT_ZERO:
        return np.zeros((V, K), dtype=dtype)
    if mode == INIT_INHERIT:
        src = np.asarray(src)
        if src.shape != (V, K):
            raise ValueError("inherited matrix must be [V, K]")
        return src.astype(dtype).copy()
    if mode == INIT_RANDOM:
        M = np.empty((V, K), dtype=dtype)
        for i in range(V):
            for j in range(K):
                M[i, j] = mix64_stream(seed, (seq * V + i) * K + j) % V
        return M
    raise ValueError("unknown init mode")


def retrieve(M, root, plan):
    """Draft tree tokens in BFS order.

    Blog "token-recycling", 完整工作流程 steps 1-2: the root is the last token
    of the context; its row gives the first layer, and each candidate is
    expanded again through its own row, as far as the static tree allows.
    Child r of a node holding token x is M[x][r].  Retrieval reads the matrix
    as it was before this step's update (same blog, the note on update
    timing: the whole tree is built from the old matrix).
    """
    tok = np.empty(plan.N, dtype=np.int64)
    tok[0] = int(root)
    for n in range(1, plan.N):
        tok[n] = M[tok[plan.parent[n]], plan.rank[n]]
    return tok


def tree_attention(q, kc, vc, L, kt, vt, plan, scale):
    """Tree attention for one sequence, in fp64.

    Blog "token-recycling", 完整工作流程 step 3, and the speculative-decoding
    lesson's tree drafting: the tree is flattened into one merged sequence
    placed after the prefix; a node attends to the whole prefix and, inside
    the tree, only to its own root-to-node path (itself included).  Siblings
    never see each other.  Query head h reads KV head h // (Hq / Hkv).

    q [N, Hq, d]; kc, vc [Hkv, cap, d] with the first L positions valid;
    kt, vt [N, Hkv, d]; returns O [N, Hq, d] (fp64).
    """
    q = np.asarray(q, dtype=np.float64)
    N, Hq, d = q.shape
    Hkv = kc.shape[0]
    group = Hq // Hkv
    visible = np.concatenate([np.ones((N, L), dtype=bool), plan.mask], axis=1)
    out = np.empty((N, Hq, d), dtype=np.float64)
    for h in range(Hq):
        g = h // group
        keys = np.concatenate([np.asarray(kc[g, :L], np.float64), np.asarray(kt[:, g], np.float64)])
        vals = np.concatenate([np.asarray(vc[g, :L], np.float64), np.asarray(vt[:, g], np.float64)])
        s = (q[:, h] @ keys.T) * scale
        s = np.where(visible, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h] = p @ vals
    return out


def topk(row, K):
    """The K most probable next tokens of one distribution, best first.

    Chinese hyper.ai summary, "方法", the update equation's argtopk; blog
    "token-recycling", 为什么叫 Token Recycling: keep the K highest tokens of
    each node's distribution.  Ties go to the lower token ID (the pages are
    silent; this reading is listed): a stable sort of the negated values keeps
    equal values in ascending ID order, and -0.0 compares equal to +0.0.
    """
    row = np.asarray(row)
    if not np.all(np.isfinite(row)):
        raise ValueError("logits must be finite")
    order = np.argsort(-row.astype(np.float64), kind="stable")
    return order[:K].astype(np.int64)


def topk_rows(rows, K):
    """topk of every row: ids [R, K] and their values [R, K]."""
    rows = np.asarray(rows)
    ids = np.stack([topk(r, K) for r in rows]) if len(rows) else np.zeros((0, K), np.int64)
    vals = np.take_along_axis(rows, ids, axis=1) if len(rows) else np.zeros((0, K), rows.dtype)
    return ids, vals


def accept(plan, tok, top1):
    """Greedy acceptance of the longest correct path, plus the bonus token.

    Blog "token-recycling", 完整工作流程 step 4, and the hyper.ai summary,
    "Method": the longest draft path that matches the target's greedy output
    is accepted, and the target's own token at the first mismatch is appended
    (the lesson's bonus token), so the output equals plain greedy decoding.

    Written as brute force: every node whose whole root path matches is a
    candidate; the deepest one wins, and among equally deep ones the smallest
    BFS index (a reading; the pages do not say).

    Returns (acc_len, path, committed, bonus): path is the node indices from
    the root to the chosen node; committed is the accepted tokens followed by
    the bonus.
    """
    best = 0
    for n in range(plan.N):
        p = plan.path[n]
        if all(tok[m] == top1[plan.parent[m]] for m in p[1:]):
            if plan.depth[n] > plan.depth[best]:
                best = n
    path = list(plan.path[best])
    bonus = int(top1[best])
    committed = [int(tok[m]) for m in path[1:]] + [bonus]
    return plan.depth[best], path, committed, bonus


def softmax_stats(row, T):
    """(max, Z) of one row at temperature T, in fp64: Z = sum_v exp((x_v - max) / T).

    The target's distribution at a node is p = softmax(x / T), so
    p(v) = exp((x_v - max) / T) / Z (the speculative-decoding lesson's
    sampling setting; T = 1 is plain sampling, T -> 0 greedy decoding)."""
    x = np.asarray(row, dtype=np.float64)
    m = x.max()
    return m, float(np.exp((x - m) / T).sum())


def target_probs(row, T):
    """The target's sampling distribution softmax(row / T) at one node, fp64."""
    m, Z = softmax_stats(row, T)
    return np.exp((np.asarray(row, dtype=np.float64) - m) / T) / Z


def accept_sampled(plan, tok, logits, T, U):
    """Acceptance under sampling at temperature T: the path taken, the tokens
    committed, and how close each decision came to its threshold.

    Speculative-decoding lesson, the acceptance rule: walking the draft, a
    drafted token x is accepted with probability min(1, p(x) / q(x)); on the
    first rejection the token is resampled from norm(max(0, p - q)), and when
    every drafted token is accepted one more token is sampled from p (the
    bonus).  The output is then distributed exactly as sampling from p alone.
    hyper.ai summary, "Experiment": Token Recycling stays effective under
    sampling, but the pages give no rule for its tree.  The reading taken
    here: Token Recycling's draft is deterministic -- the child tokens are
    fixed by the matrix -- so each child's draft distribution q is one-hot on
    its token, and the rule is applied to a node's children in rank order:
    child x is accepted with probability min(1, r(x) / 1) = r(x) under the
    current residual r (at first r = p); when it is rejected,
    r <- norm(max(0, r - onehot(x))), which zeroes r(x) and renormalises, and
    the next child is tried.  An accepted child's node becomes the current
    node and the walk continues with its own distribution; when every child
    of the current node is rejected (or it has none), the next token is drawn
    from the residual r there.  T -> 0 is greedy Token Recycling.

    The random numbers are inputs: U [N, K+1] uniforms in [0, 1); the i-th
    child test at node n compares U[n, i] with r(x) (accept when smaller), and
    the draw at the final node n* is the inverse CDF of r at U[n*, K] over
    token IDs in ascending order (the smallest v with r(0) + ... + r(v) >
    U[n*, K]).  logits [N, V]: the target's logits at every node.

    Returns (acc_len, path, committed, bonus, margins, cdf): margins =
    (smallest distance between a child test's uniform and its threshold,
    distance of U[n*, K] to the nearer end of the drawn token's CDF interval),
    so a caller can tell a decision that fp32 arithmetic could flip; cdf is the
    residual's CDF at n* (the tokens whose interval lies within a tolerance of
    U[n*, K] are the draws such arithmetic can make)."""
    K1 = np.asarray(U).shape[1]
    n, path, margin = 0, [0], np.inf
    while True:
        r = target_probs(logits[n], T)
        moved = False
        for i, c in enumerate(plan.children[n]):
            x = int(tok[c])
            u = float(U[n, i])
            margin = min(margin, abs(u - r[x]))
            if u < min(1.0, r[x]):
                n = c
                path.append(c)
                moved = True
                break
            r[x] = 0.0       # max(0, r - onehot(x)): every other entry is at most 1
            r = r / r.sum()
        if not moved:
            break
    u = float(U[n, K1 - 1])
    cdf = np.cumsum(r)
    y = int(np.searchsorted(cdf, u, side="right"))
    if y >= len(r):                          # rounding left the total just below u
        y = int(np.nonzero(r > 0)[0][-1])
    draw_margin = min(abs(cdf[y] - u), abs(u - (cdf[y - 1] if y > 0 else 0.0)))
    committed = [int(tok[m]) for m in path[1:]] + [y]
    return plan.depth[n], path, committed, y, (margin, draw_margin), cdf


def draw_is_valid(cdf, u, y, tol):
    """True when token y's interval [cdf(y-1), cdf(y)) of a residual CDF lies
    within tol of u: a draw that arithmetic with error below tol can make."""
    lo = cdf[y - 1] if y > 0 else 0.0
    return cdf[y] > lo and lo - tol <= u < cdf[y] + tol


def update(M, tok, ids, plan, mode=UPD_ALL, path=None):
    """Overwrite the matrix rows of the verified nodes with their top-K.

    Chinese hyper.ai summary, "方法": M[x~_i] = argtopk(p~_{i+1}) for every
    draft token of the verified sequence; duplicates get no conflict logic.
    Blog "token-recycling", 为什么叫 Token Recycling: nodes on rejected
    branches write their rows too.  A plain loop in BFS order, so when a token
    appears at several nodes the last one written stays (the listed reading of
    "no conflict logic").  UPD_ACCEPTED is the ablation that updates from the
    accepted path only (hyper.ai summary, "Experiment").
    """
    keep = set(path) if mode == UPD_ACCEPTED else None
    for n in range(plan.N):
        if keep is None or n in keep:
            M[tok[n]] = ids[n]
    return M


def kv_commit(kc, vc, kt, vt, L, path):
    """Append the K/V rows of the root and the accepted nodes to the cache.

    The pages are silent here; this is standard tree decoding (a listed
    reading): the root (the previous bonus, which had no KV yet) and the
    accepted nodes join the cache in path order at positions L, L+1, ...;
    the new bonus waits for the next step.  Returns the new length.
    """
    for i, n in enumerate(path):
        kc[:, L + i] = kt[n]
        vc[:, L + i] = vt[n]
    return L + len(path)


def lmhead_logits(H, Wt):
    """Logits of the fused LM head: H [R, D] times Wt [V, D] transposed, in fp64."""
    return np.asarray(H, dtype=np.float64) @ np.asarray(Wt, dtype=np.float64).T
