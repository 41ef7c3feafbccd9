"""Seeded synthetic inputs for the Token Recycling hot path.

This module is shared by the oracle tests, the GPU parity tests and the
benchmark, and by nothing else.  It holds no Token Recycling arithmetic: it
only produces *inputs* -- the workload shapes, the static draft-tree specs, a
synthetic target model's logits and hidden states, the attention operands and a
warm-start adjacency matrix.

Randomness comes from one counter-based generator, splitmix64 (Steele, Lea and
Flood, "Fast Splittable Pseudorandom Number Generators", OOPSLA 2014): the
i-th output of a stream started at state ``s`` is ``mix64(s + (i+1)*GAMMA)``.
Keys are chained field by field, ``h <- mix64(h + GAMMA + field)``, so every
value is a pure function of (seed, tag, indices) and can be regenerated one
row at a time.  The CUDA library carries its own implementation of the same
definition for generating the workload on the device; a GPU test compares the
two bit for bit.

Normal-looking noise is Irwin-Hall of twelve 16-bit uniforms, centred and
scaled by 2^-16: mean 0, standard deviation ~1, support [-6, 6], and every value
is exact in fp32 (an integer below 2^19 times 2^-16).  This stands in for N(0,1)
wherever the workloads ask for it; the truncation at 6 sigma is the only
difference that matters.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB

# field tags, one per kind of generated value
TAG_NEXT, TAG_ALT, TAG_NOISE, TAG_PREFIX, TAG_WARM = 1, 2, 3, 4, 5
TAG_Q, TAG_KT, TAG_VT, TAG_KC, TAG_VC = 6, 7, 8, 9, 10
TAG_ROOT, TAG_H, TAG_W, TAG_CLASS, TAG_E, TAG_G = 11, 12, 13, 14, 15, 16
TAG_U = 17

N_ALT = 7            # seeded alternates per token
BOOST_NEXT = 6.0     # logit boost of the Markov successor
BOOST_ALT = 3.0      # logit boost of each alternate
IH_CENTRE = 393210   # 12 * 32767.5
IH_SCALE = 2.0 ** -16

# fused LM-head workload: hidden states on a 2^-5 grid, weights on a 2^-10 grid,
# so every product is a multiple of 2^-15 and every fp32 partial sum is exact.
LM_CLASSES = 16
LM_H_GRID = 32.0
LM_W_GRID = 1024.0
LM_E_AMP = 0.25          # +-amplitude of a class pattern in the hidden state
LM_W_BIAS = 8.0 / 1024   # +-amplitude of the pattern in the successor's column
LM_W_STD = 0.02


# ----------------------------------------------------------------------------
# splitmix64
# ----------------------------------------------------------------------------

def mix64(z):
    """splitmix64 output function on uint64 arrays (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_C1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_C2)
        return z ^ (z >> np.uint64(31))


def hkey(*fields):
    """Chain integer fields (scalars or broadcastable arrays) into one key."""
    h = np.uint64(0)
    with np.errstate(over="ignore"):
        for f in fields:
            f = np.asarray(f).astype(np.uint64)
            h = mix64(h + np.uint64(GAMMA) + f)
    return h


def stream(key, i):
    """i-th output of the splitmix64 stream whose state starts at ``key``."""
    key = np.asarray(key, dtype=np.uint64)
    i = np.asarray(i).astype(np.uint64)
    with np.errstate(over="ignore"):
        return mix64(key + np.uint64(GAMMA) * (i + np.uint64(1)))


def irwin_hall12(key, i):
    """Element i of the noise stream at ``key`` as exact fp32 (shape broadcast)."""
    key = np.asarray(key, dtype=np.uint64)
    i = np.asarray(i).astype(np.uint64)
    total = np.zeros(np.broadcast(key, i).shape, dtype=np.int64)
    for j in range(3):
        w = stream(key, np.uint64(3) * i + np.uint64(j))
        for q in range(4):
            total += ((w >> np.uint64(16 * q)) & np.uint64(0xFFFF)).astype(np.int64)
    return ((total - IH_CENTRE).astype(np.float32) * np.float32(IH_SCALE)).astype(np.float32)


def bf16_bits(x):
    """Round fp32 to bf16 (round to nearest even); returns the uint16 bit pattern."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits):
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# static draft trees (per-level child counts, earlier = more probable)
# ----------------------------------------------------------------------------

def _levels(*levels):
    out = []
    for lv in levels:
        for count, times in lv:
            out.extend([count] * times)
    return tuple(out)


# 80 nodes, depth 6; the top-ranked path has child counts [8, 4, 2, 1, 1, 1].
TREE_T80 = _levels(
    [(8, 1)],
    [(4, 2), (3, 2), (2, 2), (1, 2)],
    [(2, 6), (1, 8), (0, 6)],
    [(1, 15), (0, 5)],
    [(1, 10), (0, 5)],
    [(1, 6), (0, 4)],
    [(0, 6)],
)

# 128 nodes, depth 8, same taper.
TREE_T128 = _levels(
    [(8, 1)],
    [(5, 1), (4, 2), (3, 2), (2, 2), (1, 1)],
    [(3, 2), (2, 8), (1, 8), (0, 6)],
    [(2, 3), (1, 18), (0, 9)],
    [(1, 16), (0, 8)],
    [(1, 11), (0, 5)],
    [(1, 8), (0, 3)],
    [(1, 6), (0, 2)],
    [(0, 6)],
)

# Tree-shape sweep at the same 80-node budget (breadth against depth).
# W80: wide and shallow, depth 3 (level sizes 1, 8, 32, 39).
TREE_W80 = _levels(
    [(8, 1)],
    [(4, 8)],
    [(2, 7), (1, 25)],
    [(0, 39)],
)

# D80: narrow and deep, depth 11 (level sizes 1, 4, then 8 for nine levels, 3).
TREE_D80 = _levels(
    [(4, 1)],
    [(2, 4)],
    *([[(1, 8)]] * 8),
    [(1, 3), (0, 5)],
    [(0, 3)],
)

TREES = {"T80": TREE_T80, "T128": TREE_T128, "W80": TREE_W80, "D80": TREE_D80}


def chain_tree(depth):
    """A linear draft: every node has one child."""
    return tuple([1] * depth + [0])


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    V: int
    K: int
    m_dtype: str          # "int64" | "int32"
    tree: str             # key of TREES
    B: int
    prefix: tuple         # (lo, hi): prefix length uniform in [lo, hi]
    Hq: int
    Hkv: int
    d: int
    steps: int
    logits: str           # "f32" | "bf16" | "lmhead"
    D: int = 0            # LM-head hidden size
    seed: int = 1
    attention: bool = True

    @property
    def child_counts(self):
        return TREES[self.tree]

    @property
    def N(self):
        return len(self.child_counts)

    def prefix_lengths(self):
        lo, hi = self.prefix
        if lo == hi:
            return np.full(self.B, lo, dtype=np.int32)
        b = np.arange(self.B)
        return (lo + hkey(self.seed, TAG_PREFIX, b) % np.uint64(hi - lo + 1)).astype(np.int32)

    def depth(self):
        return _tree_depth(self.child_counts)

    def capacity(self):
        return int(self.prefix[1]) + self.steps * (self.depth() + 1)

    def scaled(self, **kw):
        return replace(self, **kw)


def _tree_depth(child_counts):
    # depth of the deepest node of a BFS-ordered child-count list
    depth = [0]
    for n, c in enumerate(child_counts):
        depth.extend([depth[n] + 1] * c)
    return max(depth)


WORKLOADS = {
    # tiny loop: one sequence, 80-node tree, prefix 512, 64 steps
    "tiny": Workload("tiny", 32000, 8, "int64", "T80", 1, (512, 512), 32, 32, 128, 64, "f32", seed=11),
    # batched: 16 sequences, own M each, prefix uniform in 1k..4k, 256 steps
    "batched": Workload("batched", 32000, 8, "int64", "T80", 16, (1024, 4096), 32, 32, 128, 256, "f32", seed=22),
    # large vocabulary with grouped-query attention, bf16 logits
    "gqa": Workload("gqa", 128256, 8, "int32", "T128", 8, (4096, 4096), 32, 8, 128, 128, "bf16", seed=33),
    # long context: prefix 32768, split-KV verification dominates
    "long": Workload("long", 32000, 8, "int64", "T128", 4, (32768, 32768), 32, 32, 128, 64, "f32", seed=44),
    # fused LM head + top-K: 32 x 80 = 2560 hidden rows of width 4096
    "lmhead": Workload("lmhead", 32000, 8, "int64", "T80", 32, (0, 0), 32, 32, 128, 128, "lmhead",
                       D=4096, seed=55, attention=False),
}


# ----------------------------------------------------------------------------
# synthetic target: logits of a hidden Markov table plus noise
# ----------------------------------------------------------------------------

def markov_next(seed, b, tok, V):
    return (hkey(seed, TAG_NEXT, b, tok) % np.uint64(V)).astype(np.int64)


def markov_alt(seed, b, tok, V):
    """[..., N_ALT] alternates of each token."""
    tok = np.asarray(tok)
    j = np.arange(N_ALT)
    return (hkey(seed, TAG_ALT, np.asarray(b)[..., None], tok[..., None], j) % np.uint64(V)).astype(np.int64)


def logits_rows(seed, b, pos, tok, V, dtype="f32", v_lo=0, v_hi=None):
    """Logits of the synthetic target for rows (b, pos, tok) over vocab [v_lo, v_hi).

    The target depends on the context only through (sequence, position, last
    token), so it is a deterministic function of the context and greedy
    decoding under it is well defined.  Returns fp32, or bf16 bits (uint16)
    when dtype == "bf16".
    """
    b, pos, tok = np.broadcast_arrays(np.asarray(b), np.asarray(pos), np.asarray(tok))
    b, pos, tok = b.ravel(), pos.ravel(), tok.ravel()
    v_hi = V if v_hi is None else v_hi
    v = np.arange(v_lo, v_hi, dtype=np.int64)
    rk = hkey(seed, TAG_NOISE, b, pos, tok)
    x = irwin_hall12(rk[:, None], v[None, :])
    nxt = markov_next(seed, b, tok, V)
    alt = markov_alt(seed, b, tok, V)
    is_alt = (v[None, :, None] == alt[:, None, :]).any(axis=2)
    boost = np.where(v[None, :] == nxt[:, None], np.float32(BOOST_NEXT),
                     np.where(is_alt, np.float32(BOOST_ALT), np.float32(0.0)))
    x = (x + boost.astype(np.float32)).astype(np.float32)
    if dtype == "bf16":
        return bf16_bits(x)
    return x


def logits_f32(seed, b, pos, tok, V, dtype="f32"):
    """Logits as fp32 values (bf16 rows widened exactly)."""
    x = logits_rows(seed, b, pos, tok, V, dtype)
    return bf16_to_f32(x) if dtype == "bf16" else x


# ----------------------------------------------------------------------------
# attention operands: bf16 rows of Irwin-Hall noise
# ----------------------------------------------------------------------------

def noise_rows_bf16(keys, d):
    """[len(keys), d] bf16 bit patterns, row r from the stream at keys[r]."""
    keys = np.asarray(keys, dtype=np.uint64).ravel()
    i = np.arange(d)
    return bf16_bits(irwin_hall12(keys[:, None], i[None, :]))


def q_rows(seed, step, b, n, h, d):
    return noise_rows_bf16(hkey(seed, TAG_Q, step, b, n, h), d)


def kt_rows(seed, step, b, n, h, d):
    return noise_rows_bf16(hkey(seed, TAG_KT, step, b, n, h), d)


def vt_rows(seed, step, b, n, h, d):
    return noise_rows_bf16(hkey(seed, TAG_VT, step, b, n, h), d)


def kc_rows(seed, b, h, pos, d):
    return noise_rows_bf16(hkey(seed, TAG_KC, b, h, pos), d)


def vc_rows(seed, b, h, pos, d):
    return noise_rows_bf16(hkey(seed, TAG_VC, b, h, pos), d)


def step_qkv(w: Workload, step, seqs=None):
    """Q [S,N,Hq,d], Kt/Vt [S,N,Hkv,d] of one step as bf16 bit patterns, for the
    sequences ``seqs`` (all B by default)."""
    seqs = np.arange(w.B) if seqs is None else np.asarray(seqs)
    S, N, Hq, Hkv, d = len(seqs), w.N, w.Hq, w.Hkv, w.d
    b, n, h = np.meshgrid(seqs, np.arange(N), np.arange(Hq), indexing="ij")
    q = q_rows(w.seed, step, b, n, h, d).reshape(S, N, Hq, d)
    b, n, h = np.meshgrid(seqs, np.arange(N), np.arange(Hkv), indexing="ij")
    kt = kt_rows(w.seed, step, b, n, h, d).reshape(S, N, Hkv, d)
    vt = vt_rows(w.seed, step, b, n, h, d).reshape(S, N, Hkv, d)
    return q, kt, vt


def initial_cache(w: Workload, cap=None):
    """K/V cache [B,Hkv,cap,d] bf16 bits, positions [0, L_b) filled, rest zero."""
    cap = w.capacity() if cap is None else cap
    L = w.prefix_lengths()
    kc = np.zeros((w.B, w.Hkv, cap, w.d), dtype=np.uint16)
    vc = np.zeros_like(kc)
    for b in range(w.B):
        hh, pp = np.meshgrid(np.arange(w.Hkv), np.arange(L[b]), indexing="ij")
        kc[b, :, :L[b]] = kc_rows(w.seed, b, hh, pp, w.d).reshape(w.Hkv, L[b], w.d)
        vc[b, :, :L[b]] = vc_rows(w.seed, b, hh, pp, w.d).reshape(w.Hkv, L[b], w.d)
    return kc, vc


# ----------------------------------------------------------------------------
# uniforms for acceptance under sampling
# ----------------------------------------------------------------------------

def uniforms(seed, step, b, N, K1):
    """[N, K1] uniforms in [0, 1) for sequence b at one step: entry (n, j) is
    the top 24 bits of output j of the stream keyed on (seed, step, b, n),
    times 2^-24, so every value is exact in fp32 and fp64."""
    key = hkey(seed, TAG_U, step, b, np.arange(N))
    j = np.arange(K1)
    return ((stream(key[:, None], j[None, :]) >> np.uint64(40)).astype(np.float64) * 2.0 ** -24).astype(np.float32)


# ----------------------------------------------------------------------------
# starting state
# ----------------------------------------------------------------------------

def initial_roots(w: Workload):
    return (hkey(w.seed, TAG_ROOT, np.arange(w.B)) % np.uint64(w.V)).astype(np.int32)


def warm_matrix(seed, b, V, K):
    """A stand-in for a matrix inherited from earlier requests.

    Rows whose key is even hold the target's successor followed by its
    alternates (what earlier decoding would have left there); the other rows
    hold uniform random IDs.  Returns int64 [V, K].
    """
    t = np.arange(V)
    good = (hkey(seed, TAG_WARM, b, t) & np.uint64(1)) == np.uint64(0)
    j = np.arange(K)
    rnd = (hkey(seed, TAG_WARM, b, t[:, None], j[None, :] + 1) % np.uint64(V)).astype(np.int64)
    learned = np.concatenate([markov_next(seed, b, t, V)[:, None], markov_alt(seed, b, t, V)], axis=1)
    if K <= learned.shape[1]:
        learned = learned[:, :K]
    else:
        learned = np.concatenate([learned, rnd[:, learned.shape[1]:]], axis=1)
    return np.where(good[:, None], learned, rnd)


# ----------------------------------------------------------------------------
# fused LM-head workload (hidden states and an output projection)
# ----------------------------------------------------------------------------

def lm_class(seed, tok):
    return (hkey(seed, TAG_CLASS, tok) % np.uint64(LM_CLASSES)).astype(np.int64)


def lm_pattern(seed, D):
    """[LM_CLASSES, D] signs (+1/-1) of each class pattern."""
    c, dd = np.meshgrid(np.arange(LM_CLASSES), np.arange(D), indexing="ij")
    return np.where((hkey(seed, TAG_E, c, dd) & np.uint64(1)) == np.uint64(0), 1.0, -1.0).astype(np.float32)


def lm_successor(seed, V):
    """Token that follows every token of class c under the synthetic target."""
    return (hkey(seed, TAG_G, np.arange(LM_CLASSES)) % np.uint64(V)).astype(np.int64)


def lm_hidden_rows(seed, b, pos, tok, D):
    """Hidden states [rows, D] as bf16 bits: grid-rounded noise plus the class pattern.

    Every value is a multiple of 2^-5 below 8 in magnitude, so bf16 holds it
    exactly.  Keyed on (sequence, position, token) like the logits target.
    """
    b, pos, tok = (np.asarray(a).ravel() for a in np.broadcast_arrays(np.asarray(b), np.asarray(pos), np.asarray(tok)))
    i = np.arange(D)
    noise = irwin_hall12(hkey(seed, TAG_H, b, pos, tok)[:, None], i[None, :])
    noise = np.rint(noise * np.float32(LM_H_GRID)) / np.float32(LM_H_GRID)
    pat = lm_pattern(seed, D)[lm_class(seed, tok)]
    return bf16_bits((noise + np.float32(LM_E_AMP) * pat).astype(np.float32))


def lm_weight_rows(seed, V, D, v_lo=0, v_hi=None):
    """Output projection stored vocabulary-major, Wt [V, D], as bf16 bits.

    Column v of W is grid-rounded N(0, 0.02^2)-like noise; the successor
    token of each class also carries that class's pattern, which biases the
    target toward a low-rank Markov table.
    """
    v_hi = V if v_hi is None else v_hi
    out = np.empty((v_hi - v_lo, D), dtype=np.uint16)
    i = np.arange(D)
    succ = lm_successor(seed, V)
    pat = lm_pattern(seed, D)
    for lo in range(v_lo, v_hi, _ROW_CHUNK):
        v = np.arange(lo, min(v_hi, lo + _ROW_CHUNK))
        noise = irwin_hall12(hkey(seed, TAG_W, v)[:, None], i[None, :]) * np.float32(LM_W_STD)
        w = np.rint(noise.astype(np.float32) * np.float32(LM_W_GRID)) / np.float32(LM_W_GRID)
        for c in range(LM_CLASSES):
            hit = v == succ[c]
            if hit.any():
                w[hit] += np.float32(LM_W_BIAS) * pat[c]
        out[lo - v_lo:lo - v_lo + len(v)] = bf16_bits(w.astype(np.float32))
    return out


_ROW_CHUNK = 1024


def lm_realistic(seed, rows, V, D):
    """Off-grid bf16 operands (H ~ N(0,1), Wt ~ N(0, 0.02^2)) for the tolerance test."""
    h = noise_rows_bf16(hkey(seed, TAG_H, 7, np.arange(rows)), D)
    wt = np.empty((V, D), dtype=np.uint16)
    for lo in range(0, V, _ROW_CHUNK):
        v = np.arange(lo, min(V, lo + _ROW_CHUNK))
        wn = irwin_hall12(hkey(seed, TAG_W, 7, v)[:, None], np.arange(D)[None, :])
        wt[lo:lo + len(v)] = bf16_bits((wn * np.float32(LM_W_STD)).astype(np.float32))
    return h, wt
