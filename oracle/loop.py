"""Multi-step Token Recycling loop and plain greedy decoding (test infrastructure only).

One step follows the order the blog "token-recycling" fixes (完整工作流程 and
the note on update timing): retrieve the whole tree from the old matrix,
verify it in one pass, accept the longest correct path plus the bonus, and
only then overwrite the matrix for the next step.  The target model is a
callback ``target(b, pos, tok) -> logits [len(tok), V]``; the tests supply the
synthetic one.  A node at depth k sits at position L + k, where L is the
number of cached positions before the step and the root sits at L.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .tr import UPD_ALL, accept, accept_sampled, kv_commit, retrieve, topk_rows, tree_attention, update


@dataclass
class TRState:
    """State of one sequence: its matrix, its root token and its cache length."""
    M: np.ndarray
    root: int
    L: int
    kc: np.ndarray | None = None   # [Hkv, cap, d]
    vc: np.ndarray | None = None
    emitted: list = field(default_factory=list)


def tr_loop(plan, states, target, steps, K, mode=UPD_ALL, qkv=None, scale=None,
            on_step=None, seqs=None, temperature=None, uniforms=None):
    """Run ``steps`` Token Recycling steps over the sequences in ``states``.

    ``qkv(step)`` (optional) returns (q [B,N,Hq,d], kt [B,N,Hkv,d],
    vt [B,N,Hkv,d]) as float arrays; with it the step also computes tree
    attention and commits the accepted K/V rows to each cache.  ``seqs``
    maps state index to the sequence index handed to the target.
    ``on_step(step, b, rec)`` receives every sequence's record.
    With ``temperature`` the acceptance samples (accept_sampled) with the
    uniforms ``uniforms(step, b)`` [N, K+1]; the matrix update is the same
    top-K of every node either way.
    """
    seqs = list(range(len(states))) if seqs is None else list(seqs)
    depth = np.asarray(plan.depth)
    for s in range(steps):
        q = kt = vt = None
        if qkv is not None:
            q, kt, vt = qkv(s)
        for i, st in enumerate(states):
            b = seqs[i]
            tok = retrieve(st.M, st.root, plan)
            rec = {"tok": tok, "L": st.L, "root": st.root}
            if q is not None:
                rec["O"] = tree_attention(q[i], st.kc, st.vc, st.L, kt[i], vt[i], plan, scale)
            rows = target(b, st.L + depth, tok)
            ids, vals = topk_rows(rows, K)
            rec["ids"], rec["vals"] = ids, vals
            if temperature is None:
                acc_len, path, committed, bonus = accept(plan, tok, ids[:, 0])
            else:
                acc_len, path, committed, bonus, rec["margins"], rec["cdf"] = accept_sampled(
                    plan, tok, rows, temperature, uniforms(s, b))
                rec["u_draw"] = float(uniforms(s, b)[path[-1], -1])
            update(st.M, tok, ids, plan, mode, path)
            if q is not None:
                st.L = kv_commit(st.kc, st.vc, kt[i], vt[i], st.L, path)
            else:
                st.L += len(path)
            st.root = bonus
            st.emitted.extend(committed)
            rec.update(acc_len=acc_len, path=path, committed=committed, bonus=bonus)
            if on_step is not None:
                on_step(s, i, rec)
    return states


def greedy_decode(top1, root, L, n_tokens):
    """Plain greedy decoding: the token stream the target alone would emit.

    ``top1(pos, tok)`` is the target's most probable next token after ``tok``
    at position ``pos`` (lowest ID on ties).  Speculative-decoding lesson:
    greedy speculative decoding matches this stream token for token.
    """
    out, x, pos = [], int(root), int(L)
    for _ in range(n_tokens):
        x = int(top1(pos, x))
        out.append(x)
        pos += 1
    return out
