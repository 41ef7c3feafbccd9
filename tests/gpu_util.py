"""Helpers shared by the GPU tests: run the CUDA loop and the oracle loop on the
same seeded inputs and compare them step by step."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

ATTN_TOL = 2e-3     # per (node, head) row: max|O - O_ref| / max|O_ref|


def bf16_tensor(bits, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_numpy(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def rows_rel_err(o, ref):
    """max over rows of max|o - ref| / max|ref|, rows = all but the last axis."""
    o = np.asarray(o, np.float64).reshape(-1, o.shape[-1])
    ref = np.asarray(ref, np.float64).reshape(-1, ref.shape[-1])
    den = np.abs(ref).max(axis=1)
    return float((np.abs(o - ref).max(axis=1) / den).max())


def target_fn(w):
    if w.logits == "lmhead":
        Wt = synth.bf16_to_f32(synth.lm_weight_rows(w.seed, w.V, w.D)).astype(np.float64)

        def target(b, pos, tok):
            H = synth.bf16_to_f32(synth.lm_hidden_rows(w.seed, b, pos, tok, w.D))
            return oracle.lmhead_logits(H, Wt)
        return target

    def target(b, pos, tok):
        return synth.logits_f32(w.seed, b, pos, tok, w.V, w.logits)
    return target


def oracle_qkv(w, seqs=None):
    def qkv(step):
        q, kt, vt = synth.step_qkv(w, step, seqs)
        return synth.bf16_to_f32(q), synth.bf16_to_f32(kt), synth.bf16_to_f32(vt)
    return qkv


INIT_SEED = 0x5EED_0F_7E57   # seed of tr_init_matrix(RANDOM) in the loop tests


def oracle_matrix(w, b, init="warm"):
    """Sequence b's starting matrix on the oracle side.

    "warm": the synthetic inherited matrix of sequence b (the GPU copies it in,
    or inherits it through tr_init_matrix); "zero" / "random": what
    tr_init_matrix leaves (random at INIT_SEED)."""
    dt = np.int64 if w.m_dtype == "int64" else np.int32
    if init == "zero":
        return oracle.init_matrix(oracle.INIT_ZERO, w.V, w.K, dtype=dt)
    if init == "random":
        return oracle.init_matrix(oracle.INIT_RANDOM, w.V, w.K, seed=INIT_SEED, seq=b, dtype=dt)
    return synth.warm_matrix(w.seed, b, w.V, w.K).astype(dt)


def oracle_states(w, seqs=None, with_cache=True, init="warm"):
    seqs = range(w.B) if seqs is None else seqs
    L0 = w.prefix_lengths()
    roots = synth.initial_roots(w)
    states = []
    cap = w.capacity()
    for b in seqs:
        st = oracle.TRState(M=oracle_matrix(w, b, init), root=int(roots[b]), L=int(L0[b]))
        if with_cache and w.attention:
            st.kc = np.zeros((w.Hkv, cap, w.d), np.float32)
            st.vc = np.zeros((w.Hkv, cap, w.d), np.float32)
            hh, pp = np.meshgrid(np.arange(w.Hkv), np.arange(L0[b]), indexing="ij")
            st.kc[:, :L0[b]] = synth.bf16_to_f32(synth.kc_rows(w.seed, b, hh, pp, w.d)).reshape(w.Hkv, L0[b], w.d)
            st.vc[:, :L0[b]] = synth.bf16_to_f32(synth.vc_rows(w.seed, b, hh, pp, w.d)).reshape(w.Hkv, L0[b], w.d)
        states.append(st)
    return states


def gpu_start(w, st, init="warm"):
    """Initialise the matrices of a TRState and retrieve the first trees.

    "warm": every sequence inherits its own synthetic matrix through
    tr_init_matrix(INHERIT) (one call per sequence); "zero" / "random":
    tr_init_matrix over the whole batch."""
    import free_speculative_decoding_gb300 as tr
    from synth import device as sd
    roots, L0 = synth.initial_roots(w), w.prefix_lengths()
    if init == "warm":
        sd.warm_matrices(w, st)
        src = st.M.clone()
        for b in range(w.B):
            tr.tr_init_matrix(st.M[b:b + 1], tr.TR_INIT_INHERIT, src[b])
        st.start(roots, L0, M_src=None, mode=None)
    elif init == "zero":
        st.start(roots, L0, M_src=None, mode=tr.TR_INIT_ZERO)
    elif init == "random":
        st.start(roots, L0, M_src=None, mode=tr.TR_INIT_RANDOM, seed=INIT_SEED)
    else:
        raise ValueError(init)


U_SEED = 0xACC_E97      # seed of the acceptance uniforms in the sampling tests


def oracle_uniforms(w, N):
    return lambda step, b: synth.uniforms(U_SEED, step, b, N, w.K + 1)


def run_gpu_loop(w, steps, record=True, keep_M_every=1, o_seqs=None, o_steps=None, device="cuda",
                 init="warm", mode=0, temperature=None):
    """Run `steps` Token Recycling steps of workload w on the GPU; return per-step records.

    Attention outputs are kept for the sequences ``o_seqs`` at the steps
    ``o_steps`` (all by default).  ``init`` picks the starting matrices
    (gpu_start), ``mode`` the update rule (TR_UPD_ALL or TR_UPD_ACCEPTED).
    With ``temperature`` every step is tr_step_sampled with the uniforms of
    trsyn_uniforms(U_SEED, step)."""
    import free_speculative_decoding_gb300 as tr
    from free_speculative_decoding_gb300.engine import TRState
    from synth import device as sd

    tree = tr.Tree(w.child_counts, w.K)
    mdt = torch.int64 if w.m_dtype == "int64" else torch.int32
    ldt = torch.bfloat16 if w.logits == "bf16" else torch.float32
    cap = w.capacity()
    st = TRState(tree, w.B, w.V, m_dtype=mdt, Hq=w.Hq if w.attention else 0, Hkv=w.Hkv, d=w.d, cap=cap,
                 logits_dtype=ldt, D=w.D if w.logits == "lmhead" else 0, device=device)
    tgt = sd.DeviceTarget(w, tree, device)
    if w.attention:
        sd.fill_cache(w, st)
    gpu_start(w, st, init)
    U = torch.empty(w.B, tree.N, w.K + 1, dtype=torch.float32, device=device) if temperature else None
    recs = []
    for s in range(steps):
        rec = {"tok": st.tree_tok.cpu().numpy().copy(), "L": st.L.cpu().numpy().copy()}
        kt = vt = None
        if w.attention:
            q, kt, vt = sd.step_qkv(w, s, tree.N, device)
            st.verify(q, kt, vt)
            if record and (o_steps is None or s in o_steps):
                O = st.O if o_seqs is None else st.O[list(o_seqs)]
                rec["O"] = O.cpu().numpy().copy()
                rec["O_seqs"] = list(range(w.B)) if o_seqs is None else list(o_seqs)
        if w.logits == "lmhead":
            st.finish(H=tgt.hidden_for(st), Wt=tgt.Wt, Kt=kt, Vt=vt, mode=mode)
        elif temperature:
            tr.trsyn_uniforms(U_SEED, s, U)
            st.finish(logits=tgt.logits_for(st), Kt=kt, Vt=vt, mode=mode, temperature=temperature, U=U)
        else:
            st.finish(logits=tgt.logits_for(st), Kt=kt, Vt=vt, mode=mode)
        if record:
            rec.update(ids=st.ids.cpu().numpy().reshape(w.B, tree.N, w.K).copy(),
                       vals=st.vals.cpu().numpy().reshape(w.B, tree.N, w.K).copy(),
                       acc_len=st.acc_len.cpu().numpy().copy(), path=st.path.cpu().numpy().copy(),
                       committed=st.committed.cpu().numpy().copy(), root=st.root.cpu().numpy().copy())
            if keep_M_every and (s % keep_M_every == 0 or s == steps - 1):
                rec["M"] = st.M.cpu().numpy().copy()
        recs.append(rec)
    status = st.status()
    return recs, st, status


def compare_step(w, plan, s, i, b, rec_o, rec_g, attn=True):
    """Assert one sequence's oracle record equals the GPU record of step s."""
    D1 = plan.max_depth + 1
    assert np.array_equal(rec_g["tok"][b], rec_o["tok"]), "tree tokens, step %d seq %d" % (s, b)
    assert np.array_equal(rec_g["ids"][b], rec_o["ids"]), "top-K ids, step %d seq %d" % (s, b)
    assert rec_g["acc_len"][b] == rec_o["acc_len"], "acc_len, step %d seq %d" % (s, b)
    path = list(rec_o["path"]) + [-1] * (D1 - len(rec_o["path"]))
    assert list(rec_g["path"][b]) == path, "path, step %d seq %d" % (s, b)
    com = list(rec_o["committed"]) + [-1] * (D1 - len(rec_o["committed"]))
    assert list(rec_g["committed"][b]) == com, "committed, step %d seq %d" % (s, b)
    if attn and "O" in rec_o and "O" in rec_g:
        err = rows_rel_err(rec_g["O"][rec_g["O_seqs"].index(b)], rec_o["O"])
        assert err <= ATTN_TOL, "attention rel err %.3g, step %d seq %d" % (err, s, b)
