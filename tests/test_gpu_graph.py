"""A whole Token Recycling decoding loop captured in one CUDA graph (GB300 only).

Every step of the loop (tree attention, then tr_step: top-K, acceptance,
update, KV commit, next retrieval) is an asynchronous launch on the current
stream that allocates nothing and needs no host synchronisation, so several
steps can be recorded into one graph and replayed.  The replay must end in
exactly the state the eager loop reaches from the same start: matrices, cache
lengths, roots, next tree tokens and the committed cache rows.
"""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def test_graph_captured_steps_match_eager():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from free_speculative_decoding_gb300 import build as b
    b.build()
    import free_speculative_decoding_gb300 as tr
    from free_speculative_decoding_gb300.engine import TRState
    from synth import device as sd

    S = 6
    w = synth.WORKLOADS["batched"].scaled(B=4, steps=S, prefix=(300, 900))
    tree = tr.Tree(w.child_counts, w.K)
    N = tree.N
    st = TRState(tree, w.B, w.V, Hq=w.Hq, Hkv=w.Hkv, d=w.d, cap=w.capacity())
    tgt = sd.DeviceTarget(w, tree)
    sd.warm_matrices(w, st)
    sd.fill_cache(w, st)
    st.start(synth.initial_roots(w), w.prefix_lengths(), M_src=st.M.clone())

    names = ("M", "L", "root", "tree_tok", "Kc", "Vc")
    snap = {k: getattr(st, k).clone() for k in names}

    # the target depends on each step's tree: record every step's inputs eagerly
    q = torch.empty(S, w.B, N, w.Hq, w.d, dtype=torch.bfloat16, device="cuda")
    kt = torch.empty(S, w.B, N, w.Hkv, w.d, dtype=torch.bfloat16, device="cuda")
    vt = torch.empty_like(kt)
    logits = torch.empty(S, w.B * N, w.V, dtype=torch.float32, device="cuda")
    for s in range(S):
        sd.step_qkv(w, s, N, out=(q[s], kt[s], vt[s]))
        tgt.logits_for(st, logits[s])
        st.verify(q[s], kt[s], vt[s])
        st.finish(logits=logits[s], Kt=kt[s], Vt=vt[s])
    torch.cuda.synchronize()
    eager = {k: getattr(st, k).clone() for k in names}
    assert int((eager["L"] - snap["L"]).min()) >= S     # every step committed at least the root

    def restore():
        for k in names:
            getattr(st, k).copy_(snap[k])
        torch.cuda.synchronize()

    restore()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for s in range(S):
            st.verify(q[s], kt[s], vt[s])
            st.finish(logits=logits[s], Kt=kt[s], Vt=vt[s])
    torch.cuda.synchronize()
    for rep in range(2):    # the graph replays from the snapshot twice, identically
        restore()
        graph.replay()
        torch.cuda.synchronize()
        for k in names:
            assert torch.equal(getattr(st, k), eager[k]), "%s differs after replay %d" % (k, rep)
    assert tr.tr_get_status() == 0
