"""Multi-step parity of the CUDA Token Recycling loop against the oracle (GB300 only).

The GPU loop runs exactly the calls the benchmark times (tr_verify_attn, then
tr_step: top-K or fused LM head + top-K, acceptance, update, KV commit, next
retrieval); the synthetic target is generated on the device.  The oracle
replays the same seeded loop on the CPU.  Integer state must be bit-exact at
every step (tree tokens, top-K IDs, accepted lengths, paths, committed
tokens, every matrix row); attention within 2e-3 per (node, head) row.

Full-size runs are checked on samples the oracle can afford and on the
losslessness invariant (the committed stream equals plain greedy decoding
under the target), which holds at any size.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import compare_step, oracle_qkv, oracle_states, rows_rel_err, run_gpu_loop, target_fn, ATTN_TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from free_speculative_decoding_gb300 import build as b
    b.build()


def _check_loop(w, steps, seqs=None, attn=True, M_every=1, init="warm", mode=0):
    plan = oracle.TreePlan(w.child_counts, w.K)
    recs, st, status = run_gpu_loop(w, steps, keep_M_every=M_every, init=init, mode=mode)
    assert status == 0
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    states = oracle_states(w, seqs, with_cache=attn and w.attention, init=init)
    target = target_fn(w)

    def on_step(s, i, rec):
        b = seqs[i]
        compare_step(w, plan, s, i, b, rec, recs[s], attn=attn)
        if "M" in recs[s]:
            assert np.array_equal(recs[s]["M"][b], states[i].M), "M after step %d seq %d" % (s, b)

    oracle.tr_loop(plan, states, target, steps, w.K, mode=mode,
                   qkv=oracle_qkv(w, seqs) if (attn and w.attention) else None,
                   scale=w.d ** -0.5, on_step=on_step, seqs=seqs)
    return recs


def test_tiny_loop_full_config():
    """One sequence, 80-node tree, V=32000 int64, prefix 512, 64 steps, 32 heads."""
    w = synth.WORKLOADS["tiny"]
    recs = _check_loop(w, w.steps)
    mat = np.mean([r["acc_len"][0] + 1 for r in recs])
    assert mat > 1.5   # acceptance is nontrivial on this target


@pytest.mark.parametrize("tree", ["W80", "D80"])
def test_tree_shape_sweep_loop(tree):
    """The sweep's wide and deep 80-node trees through the same loop."""
    w = synth.WORKLOADS["tiny"].scaled(tree=tree, steps=8)
    _check_loop(w, w.steps)


def test_batched_reduced():
    """Sequences with their own matrices and ragged prefixes (1k..4k)."""
    w = synth.WORKLOADS["batched"].scaled(B=3, steps=10)
    _check_loop(w, w.steps)


def test_gqa_large_vocab_reduced():
    """V=128256, int32 matrix, 128-node tree, bf16 logits, 32/8 grouped-query heads."""
    w = synth.WORKLOADS["gqa"].scaled(B=2, steps=3)
    _check_loop(w, w.steps)


def test_long_context_reduced():
    """Prefix 32768 (the full length), 128-node tree."""
    w = synth.WORKLOADS["long"].scaled(B=1, steps=2)
    _check_loop(w, w.steps)


def test_lmhead_loop_reduced():
    """Fused LM head (D=4096, V=32000) feeding accept and update."""
    w = synth.WORKLOADS["lmhead"].scaled(B=3, steps=4)
    _check_loop(w, w.steps, attn=False)


@pytest.mark.parametrize("init", ["zero", "random", "warm"])
@pytest.mark.parametrize("mode", [0, 1], ids=["update_all", "update_accepted"])
def test_init_and_update_ablation_loops(init, mode):
    """The hyper.ai summary's ablations ("Experiment": all-zero, random and
    inherited initial matrices; updates from all draft tokens or from the
    accepted ones only) through the whole GPU loop: tr_init_matrix starts the
    matrices, tr_step runs with the chosen update rule, and every step's
    integer state and matrix equal the oracle's."""
    w = synth.WORKLOADS["batched"].scaled(B=2, steps=5, prefix=(100, 300))
    _check_loop(w, w.steps, init=init, mode=mode)


def test_loop_from_random_init_full_vocab():
    """The tiny workload's loop started from tr_init_matrix(RANDOM) at V=32000
    instead of a copied matrix."""
    w = synth.WORKLOADS["tiny"].scaled(steps=6)
    _check_loop(w, w.steps, init="random")


def test_finish_grid_beyond_one_wave():
    """128 sequences x (1 + 8) step-end CTAs: more than one wave of the step-end
    kernel, so some KV-commit CTAs start after their sequence's CTA 0 has left
    the next tree.  Tree tokens, acceptance, L and every committed cache row
    must still equal the oracle's."""
    w = synth.WORKLOADS["batched"].scaled(B=128, V=4096, Hq=8, Hkv=8, prefix=(64, 192), steps=3)
    plan = oracle.TreePlan(w.child_counts, w.K)
    recs, st, status = run_gpu_loop(w, w.steps, keep_M_every=1, o_seqs=[0, 77])
    assert status == 0
    states = oracle_states(w, range(w.B), with_cache=True)
    target = target_fn(w)

    def on_step(s, i, rec):
        compare_step(w, plan, s, i, i, rec, recs[s], attn=i in (0, 77))
        assert np.array_equal(recs[s]["M"][i], states[i].M), "M after step %d seq %d" % (s, i)

    oracle.tr_loop(plan, states, target, w.steps, w.K, qkv=oracle_qkv(w), scale=w.d ** -0.5, on_step=on_step)
    Lg = st.L.cpu().numpy()
    Kc = st.Kc.float().cpu().numpy()
    Vc = st.Vc.float().cpu().numpy()
    for b in range(w.B):
        assert Lg[b] == states[b].L
        assert np.array_equal(Kc[b, :, :Lg[b]], states[b].kc[:, :Lg[b]]), "K cache of seq %d" % b
        assert np.array_equal(Vc[b, :, :Lg[b]], states[b].vc[:, :Lg[b]]), "V cache of seq %d" % b


def test_accepted_only_update_mode():
    import free_speculative_decoding_gb300 as tr
    from free_speculative_decoding_gb300.engine import TRState
    from synth import device as sd
    w = synth.WORKLOADS["tiny"].scaled(steps=6)
    plan = oracle.TreePlan(w.child_counts, w.K)
    tree = tr.Tree(w.child_counts, w.K)
    st = TRState(tree, 1, w.V)
    sd.warm_matrices(w, st)
    st.start(synth.initial_roots(w), w.prefix_lengths(), M_src=st.M.clone())
    tgt = sd.DeviceTarget(w, tree)
    for _ in range(w.steps):
        st.finish(logits=tgt.logits_for(st), mode=tr.TR_UPD_ACCEPTED)
    ostate = oracle_states(w, [0], with_cache=False)
    oracle.tr_loop(plan, ostate, target_fn(w), w.steps, w.K, mode=oracle.UPD_ACCEPTED)
    assert np.array_equal(st.M[0].cpu().numpy(), ostate[0].M)
    assert st.root.item() == ostate[0].root and st.L.item() == ostate[0].L


# ----------------------------------------------------------------------------
# full-size workloads, in the benchmark's launch configuration
# ----------------------------------------------------------------------------

def _greedy_ok(w, b, emitted, L0, root):
    def top1(pos, x):
        return int(np.argmax(synth.logits_f32(w.seed, b, pos, [x], w.V, w.logits)[0]))
    return emitted == oracle.greedy_decode(top1, root, L0, len(emitted))


def _emitted(recs, b):
    out = []
    for r in recs:
        a = int(r["acc_len"][b])
        out.extend(int(x) for x in r["committed"][b][:a + 1])
    return out


def test_batched_full_size_samples_and_losslessness():
    """16 sequences x 256 steps: losslessness on sampled sequences, full integer
    replay of one sequence over the first 48 steps, attention at step 0."""
    w = synth.WORKLOADS["batched"]
    b = 5
    recs, st, status = run_gpu_loop(w, w.steps, keep_M_every=0, o_seqs=[b])
    assert status == 0
    L0, roots = w.prefix_lengths(), synth.initial_roots(w)
    for bb in (0, 7, 15):
        em = _emitted(recs, bb)
        assert len(em) >= w.steps
        assert _greedy_ok(w, bb, em, int(L0[bb]), int(roots[bb]))
    plan = oracle.TreePlan(w.child_counts, w.K)
    states = oracle_states(w, [b], with_cache=True)
    steps = 48

    def on_step(s, i, rec):
        compare_step(w, plan, s, i, b, rec, recs[s], attn=True)

    oracle.tr_loop(plan, states, target_fn(w), steps, w.K, qkv=oracle_qkv(w, [b]), scale=w.d ** -0.5,
                   on_step=on_step, seqs=[b])
    assert sum(int(r["acc_len"][b]) + 1 for r in recs[:steps]) == states[0].L - int(L0[b])


def test_gqa_full_size_losslessness():
    w = synth.WORKLOADS["gqa"].scaled(steps=24)
    recs, st, status = run_gpu_loop(w, w.steps, keep_M_every=0, o_seqs=[3], o_steps={0})
    assert status == 0
    L0, roots = w.prefix_lengths(), synth.initial_roots(w)
    for b in (0, 5):
        assert _greedy_ok(w, b, _emitted(recs, b), int(L0[b]), int(roots[b]))
    # attention of sampled nodes at step 0 in fp64
    plan = oracle.TreePlan(w.child_counts, w.K)
    st0 = oracle_states(w, [3], with_cache=True)[0]
    q, kt, vt = synth.step_qkv(w, 0)
    ref = oracle.tree_attention(synth.bf16_to_f32(q[3]), st0.kc, st0.vc, st0.L, synth.bf16_to_f32(kt[3]),
                                synth.bf16_to_f32(vt[3]), plan, w.d ** -0.5)
    assert rows_rel_err(recs[0]["O"][0], ref) <= ATTN_TOL


def test_long_full_size_samples_and_losslessness():
    """4 sequences x prefix 32768, 128-node tree (the long-context workload at
    its full batch, in the benchmark's launch configuration): losslessness on
    every sequence, attention of two sampled heads of one sequence at step 0."""
    w = synth.WORKLOADS["long"].scaled(steps=10)
    b = 2
    recs, st, status = run_gpu_loop(w, w.steps, keep_M_every=0, o_seqs=[b], o_steps={0})
    assert status == 0
    L0, roots = w.prefix_lengths(), synth.initial_roots(w)
    for bb in range(w.B):
        em = _emitted(recs, bb)
        assert len(em) >= w.steps
        assert _greedy_ok(w, bb, em, int(L0[bb]), int(roots[bb]))
    plan = oracle.TreePlan(w.child_counts, w.K)
    q, kt, vt = synth.step_qkv(w, 0, [b])
    L = int(L0[b])
    pos = np.arange(L)
    for h in (0, 17):
        kc = synth.bf16_to_f32(synth.kc_rows(w.seed, b, np.full(L, h), pos, w.d)).reshape(1, L, w.d)
        vc = synth.bf16_to_f32(synth.vc_rows(w.seed, b, np.full(L, h), pos, w.d)).reshape(1, L, w.d)
        ref = oracle.tree_attention(synth.bf16_to_f32(q[0][:, h:h + 1]), kc, vc, L,
                                    synth.bf16_to_f32(kt[0][:, h:h + 1]), synth.bf16_to_f32(vt[0][:, h:h + 1]),
                                    plan, w.d ** -0.5)
        assert rows_rel_err(recs[0]["O"][0][:, h:h + 1], ref) <= ATTN_TOL


def test_lmhead_full_size_losslessness_and_replay():
    """32 sequences x 80 nodes = 2560 LM-head rows per step (the fused LM-head
    workload at its full size): losslessness on sampled sequences and the
    full integer replay of one sequence."""
    w = synth.WORKLOADS["lmhead"].scaled(steps=5)
    recs, st, status = run_gpu_loop(w, w.steps, keep_M_every=w.steps)
    assert status == 0
    target = target_fn(w)
    L0, roots = w.prefix_lengths(), synth.initial_roots(w)
    for bb in (0, 31):
        def top1(pos, x, bb=bb):
            return int(np.argmax(target(bb, pos, [x])[0]))
        em = _emitted(recs, bb)
        assert em == oracle.greedy_decode(top1, int(roots[bb]), int(L0[bb]), len(em))
    b = 13
    plan = oracle.TreePlan(w.child_counts, w.K)
    states = oracle_states(w, [b], with_cache=False)

    def on_step(s, i, rec):
        compare_step(w, plan, s, i, b, rec, recs[s], attn=False)

    oracle.tr_loop(plan, states, target, w.steps, w.K, qkv=None, on_step=on_step, seqs=[b])
    assert np.array_equal(recs[-1]["M"][b], states[0].M)
