"""Acceptance under sampling on the GPU against the oracle (GB300 only).

The speculative-decoding lesson's acceptance rule, applied to Token
Recycling's deterministic children (oracle.accept_sampled states the
reading): the top-K also returns each row's softmax statistics, the fused
step end walks the tree with the uniforms given as inputs, and the token after
the accepted path is drawn from the final node's residual distribution.

The kernels compute in fp32 (the draw's running sums compensated, its scan in
fp64) and the oracle in fp64, so a decision whose uniform lies within the
arithmetic's error of its threshold may go either way; the oracle reports
each step's margins.  A child test within TOL_TEST of its threshold ends the
comparison of that sequence (its path may legitimately differ).  Otherwise
the path must be bit-exact, and so must the drawn token wherever the draw's
margin exceeds TOL_DRAW; below it the token must be a valid draw (its CDF
interval within TOL_DRAW of the uniform), and a different valid token also
ends that sequence's comparison.  Such endings are counted and must be rare.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import U_SEED, compare_step, oracle_qkv, oracle_states, oracle_uniforms, run_gpu_loop, target_fn

pytestmark = pytest.mark.gpu

# probability units, ~5x the arithmetic's error: a child threshold r(x) uses the
# top-K pass's fp32 normaliser (relative error up to ~1e-6); the draw's running
# sum errs by the weights' own fp32 rounding only (~1e-7)
TOL_TEST = 4e-6
TOL_DRAW = 1e-6


@pytest.fixture(scope="module")
def tr():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from free_speculative_decoding_gb300 import build as b
    b.build()
    import free_speculative_decoding_gb300 as m
    return m


def test_device_uniforms_match_numpy(tr):
    out = torch.empty(3, 80, 9, dtype=torch.float32, device="cuda")
    tr.trsyn_uniforms(U_SEED, 5, out)
    got = out.cpu().numpy()
    for b in range(3):
        assert np.array_equal(got[b], synth.uniforms(U_SEED, 5, b, 80, 9))
    assert got.min() >= 0.0 and got.max() < 1.0


@pytest.mark.parametrize("rows,V,K,dtype,T", [
    (80, 32000, 8, torch.float32, 0.5),      # rows of 16 steps split between warps
    (1280, 32000, 8, torch.float32, 1.0),
    (64, 128256, 8, torch.bfloat16, 0.7),
    (40, 2000, 8, torch.float32, 0.3),       # one step per row: no split rows
    (33, 20480, 16, torch.bfloat16, 2.0),
])
def test_topk_softmax_statistics(tr, rows, V, K, dtype, T):
    """Top-K identical to tr_topk; stats = (row maximum exactly, Z within 1e-5
    relative of the fp64 sum)."""
    w = synth.WORKLOADS["tiny"]
    tok = np.arange(rows) * 7919 % V
    x = synth.logits_rows(w.seed, 0, np.arange(rows), tok, V, "bf16" if dtype == torch.bfloat16 else "f32")
    xf = synth.bf16_to_f32(x) if dtype == torch.bfloat16 else x
    xd = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) if dtype == torch.bfloat16
          else torch.from_numpy(x)).cuda()
    ids = torch.zeros(rows, K, dtype=torch.int32, device="cuda")
    vals = torch.zeros(rows, K, dtype=torch.float32, device="cuda")
    stats = torch.zeros(rows, 2, dtype=torch.float32, device="cuda")
    S = tr.tr_softmax_steps(V, dtype)
    E = 8192 // (4 if dtype == torch.float32 else 2)
    assert S == -(-V // E)
    sstats = torch.zeros(rows, S, 2, dtype=torch.float32, device="cuda")
    ws = tr.workspace(tr.tr_topk_workspace_bytes(rows, V, K))
    ids_ref, vals_ref = oracle.topk_rows(xf, K)
    for _ in range(2):
        tr.tr_topk_softmax(xd, K, T, ids, vals, stats, sstats, ws)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        assert np.array_equal(vals.cpu().numpy(), vals_ref.astype(np.float32))
        st, sst = stats.cpu().numpy(), sstats.cpu().numpy()
        for r in range(rows):
            m, Z = oracle.softmax_stats(xf[r], T)
            assert st[r, 0] == m
            assert abs(st[r, 1] - Z) <= 1e-5 * Z, (r, st[r, 1], Z)
            for k in range(S):   # every step: (its maximum, its sum against that maximum)
                ms, Zs = oracle.softmax_stats(xf[r, k * E:(k + 1) * E], T)
                assert sst[r, k, 0] == ms and abs(sst[r, k, 1] - Zs) <= 1e-5 * Zs, (r, k)
    assert tr.tr_get_status() == 0


@pytest.mark.parametrize("dtype,T", [("f32", 0.4), ("bf16", 0.6), ("f32", 1.0)])
def test_accept_sampled_matches_oracle(tr, dtype, T):
    """tr_accept_sampled on synthetic-target logits of random-token trees (T80
    and T128), many uniforms: path, accepted length, committed tokens and the
    drawn token equal the oracle's wherever its margins exceed the tolerances."""
    rng = np.random.default_rng(17)
    exceptions = checked = near_draws = other_valid = 0
    for trial in range(6):
        counts = synth.TREE_T80 if trial % 2 == 0 else synth.TREE_T128
        tree, plan = tr.Tree(counts, 8), oracle.TreePlan(counts, 8)
        B, V, N = 8, 32000 if trial < 4 else 5003 * 8, plan.N
        w = synth.WORKLOADS["tiny"].scaled(V=V)
        M = rng.integers(0, V, (B, V, 8))
        # plant the target's successors so that acceptance goes deep
        nxt = synth.markov_next(w.seed, 0, np.arange(V), V)
        keep = rng.random((B, V)) < 0.7
        M[:, :, 0] = np.where(keep, nxt[None, :], M[:, :, 0])
        roots = rng.integers(0, V, B)
        tok = np.stack([oracle.retrieve(M[b], roots[b], plan) for b in range(B)])
        pos = 100 + np.asarray(plan.depth)
        x = np.concatenate([synth.logits_rows(w.seed, 0, pos, tok[b], V, dtype) for b in range(B)])
        xf = synth.bf16_to_f32(x) if dtype == "bf16" else x
        xd = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) if dtype == "bf16"
              else torch.from_numpy(x)).cuda()
        U = np.stack([synth.uniforms(U_SEED + trial, 0, b, N, 9) for b in range(B)])
        ids = torch.zeros(B * N, 8, dtype=torch.int32, device="cuda")
        stats = torch.zeros(B * N, 2, dtype=torch.float32, device="cuda")
        sstats = torch.zeros(B * N, tr.tr_softmax_steps(V, xd.dtype), 2, dtype=torch.float32, device="cuda")
        tr.tr_topk_softmax(xd, 8, T, ids, None, stats, sstats,
                           tr.workspace(tr.tr_topk_workspace_bytes(B * N, V, 8)))
        tokd = torch.from_numpy(tok.astype(np.int32)).cuda()
        acc = torch.zeros(B, dtype=torch.int32, device="cuda")
        path = torch.zeros(B, plan.max_depth + 1, dtype=torch.int32, device="cuda")
        com = torch.zeros_like(path)
        bonus = torch.zeros(B, dtype=torch.int32, device="cuda")
        tr.tr_accept_sampled(tree, tokd, ids.view(B, N, 8), xd, stats, sstats, T, torch.from_numpy(U).cuda(), acc,
                             path, com, bonus)
        assert tr.tr_get_status() == 0
        for b in range(B):
            a, p, c, y, (tm, dm), cdf = oracle.accept_sampled(plan, tok[b], xf[b * N:(b + 1) * N], T, U[b])
            if tm < TOL_TEST:
                exceptions += 1
                continue
            checked += 1
            D1 = plan.max_depth + 1
            assert acc[b].item() == a, (trial, b)
            assert path[b].tolist() == p + [-1] * (D1 - len(p))
            yg = bonus[b].item()
            if dm >= TOL_DRAW:
                assert yg == y, (trial, b, yg, y, dm)
            else:
                near_draws += 1
                assert oracle.draw_is_valid(cdf, float(U[b][p[-1], -1]), yg, TOL_DRAW), (trial, b, yg, y)
                other_valid += yg != y
            assert com[b].tolist() == c[:-1] + [yg] + [-1] * (D1 - len(c))
    assert exceptions <= 1 and checked >= 47
    print("sampled acceptance: %d checked, %d child tests within %.0e, %d draws within %.0e (%d drew another "
          "valid token)" % (checked, exceptions, TOL_TEST, near_draws, TOL_DRAW, other_valid))


def _check_sampled_loop(w, T, seqs=None):
    plan = oracle.TreePlan(w.child_counts, w.K)
    recs, st, status = run_gpu_loop(w, w.steps, keep_M_every=1, temperature=T)
    assert status == 0
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    states = oracle_states(w, seqs, with_cache=w.attention)
    diverged, compared = {}, [0]

    def on_step(s, i, rec):
        b = seqs[i]
        if b in diverged:
            return
        tm, dm = rec["margins"]
        if tm < TOL_TEST:
            diverged[b] = (s, "child test within %.1e" % tm)
            return
        yg = int(recs[s]["root"][b])
        if dm < TOL_DRAW:
            assert oracle.draw_is_valid(rec["cdf"], rec["u_draw"], yg, TOL_DRAW), (s, b)
            if yg != rec["bonus"]:
                diverged[b] = (s, "another valid draw")
                return
        compare_step(w, plan, s, i, b, rec, recs[s], attn=True)
        assert np.array_equal(recs[s]["M"][b], states[i].M), "M after step %d seq %d" % (s, b)
        compared[0] += 1

    oracle.tr_loop(plan, states, target_fn(w), w.steps, w.K, qkv=oracle_qkv(w, seqs) if w.attention else None,
                   scale=w.d ** -0.5, on_step=on_step, seqs=seqs, temperature=T, uniforms=oracle_uniforms(w, plan.N))
    print("sampled loop %s at T=%g: %d sequence-steps compared, ended early: %s"
          % (w.name, T, compared[0], diverged or "none"))
    return recs, diverged, compared[0]


def test_sampled_loop_tiny_workload():
    """The tiny workload (V=32000 int64, 80-node tree, prefix 512, 32 heads)
    under sampling at T = 0.3 (the target's successor then has p ~ 0.9) for
    32 steps: every step's integer state and the matrix equal the oracle's,
    attention within 2e-3."""
    w = synth.WORKLOADS["tiny"].scaled(steps=32)
    recs, diverged, compared = _check_sampled_loop(w, 0.3)
    assert compared >= 24
    mat = np.mean([r["acc_len"][0] + 1 for r in recs])
    assert mat > 1.2   # acceptance under sampling is nontrivial on this target


@pytest.mark.parametrize("wl,B,steps,T", [("batched", 3, 8, 0.3), ("gqa", 2, 4, 0.8)])
def test_sampled_loop_reduced_workloads(wl, B, steps, T):
    """Several sequences with their own matrices (fp32 logits), and the
    large-vocabulary grouped-query workload (bf16 logits, int32 matrix)."""
    w = synth.WORKLOADS[wl].scaled(B=B, steps=steps, prefix=(300, 700))
    recs, diverged, compared = _check_sampled_loop(w, T)
    assert compared >= 0.75 * B * steps


def test_sampled_loop_at_vanishing_temperature_is_the_greedy_loop():
    """At T = 1e-7 (logits on a 2^-16 grid: distinct values differ by at least
    150 in units of T) tr_step_sampled commits exactly what tr_step commits,
    step for step, matrices included."""
    w = synth.WORKLOADS["batched"].scaled(B=4, steps=12, prefix=(200, 900))
    g, _, _ = run_gpu_loop(w, w.steps, keep_M_every=1)
    s, _, _ = run_gpu_loop(w, w.steps, keep_M_every=1, temperature=1e-7)
    for a, b in zip(g, s):
        for k in ("tok", "ids", "acc_len", "path", "committed", "root", "M"):
            assert np.array_equal(a[k], b[k]), k
