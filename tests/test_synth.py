"""Sanity of the seeded synthetic inputs (no GPU)."""
import numpy as np
import torch

import oracle
import synth


def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(1)
    x = torch.randn(100000, generator=g) * 10
    x[:4] = torch.tensor([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8])   # ties to even
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.bf16_bits(x.numpy()), want)
    assert np.array_equal(synth.bf16_to_f32(want), x.to(torch.bfloat16).float().numpy())


def test_irwin_hall_moments_and_exactness():
    z = synth.irwin_hall12(synth.hkey(1, 2), np.arange(200000))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert z.min() >= -6 and z.max() <= 6
    # values are integers times 2^-16
    assert np.array_equal(z * 65536, np.rint(z * 65536))


def test_mix64_matches_the_oracles_independent_copy():
    # two independent restatements of splitmix64 must agree
    s = 123456789
    for i in range(50):
        assert int(synth.stream(s, i)) == oracle.mix64_stream(s, i)


def test_logits_structure():
    w = synth.WORKLOADS["tiny"]
    rows = synth.logits_rows(w.seed, 0, [3, 4], [10, 11], w.V)
    nxt = synth.markov_next(w.seed, 0, np.array([10, 11]), w.V)
    alt = synth.markov_alt(w.seed, 0, np.array([10, 11]), w.V)
    for r in range(2):
        base = rows[r].copy()
        mask = np.ones(w.V, bool)
        mask[nxt[r]] = False
        mask[alt[r]] = False
        assert base[mask].max() < 6.0 and base[mask].min() > -6.0
    # the boosted successor is the greedy choice in most rows
    toks = np.arange(200)
    many = synth.logits_rows(w.seed, 0, 7, toks, w.V)
    assert (np.argmax(many, axis=1) == synth.markov_next(w.seed, 0, toks, w.V)).mean() > 0.8
    # bf16 variant is the rounded fp32 variant
    b = synth.logits_rows(w.seed, 0, [3], [10], w.V, "bf16")
    assert np.array_equal(b[0], synth.bf16_bits(rows[0]))


def test_tree_depths_and_capacity():
    assert synth.WORKLOADS["tiny"].depth() == 6
    assert synth.WORKLOADS["gqa"].depth() == 8
    w = synth.WORKLOADS["batched"]
    L = w.prefix_lengths()
    assert L.min() >= 1024 and L.max() <= 4096 and len(set(L.tolist())) > 8
    assert w.capacity() == 4096 + 256 * 7


def test_lmhead_operands_are_exact_on_grid():
    D, V = 256, 512
    h = synth.bf16_to_f32(synth.lm_hidden_rows(5, 0, np.arange(4), np.arange(4), D))
    assert np.array_equal(h * 32, np.rint(h * 32))
    wt = synth.bf16_to_f32(synth.lm_weight_rows(5, V, D))
    assert np.array_equal(wt * 1024, np.rint(wt * 1024))
    assert np.abs(wt).max() * 1024 <= 256


def test_tree_shape_sweep_trees():
    """The sweep's trees share the 80-node budget: wide (depth 3) and deep
    (depth 11) against T80 (depth 6); per-level child counts never increase
    in BFS order, so the first of equal-token siblings has the largest subtree."""
    import collections
    import oracle
    want = {"T80": (6, [1, 8, 20, 20, 15, 10, 6]), "W80": (3, [1, 8, 32, 39]),
            "D80": (11, [1, 4] + [8] * 9 + [3])}
    for name, (depth, sizes) in want.items():
        counts = synth.TREES[name]
        plan = oracle.TreePlan(counts, 8)
        assert plan.N == 80 and plan.max_depth == depth
        per = collections.Counter(plan.depth)
        assert [per[d] for d in range(depth + 1)] == sizes
        for d in range(depth + 1):
            level = [counts[n] for n in range(plan.N) if plan.depth[n] == d]
            assert level == sorted(level, reverse=True)
        w = synth.WORKLOADS["batched"].scaled(tree=name)
        assert w.N == 80 and w.depth() == depth
