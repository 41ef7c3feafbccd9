"""Pins of the CPU oracle against what the pages and mathematics fix (no GPU).

Each test checks the oracle against something other than itself: the blog's
worked example, brute force or an independent algorithm on tiny inputs, a
closed form, an invariant, or a special case that reduces to a library
routine.  A plausible slip anywhere in the oracle (wrong parent or rank, a
dropped mask term, a transposed operand, an off-by-one position, a wrong tie
rule, a wrong writer order) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import TreePlan


# ----------------------------------------------------------------------------
# the blog's worked example (K = 3)
# ----------------------------------------------------------------------------

@pytest.fixture(scope="module")
def t1(golden_dir):
    with open(os.path.join(golden_dir, "t1_worked_example.json")) as f:
        g = json.load(f)
    ix = {w: i for i, w in enumerate(g["vocab"])}
    g["ix"] = ix
    g["V"] = len(g["vocab"])
    return g


def _t1_matrix(g):
    M = np.zeros((g["V"], g["K"]), dtype=np.int64)
    for w, row in g["old_rows"].items():
        M[g["ix"][w]] = [g["ix"][x] for x in row]
    return M


def _t1_logits(g, tok):
    """Logits whose top-3 are the page's lists (descending scores 3, 2, 1)."""
    lists = dict(g["top_lists"], **g["top_lists_unstated"])
    rows = np.zeros((len(tok), g["V"]), dtype=np.float32)
    for n, t in enumerate(tok):
        for r, w in enumerate(lists[g["vocab"][t]]):
            rows[n, g["ix"][w]] = 3.0 - r
    return rows


def test_t1_retrieve_tree_tokens(t1):
    plan = TreePlan(t1["child_counts"], t1["K"])
    tok = oracle.retrieve(_t1_matrix(t1), t1["ix"][t1["root"]], plan)
    assert [t1["vocab"][t] for t in tok] == t1["tree_tokens"]


def test_t1_mask_sees_only_own_path(t1):
    plan = TreePlan(t1["child_counts"], t1["K"])
    words = t1["tree_tokens"]
    for w, seen in t1["visible"].items():
        i = words.index(w)
        assert sorted(words[j] for j in np.flatnonzero(plan.mask[i])) == sorted(seen)


def test_t1_accept_update(t1):
    plan = TreePlan(t1["child_counts"], t1["K"])
    M = _t1_matrix(t1)
    tok = oracle.retrieve(M, t1["ix"][t1["root"]], plan)
    ids, _ = oracle.topk_rows(_t1_logits(t1, tok), t1["K"])
    acc_len, path, committed, bonus = oracle.accept(plan, tok, ids[:, 0])
    v = t1["vocab"]
    assert acc_len == t1["acc_len"]
    assert [v[tok[n]] for n in path[1:]] == t1["accepted"]
    assert v[bonus] == t1["bonus"]
    assert [v[c] for c in committed] == t1["committed"]
    oracle.update(M, tok, ids, plan)
    for w, row in t1["new_rows"].items():
        assert [v[x] for x in M[t1["ix"][w]]] == row, w
    for w, row in t1["top_lists_unstated"].items():
        assert [v[x] for x in M[t1["ix"][w]]] == row, w
    # the rejected-branch node 'speak' wrote its row
    assert [v[x] for x in M[t1["ix"]["speak"]]] != t1["old_rows"]["speak"]


def test_t1_accepted_only_ablation_skips_rejected_branch(t1):
    plan = TreePlan(t1["child_counts"], t1["K"])
    M = _t1_matrix(t1)
    tok = oracle.retrieve(M, t1["ix"][t1["root"]], plan)
    ids, _ = oracle.topk_rows(_t1_logits(t1, tok), t1["K"])
    _, path, _, _ = oracle.accept(plan, tok, ids[:, 0])
    oracle.update(M, tok, ids, plan, oracle.UPD_ACCEPTED, path)
    v = t1["vocab"]
    assert [v[x] for x in M[t1["ix"]["speak"]]] == t1["old_rows"]["speak"]
    assert [v[x] for x in M[t1["ix"]["speaker"]]] == t1["new_rows"]["speaker"]


# ----------------------------------------------------------------------------
# tree plans: closed-form sizes of the two static trees
# ----------------------------------------------------------------------------

def test_tree_shapes():
    p80 = TreePlan(synth.TREE_T80, 8)
    assert p80.N == 80 and p80.max_depth == 6
    assert p80.level_sizes() == [1, 8, 20, 20, 15, 10, 6]
    top = []
    n = 0
    while p80.child_counts[n]:
        top.append(p80.child_counts[n])
        n = n + 1 if n == 0 else next(m for m in range(p80.N) if p80.parent[m] == n)
    assert top == [8, 4, 2, 1, 1, 1]
    p128 = TreePlan(synth.TREE_T128, 8)
    assert p128.N == 128 and p128.max_depth == 8
    assert p128.level_sizes() == [1, 8, 24, 30, 24, 16, 11, 8, 6]
    for p in (p80, p128):
        assert all(p.depth[n] == p.depth[p.parent[n]] + 1 for n in range(1, p.N))
        assert all(p.parent[n] < n for n in range(1, p.N))


def test_tree_rejects_bad_specs():
    with pytest.raises(ValueError):
        TreePlan([4, 0, 0], 8)         # names 5 nodes, lists 3
    with pytest.raises(ValueError):
        TreePlan([1, 0, 1], 8)         # node 2 unreachable
    with pytest.raises(ValueError):
        TreePlan([9] + [0] * 9, 8)     # child count above K


# ----------------------------------------------------------------------------
# acceptance: an independent recursive search on tiny random trees
# ----------------------------------------------------------------------------

def _random_tree(rng, n_max=12, K=3):
    counts = [int(rng.integers(1, K + 1))]
    total = 1 + counts[0]
    n = 1
    while n < total:
        c = int(rng.integers(0, K + 1)) if total < n_max else 0
        c = min(c, n_max - total)
        counts.append(c)
        total += c
        n += 1
    return counts


def _dfs_longest(plan, tok, top1):
    """Longest matching root path by depth-first search in child-rank order."""
    children = [[] for _ in range(plan.N)]
    for n in range(1, plan.N):
        children[plan.parent[n]].append(n)
    best = [0]

    def visit(n):
        if plan.depth[n] > plan.depth[best[0]]:
            best[0] = n
        for c in children[n]:
            if tok[c] == top1[n]:
                visit(c)

    visit(0)
    return best[0]


def test_t3_accept_matches_recursive_search():
    rng = np.random.default_rng(3)
    for _ in range(400):
        plan = TreePlan(_random_tree(rng), 3)
        V = int(rng.integers(2, 5))          # tiny vocabulary: many matches and ties
        tok = rng.integers(0, V, plan.N)
        top1 = rng.integers(0, V, plan.N)
        acc_len, path, committed, bonus = oracle.accept(plan, tok, top1)
        n_star = _dfs_longest(plan, tok, top1)
        assert path[-1] == n_star
        assert acc_len == plan.depth[n_star] == len(path) - 1
        assert bonus == top1[n_star]
        assert committed == [int(tok[m]) for m in path[1:]] + [int(top1[n_star])]


def test_accept_hand_cases():
    # root with children a(0), b(1); a has child c; b has child d, e
    plan = TreePlan([2, 1, 2, 0, 0, 0], 2)   # nodes: 0 root, 1 a, 2 b, 3 c(a), 4 d(b), 5 e(b)
    tok = np.array([9, 5, 5, 7, 6, 7])
    # both a and b carry token 5 and match; under a, c=7 matches top1[a]=7;
    # under b, e=7 matches top1[b]=7: equal depth, smallest BFS index (c=3) wins
    top1 = np.array([5, 7, 7, 1, 2, 3])
    acc_len, path, committed, bonus = oracle.accept(plan, tok, top1)
    assert (acc_len, path, committed, bonus) == (2, [0, 1, 3], [5, 7, 1], 1)
    # nothing matches: only the bonus is emitted
    top1 = np.array([4, 0, 0, 0, 0, 0])
    assert oracle.accept(plan, tok, top1) == (0, [0], [4], 4)


# ----------------------------------------------------------------------------
# update: last writer in BFS order
# ----------------------------------------------------------------------------

def test_t5_duplicate_tokens_last_writer_wins():
    plan = TreePlan([3, 1, 0, 0, 0], 4)
    M = np.zeros((10, 4), dtype=np.int64)
    tok = np.array([1, 2, 3, 2, 3])           # token 2 at nodes 1 and 3, token 3 at 2 and 4
    ids = np.arange(20).reshape(5, 4)
    oracle.update(M, tok, ids, plan)
    assert M[1].tolist() == ids[0].tolist()
    assert M[2].tolist() == ids[3].tolist()
    assert M[3].tolist() == ids[4].tolist()
    assert not M[[0, 4, 5]].any()


# ----------------------------------------------------------------------------
# top-K
# ----------------------------------------------------------------------------

def _select_topk(row, K):
    """Selection by repeated scans: the best remaining value, lowest ID among equals."""
    taken, out = set(), []
    for _ in range(K):
        best = None
        for i, x in enumerate(row):
            if i in taken:
                continue
            if best is None or x > row[best]:
                best = i
        taken.add(best)
        out.append(best)
    return out


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(5)
    for _ in range(300):
        V = int(rng.integers(1, 40))
        K = int(rng.integers(1, V + 1))
        row = rng.integers(-3, 4, V).astype(np.float32)    # heavy ties
        row[row == 0] = rng.choice([0.0, -0.0], size=int((row == 0).sum()))
        assert oracle.topk(row, K).tolist() == _select_topk(row.tolist(), K)


def test_topk_signed_zero_tie_goes_to_lower_id():
    row = np.array([-0.0, 0.0, -1.0, -0.0], dtype=np.float32)
    assert oracle.topk(row, 3).tolist() == [0, 1, 3]
    row = np.array([0.0, -0.0], dtype=np.float32)
    assert oracle.topk(row, 2).tolist() == [0, 1]


def test_topk_matches_torch_on_distinct_values():
    g = torch.Generator().manual_seed(0)
    rows = torch.randn(20, 5000, generator=g, dtype=torch.float64)
    ids, vals = oracle.topk_rows(rows.numpy(), 8)
    tv, ti = torch.topk(rows, 8, dim=1, sorted=True)
    assert np.array_equal(ids, ti.numpy())
    assert np.array_equal(vals, tv.numpy())


# ----------------------------------------------------------------------------
# attention special cases
# ----------------------------------------------------------------------------

def _rand(rng, *shape):
    return rng.standard_normal(shape)


def test_attention_single_key_returns_its_value():
    rng = np.random.default_rng(1)
    plan = TreePlan([0], 8)
    q, kt, vt = _rand(rng, 1, 4, 16), _rand(rng, 1, 2, 16), _rand(rng, 1, 2, 16)
    kc = np.zeros((2, 5, 16))
    o = oracle.tree_attention(q, kc, kc, 0, kt, vt, plan, 0.25)
    assert np.allclose(o[0, :2], vt[0, 0]) and np.allclose(o[0, 2:], vt[0, 1])


def test_attention_zero_query_averages_visible_values():
    rng = np.random.default_rng(2)
    plan = TreePlan(synth.TREE_T80, 8)
    N, Hq, Hkv, d, L = plan.N, 4, 2, 8, 13
    q = np.zeros((N, Hq, d))
    kc, vc = _rand(rng, Hkv, 20, d), _rand(rng, Hkv, 20, d)
    kt, vt = _rand(rng, N, Hkv, d), _rand(rng, N, Hkv, d)
    o = oracle.tree_attention(q, kc, vc, L, kt, vt, plan, 0.3)
    for i in range(N):
        anc = plan.path[i]
        for h in range(Hq):
            g = h // 2
            want = (vc[g, :L].sum(0) + vt[anc, g].sum(0)) / (L + len(anc))
            assert np.allclose(o[i, h], want)


def _sdpa(q, k, v, mask, scale):
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=torch.from_numpy(mask)[None], scale=scale)[0].numpy()


def test_attention_chain_tree_is_causal_attention():
    rng = np.random.default_rng(4)
    depth, Hq, Hkv, d, L = 7, 8, 2, 32, 40
    plan = TreePlan(synth.chain_tree(depth), 8)
    N = plan.N
    q = _rand(rng, N, Hq, d)
    kc, vc = _rand(rng, Hkv, 64, d), _rand(rng, Hkv, 64, d)
    kt, vt = _rand(rng, N, Hkv, d), _rand(rng, N, Hkv, d)
    scale = d ** -0.5
    o = oracle.tree_attention(q, kc, vc, L, kt, vt, plan, scale)
    causal = np.concatenate([np.ones((N, L), bool), np.tril(np.ones((N, N), bool))], axis=1)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        k = np.concatenate([kc[g, :L], kt[:, g]])
        v = np.concatenate([vc[g, :L], vt[:, g]])
        assert np.allclose(o[:, h], _sdpa(q[:, h], k, v, causal, scale), atol=1e-12)


def test_attention_each_node_equals_attention_over_its_own_path():
    rng = np.random.default_rng(6)
    plan = TreePlan(synth.TREE_T80, 8)
    N, Hq, Hkv, d, L = plan.N, 4, 4, 16, 9
    q = _rand(rng, N, Hq, d)
    kc, vc = _rand(rng, Hkv, 12, d), _rand(rng, Hkv, 12, d)
    kt, vt = _rand(rng, N, Hkv, d), _rand(rng, N, Hkv, d)
    o = oracle.tree_attention(q, kc, vc, L, kt, vt, plan, 0.2)
    for i in rng.choice(N, 12, replace=False):
        anc = plan.path[i]
        for h in range(Hq):
            k = np.concatenate([kc[h, :L], kt[anc, h]])
            v = np.concatenate([vc[h, :L], vt[anc, h]])
            want = _sdpa(q[i:i + 1, h], k, v, np.ones((1, len(k)), bool), 0.2)
            assert np.allclose(o[i, h], want[0], atol=1e-12)


# ----------------------------------------------------------------------------
# storage closed form (blog: 32,000 x 8 x 8 bytes = 2,048,000 bytes ~ 1.95 MiB)
# ----------------------------------------------------------------------------

def test_t4_storage_closed_form():
    M = oracle.init_matrix(oracle.INIT_ZERO, 32000, 8, dtype=np.int64)
    assert M.nbytes == 32000 * 8 * 8 == 2_048_000
    assert M.nbytes / 2 ** 20 == 1.953125
    assert M.nbytes / 2 ** 20 < 2.0 < M.nbytes / 1e6 + 0.1   # "< 2 MB" holds in MiB only
    M32 = oracle.init_matrix(oracle.INIT_ZERO, 128256, 8, dtype=np.int32)
    assert M32.nbytes == 4_104_192


def test_init_modes():
    src = np.arange(40).reshape(10, 4) % 10
    assert np.array_equal(oracle.init_matrix(oracle.INIT_INHERIT, 10, 4, src=src), src)
    assert not oracle.init_matrix(oracle.INIT_ZERO, 10, 4).any()
    R = oracle.init_matrix(oracle.INIT_RANDOM, 500, 8, seed=7)
    assert R.min() >= 0 and R.max() < 500
    counts = np.bincount(R.ravel() // 50, minlength=10)
    assert counts.min() > 300            # 4000 draws over 10 bins of 400 expected
    R2 = oracle.init_matrix(oracle.INIT_RANDOM, 500, 8, seed=7, seq=1)
    assert (R2 != R).mean() > 0.9
    assert np.array_equal(R, oracle.init_matrix(oracle.INIT_RANDOM, 500, 8, seed=7))


# published reference outputs of splitmix64 (Steele, Lea, Flood 2014, as in
# Vigna's splitmix64.c): the first outputs of the streams at states 0 and 1234567
SPLITMIX64_STATE0 = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
SPLITMIX64_STATE1234567 = [6457827717110365317, 3203168211198807973, 9817491932198370423,
                           4593380528125082431, 16408922859458223821]


def test_splitmix64_published_outputs():
    assert [oracle.mix64_stream(0, i) for i in range(3)] == SPLITMIX64_STATE0
    assert [oracle.mix64_stream(1234567, i) for i in range(5)] == SPLITMIX64_STATE1234567
    # the input module's restatement of the same generator agrees
    assert [int(x) for x in synth.stream(1234567, np.arange(5))] == SPLITMIX64_STATE1234567


def test_init_random_index_formula():
    """RANDOM entry (seq, i, j) is stream output (seq*V + i)*K + j, modulo V.

    Pinned on the published outputs (so a transposed index, a dropped seq
    term or an off-by-one in the stream index fails), then on a larger
    matrix against the input module's independent restatement."""
    o = SPLITMIX64_STATE0
    R = oracle.init_matrix(oracle.INIT_RANDOM, 7, 2, seed=0)
    assert R[0, 0] == o[0] % 7 and R[0, 1] == o[1] % 7 and R[1, 0] == o[2] % 7
    p = SPLITMIX64_STATE1234567
    R = oracle.init_matrix(oracle.INIT_RANDOM, 5, 1, seed=1234567)
    assert R[:, 0].tolist() == [x % 5 for x in p]
    R = oracle.init_matrix(oracle.INIT_RANDOM, 3, 1, seed=1234567, seq=1)
    assert R[0, 0] == p[3] % 3 and R[1, 0] == p[4] % 3
    V, K, seed = 37, 5, 99
    for seq in (0, 2):
        R = oracle.init_matrix(oracle.INIT_RANDOM, V, K, seed=seed, seq=seq, dtype=np.int32)
        i, j = np.meshgrid(np.arange(V), np.arange(K), indexing="ij")
        ref = synth.stream(seed, (seq * V + i) * K + j) % np.uint64(V)
        assert np.array_equal(R, ref.astype(np.int64))


def test_splitmix64_is_a_bijection_on_a_sample():
    # the output function of splitmix64 is invertible: distinct states give distinct outputs
    outs = {oracle.mix64_stream(s, 0) for s in range(20000)}
    assert len(outs) == 20000


# ----------------------------------------------------------------------------
# KV commit and the LM head
# ----------------------------------------------------------------------------

def test_kv_commit_appends_path_in_order():
    kc = np.zeros((2, 10, 3))
    vc = np.zeros((2, 10, 3))
    kt = np.arange(6 * 2 * 3, dtype=float).reshape(6, 2, 3)
    vt = -kt
    L = oracle.kv_commit(kc, vc, kt, vt, 4, [0, 2, 5])
    assert L == 7
    for i, n in enumerate([0, 2, 5]):
        assert np.array_equal(kc[:, 4 + i], kt[n]) and np.array_equal(vc[:, 4 + i], vt[n])
    assert not kc[:, :4].any() and not kc[:, 7:].any()


def test_lmhead_one_hot_rows_select_weight_rows():
    rng = np.random.default_rng(8)
    Wt = rng.standard_normal((50, 12))
    H = np.zeros((3, 12))
    H[0, 4] = 1.0
    H[1, 0] = 2.0
    H[2, 4] = 1.0
    H[2, 11] = -1.0
    lg = oracle.lmhead_logits(H, Wt)
    assert np.array_equal(lg[0], Wt[:, 4])
    assert np.array_equal(lg[1], 2 * Wt[:, 0])
    assert np.allclose(lg[2], Wt[:, 4] - Wt[:, 11])


# ----------------------------------------------------------------------------
# invariants of the whole loop
# ----------------------------------------------------------------------------

def _synth_target(seed, V, dtype="f32"):
    def target(b, pos, tok):
        return synth.logits_f32(seed, b, pos, tok, V, dtype)
    return target


def test_t2_lossless_against_greedy_decoding():
    V, K, seed = 64, 8, 9
    plan = TreePlan(synth.TREE_T80, K)
    target = _synth_target(seed, V)
    for b in range(2):
        M = synth.warm_matrix(seed, b, V, K)
        st = oracle.TRState(M=M, root=5 + b, L=100)
        oracle.tr_loop(plan, [st], target, 12, K, seqs=[b])
        emitted = st.emitted
        assert len(emitted) >= 12
        ref = oracle.greedy_decode(lambda pos, x: int(np.argmax(target(b, pos, [x])[0])), 5 + b, 100,
                                   len(emitted))
        assert emitted == ref


def test_t2_lossless_full_vocab_and_acceptance_is_nontrivial():
    w = synth.WORKLOADS["tiny"]
    plan = TreePlan(w.child_counts, w.K)
    target = _synth_target(w.seed, w.V)
    root = int(synth.initial_roots(w)[0])
    st = oracle.TRState(M=synth.warm_matrix(w.seed, 0, w.V, w.K), root=root, L=512)
    acc = []
    oracle.tr_loop(plan, [st], target, 6, w.K, on_step=lambda s, i, r: acc.append(r["acc_len"]))
    ref = oracle.greedy_decode(lambda pos, x: int(np.argmax(target(0, pos, [x])[0])), root, 512,
                               len(st.emitted))
    assert st.emitted == ref
    assert max(acc) >= 2


def test_t6_expected_tokens_per_pass_chain():
    # lesson: an i.i.d. linear draft of gamma tokens accepted with rate alpha
    # emits (1 - alpha^(gamma+1)) / (1 - alpha) tokens per pass on average
    gamma, alpha, trials = 4, 0.8, 20000
    plan = TreePlan(synth.chain_tree(gamma), 1)
    rng = np.random.default_rng(11)
    total = 0
    for _ in range(trials):
        tok = rng.integers(0, 1000, plan.N)
        hit = rng.random(plan.N) < alpha
        top1 = np.where(np.r_[hit[1:], False], np.r_[tok[1:], 0], 5000)
        acc_len, _, committed, _ = oracle.accept(plan, tok, top1)
        assert len(committed) == acc_len + 1
        total += len(committed)
    want = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(want - 3.3616) < 1e-12
    sd = math.sqrt(2.0 / trials) * 1.5
    assert abs(total / trials - want) < 4 * sd


# ----------------------------------------------------------------------------
# acceptance under sampling (lesson, the acceptance rule; hyper.ai summary,
# "Experiment": robustness under sampling)
# ----------------------------------------------------------------------------

def test_softmax_stats_against_logsumexp():
    from scipy.special import logsumexp
    rng = np.random.default_rng(21)
    for T in (0.3, 1.0, 2.5):
        row = rng.normal(size=5000) * 3
        m, Z = oracle.softmax_stats(row, T)
        assert m == row.max()
        assert abs(m / T + math.log(Z) - logsumexp(row / T)) < 1e-9
        p = oracle.target_probs(row, T)
        assert abs(p.sum() - 1) < 1e-12 and abs(p[np.argmax(row)] - 1 / Z) < 1e-15
    assert oracle.softmax_stats(np.full(77, 1.25), 0.7) == (1.25, 77.0)   # equal logits: Z = V


def test_sampled_acceptance_hand_case():
    """Worked by hand from the rule: root distribution [.1, .2, .3, .4] with
    children holding tokens 3 then 1; U = .5 rejects 3 (.5 >= .4), the residual
    becomes [1/6, 1/3, 1/2, 0], U = .3 accepts 1 (.3 < 1/3); at that leaf the
    draw at U = .05 over [.7, .1, .1, .1] gives token 0, at U = .75 token 1."""
    plan = TreePlan([2, 0, 0], 4)
    tok = np.array([2, 3, 1])
    logits = np.log(np.array([[.1, .2, .3, .4], [.25, .25, .25, .25], [.7, .1, .1, .1]]))
    U = np.zeros((3, 5))
    U[0, 0], U[0, 1], U[2, 4] = 0.5, 0.3, 0.05
    acc, path, com, bonus, _, _ = oracle.accept_sampled(plan, tok, logits, 1.0, U)
    assert (acc, path, com, bonus) == (1, [0, 2], [1, 0], 0)
    U[2, 4] = 0.75
    assert oracle.accept_sampled(plan, tok, logits, 1.0, U)[2] == [1, 1]
    # both children rejected (.5 >= .4, then .4 >= 1/3): the residual without
    # tokens 3 and 1 is [1/4, 0, 3/4, 0]; the draw at U = .6 gives token 2,
    # whose interval [.25, 1) lies .35 from U at its nearer end
    U[0, 1], U[0, 4] = 0.4, 0.6
    acc, path, com, bonus, margins, cdf = oracle.accept_sampled(plan, tok, logits, 1.0, U)
    assert (acc, path, com, bonus) == (0, [0], [2], 2)
    assert abs(margins[0] - (0.4 - 1 / 3)) < 1e-12 and abs(margins[1] - 0.35) < 1e-12
    assert np.allclose(cdf, [0.25, 0.25, 1, 1])
    assert oracle.draw_is_valid(cdf, 0.6, 2, 0.0) and not oracle.draw_is_valid(cdf, 0.6, 1, 0.05)
    assert oracle.draw_is_valid(cdf, 0.26, 0, 0.05) and not oracle.draw_is_valid(cdf, 0.6, 3, 1.0)


def _distinct_sibling_tokens(plan, V, rng):
    tok = np.zeros(plan.N, np.int64)
    tok[0] = rng.integers(0, V)
    for n in range(plan.N):
        kids = plan.children[n]
        tok[kids] = rng.choice(V, size=len(kids), replace=False)
    return tok


def test_sampled_acceptance_greedy_limit():
    """T -> 0 turns sampling into greedy Token Recycling: with distinct sibling
    tokens (so at most one child can match) the sampled walk equals the
    greedy acceptance on random tiny trees, whatever the uniforms."""
    rng = np.random.default_rng(23)
    for _ in range(300):
        K = int(rng.integers(1, 5))
        counts = [int(rng.integers(1, K + 1))]
        while len(counts) < 1 + sum(counts) and len(counts) < 30:
            counts.append(int(rng.integers(0, K + 1)) if sum(counts) < 25 else 0)
        counts += [0] * (1 + sum(counts) - len(counts))
        plan = TreePlan(counts, K)
        V = 12
        tok = _distinct_sibling_tokens(plan, V, rng)
        logits = rng.permuted(np.tile(np.arange(V, dtype=np.float64), (plan.N, 1)), axis=1)  # distinct values
        for n in range(1, plan.N):               # make many children match their parent's argmax
            if rng.random() < 0.6:
                row = logits[plan.parent[n]]
                j = int(np.argmax(row))
                row[[j, tok[n]]] = row[[tok[n], j]]
        U = rng.random((plan.N, K + 1))
        got = oracle.accept_sampled(plan, tok, logits, 1e-3, U)[:4]
        assert got == oracle.accept(plan, tok, np.argmax(logits, axis=1))


def test_sampled_first_tokens_follow_the_target():
    """Losslessness in distribution (lesson): the first committed token is
    distributed as the root's p = softmax(x / T), and after a first token that
    a child holds, the second is distributed as that child's p -- whatever the
    drafted children were.  Chi-square over 30000 draws with uniform U."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(29)
    V, T, n = 6, 0.7, 30000
    plan = TreePlan([3, 0, 0, 0], 6)
    tok = np.array([0, 2, 0, 5])
    logits = rng.normal(size=(4, V)) * 1.5
    first = np.zeros(V, np.int64)
    second = np.zeros(V, np.int64)
    for _ in range(n):
        com = oracle.accept_sampled(plan, tok, logits, T, rng.random((4, 7)))[2]
        first[com[0]] += 1
        if com[0] == 5:
            second[com[1]] += 1
    p0 = oracle.target_probs(logits[0], T)
    assert chisquare(first, p0 * n).pvalue > 1e-3
    p3 = oracle.target_probs(logits[3], T)
    assert chisquare(second, p3 * second.sum()).pvalue > 1e-3
    # the test has power: the same counts against a permuted distribution fail it
    assert chisquare(first, p0[[1, 2, 3, 4, 0, 5]] * n).pvalue < 1e-6


def test_sampled_expected_tokens_per_pass_chain():
    """Lesson: a linear draft of gamma tokens, each accepted with probability
    alpha, emits (1 - alpha^(gamma+1)) / (1 - alpha) tokens per pass.  Under
    the sampling rule a deterministic draft token is accepted with its target
    probability, so a chain whose every draft token has p = 0.8 must emit
    3.3616 tokens per pass on average."""
    gamma, alpha, V, trials = 4, 0.8, 50, 40000
    plan = TreePlan(synth.chain_tree(gamma), 1)
    tok = np.arange(plan.N) + 3
    logits = np.full((plan.N, V), math.log((1 - alpha) / (V - 1)))
    for n in range(gamma):
        logits[n, tok[n + 1]] = math.log(alpha)
    rng = np.random.default_rng(31)
    total = sum(len(oracle.accept_sampled(plan, tok, logits, 1.0, rng.random((plan.N, 2)))[2])
                for _ in range(trials))
    want = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(total / trials - want) < 0.03      # about 5 standard errors


def test_sampling_loop_at_vanishing_temperature_is_greedy_decoding():
    """The whole loop under sampling at T = 1e-7 (logits on a 2^-16 grid, so
    any two distinct values differ by over 150 / T-units) commits exactly the
    plain greedy stream, like greedy Token Recycling."""
    V, K, seed = 64, 8, 9
    plan = TreePlan(synth.TREE_T80, K)
    target = _synth_target(seed, V)
    for b in range(2):
        st = oracle.TRState(M=synth.warm_matrix(seed, b, V, K), root=5 + b, L=100)
        oracle.tr_loop(plan, [st], target, 10, K, seqs=[b], temperature=1e-7,
                       uniforms=lambda s, bb: synth.uniforms(seed, s, bb, plan.N, K + 1))
        ref = oracle.greedy_decode(lambda pos, x: int(np.argmax(target(b, pos, [x])[0])), 5 + b, 100,
                                   len(st.emitted))
        assert st.emitted == ref and len(st.emitted) >= 10
