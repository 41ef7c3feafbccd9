"""Bounded device waits that run out (GB300 only).

Every wait of the tensor-core attention, the fused LM head and the streaming
top-K is bounded in time.  Here the limit is set to 1 ns, far below any copy or
product, so each launch gives up: it must set TR_DEV_TIMEOUT in the status
word, let the copies and products it has issued complete, free its tensor
memory and return -- a status the host reads, never a hang or a fault.  With
the default limit back and the workspace cleared, the same calls on the same
context must then give the oracle's results.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import ATTN_TOL, bf16_tensor, rows_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tr():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from free_speculative_decoding_gb300 import build as b
    b.build()
    import free_speculative_decoding_gb300 as m
    return m


def _attention_case(tr):
    counts = synth.TREE_T80
    tree, plan = tr.Tree(counts, 8), oracle.TreePlan(counts, 8)
    B, Hq, Hkv, d, lens = 2, 8, 4, 128, [700, 1100]   # 2 x 4 x 2 pairs of 13-20 tiles
    cap = 1200
    g = torch.Generator().manual_seed(41)
    q = torch.randn(B, plan.N, Hq, d, generator=g).to(torch.bfloat16)
    kt = torch.randn(B, plan.N, Hkv, d, generator=g).to(torch.bfloat16)
    vt = torch.randn(B, plan.N, Hkv, d, generator=g).to(torch.bfloat16)
    kc = torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16)
    dev = [x.cuda() for x in (q, kt, vt, kc, vc)]
    L = torch.tensor(lens, dtype=torch.int32, device="cuda")
    O = torch.zeros(B, plan.N, Hq, d, dtype=torch.float32, device="cuda")
    ws = tr.workspace(tr.tr_verify_attn_workspace_bytes(B, Hq, Hkv, d, cap, tree))

    def run():
        tr.tr_verify_attn(*dev, L, tree, O, d ** -0.5, ws)

    def check():
        Og = O.cpu().numpy()
        for b in range(B):
            ref = oracle.tree_attention(q[b].float().numpy(), kc[b].float().numpy(), vc[b].float().numpy(), lens[b],
                                        kt[b].float().numpy(), vt[b].float().numpy(), plan, d ** -0.5)
            assert rows_rel_err(Og[b], ref) <= ATTN_TOL
    return run, check, ws


def _lmhead_case(tr):
    w = synth.WORKLOADS["lmhead"]
    rows, D, V, K = 300, 512, 9001, 8          # 3 x 36 output tiles
    tok = np.arange(rows) * 37 % V
    H = synth.lm_hidden_rows(w.seed, 0, np.arange(rows), tok, D)
    Wt = synth.lm_weight_rows(w.seed, V, D)
    Hd, Wd = bf16_tensor(H), bf16_tensor(Wt)
    ids = torch.zeros(rows, K, dtype=torch.int32, device="cuda")
    vals = torch.zeros(rows, K, dtype=torch.float32, device="cuda")
    ws = tr.workspace(tr.tr_lmhead_topk_workspace_bytes(rows, D, V, K))

    def run():
        tr.tr_lmhead_topk(Hd, Wd, K, ids, vals, ws)

    def check():
        # the grid-valued operands make every fp32 sum exact: the result is exact
        ids_ref, _ = oracle.topk_rows(oracle.lmhead_logits(synth.bf16_to_f32(H), synth.bf16_to_f32(Wt)), K)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
    return run, check, ws


def _topk_case(tr):
    rows, V, K = 400, 32000, 8                 # 400 rows x 16 steps over 50 warps
    g = torch.Generator().manual_seed(43)
    x = torch.randn(rows, V, generator=g)
    xd = x.cuda()
    ids = torch.zeros(rows, K, dtype=torch.int32, device="cuda")
    vals = torch.zeros(rows, K, dtype=torch.float32, device="cuda")
    ws = tr.workspace(tr.tr_topk_workspace_bytes(rows, V, K))

    def run():
        tr.tr_topk(xd, K, ids, vals, ws)

    def check():
        ids_ref, _ = oracle.topk_rows(x.numpy(), K)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
    return run, check, ws


@pytest.mark.parametrize("case", [_attention_case, _lmhead_case, _topk_case],
                         ids=["tree_attention", "lmhead_topk", "topk"])
def test_wait_limit_runs_out_then_recovers(tr, case):
    run, check, ws = case(tr)
    assert tr.tr_get_status() == 0
    prev = tr.tr_set_wait_limit_ns(1)
    try:
        for _ in range(2):   # two launches in a row on the same context
            run()
            status = tr.tr_get_status()
            assert status & tr.TR_DEV_TIMEOUT, "no wait gave up (status %#x)" % status
    finally:
        assert tr.tr_set_wait_limit_ns(prev) == 1
    assert prev == 2_000_000_000
    # the context is usable: with the limit back and the workspace cleared, the call is exact again
    tr.tr_workspace_clear(ws)
    run()
    assert tr.tr_get_status() == 0
    check()
    run()   # and it leaves its workspace ready for the next call
    assert tr.tr_get_status() == 0
    check()

