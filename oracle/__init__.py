"""CPU oracle for the Token Recycling per-step hot path.

TEST INFRASTRUCTURE ONLY.  The oracle is a plain, slow, obviously correct
restatement of what one Token Recycling decoding step computes.  Only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import it.  The CUDA library never imports, links or calls anything
here, and nothing here imports the CUDA library: the two share no code.

Sources, cited by page title and section:

* "Turning Trash into Treasure: Accelerating Inference of Large Language
  Models with Token Recycling" (ACL 2025), hyper.ai paper summary, English
  page, section "Method" -- the adjacency matrix, the static unbalanced
  tree, the BFS-like retrieval, tree-attention verification and the update;
  section "Experiment" -- the init-mode and update-mode ablations.
* The same summary, Chinese page, section "方法" (Method) -- the only copy of
  the update equation  M[x~_i] = argtopk(p~_{i+1})  (the English copy lost it).
* blog-shf.pages.dev "token-recycling" -- section "核心数据结构：邻接矩阵"
  (the K=3 example matrix), section "完整工作流程" steps 1-4 (retrieval,
  tree building, the flattened merged sequence and its mask, longest-path
  acceptance plus the corrected token), section "为什么叫 Token Recycling"
  (the new rows, rejected-branch nodes included), sections "热启动" (hot
  start) and "为什么一个很小的矩阵就够用" (the storage closed form).
* anylearn.cc "Speculative decoding" lesson -- greedy losslessness, the bonus
  token, tree attention where each node sees only its ancestors, and the
  expected tokens per pass of an i.i.d. linear draft.

Where the pages are silent or ambiguous, the reading taken is stated next to
the function it affects.

Every function here is pinned by a ``-m "not gpu"`` test against something
other than itself (a worked example, brute force, a closed form or a special
case that reduces to a library routine); none is "parity unpinned".
"""
from .tree import TreePlan
from .tr import (
    INIT_ZERO, INIT_RANDOM, INIT_INHERIT, UPD_ALL, UPD_ACCEPTED,
    init_matrix, retrieve, tree_attention, topk, topk_rows, accept, update,
    kv_commit, lmhead_logits, mix64_stream, softmax_stats, target_probs, accept_sampled, draw_is_valid,
)
from .loop import TRState, tr_loop, greedy_decode

__all__ = [
    "TreePlan", "INIT_ZERO", "INIT_RANDOM", "INIT_INHERIT", "UPD_ALL", "UPD_ACCEPTED",
    "init_matrix", "retrieve", "tree_attention", "topk", "topk_rows", "accept", "update",
    "kv_commit", "lmhead_logits", "mix64_stream", "softmax_stats", "target_probs", "accept_sampled",
    "draw_is_valid", "TRState", "tr_loop", "greedy_decode",
]
