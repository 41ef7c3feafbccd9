"""Static draft-tree plan (oracle side; test infrastructure only).

Token Recycling drafts along a *static* tree: every node has the same number
of children on every step, so the tree's shape can be prepared once
(hyper.ai summary, section "Method": the tree is static so it can be
preprocessed; it is unbalanced because nodes earlier in a layer get more
children).  Nodes are numbered level by level, which is the order of the
merged sequence (blog "token-recycling", 完整工作流程 step 3: the flattened
sequence [guest, speaker, speak, event, at, for, ing] starts with the root).

The spec is a list of child counts, one per node, in that BFS order.  Child r
of a node is the r-th candidate of the node's token (blog step 2:
M[speaker] = [at, for, is] gives guest -> speaker -> at and guest -> speaker ->
for), so a child count may not exceed K.
"""
from __future__ import annotations

import numpy as np


class TreePlan:
    """parent, rank, depth and ancestor sets of a BFS-numbered static tree."""

    def __init__(self, child_counts, K):
        counts = [int(c) for c in child_counts]
        if not counts:
            raise ValueError("a draft tree has at least the root")
        if any(c < 0 or c > K for c in counts):
            raise ValueError("child counts must lie in [0, K]")
        parent, rank, depth = [-1], [0], [0]
        for n, c in enumerate(counts):
            if n >= len(parent):
                raise ValueError("child counts leave a node unreachable from the root")
            for r in range(c):
                parent.append(n)
                rank.append(r)
                depth.append(depth[n] + 1)
        if len(parent) != len(counts):
            raise ValueError("child counts do not close the tree: %d nodes named, %d listed"
                             % (len(parent), len(counts)))
        self.K = K
        self.N = len(counts)
        self.child_counts = counts
        self.parent = parent
        self.rank = rank
        self.depth = depth
        self.max_depth = max(depth)
        # path[n]: node indices from the root down to n, both included
        self.path = []
        for n in range(self.N):
            p, m = [], n
            while m >= 0:
                p.append(m)
                m = parent[m]
            self.path.append(p[::-1])
        # children[n]: the child nodes of n in rank order
        self.children = [[] for _ in range(self.N)]
        for n in range(1, self.N):
            self.children[parent[n]].append(n)
        # mask[i, j]: tree node j is visible to node i (j is i or an ancestor)
        self.mask = np.zeros((self.N, self.N), dtype=bool)
        for i in range(self.N):
            self.mask[i, self.path[i]] = True

    def level_sizes(self):
        return [self.depth.count(L) for L in range(self.max_depth + 1)]
