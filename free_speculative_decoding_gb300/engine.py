"""Device state of a batch of sequences decoding with Token Recycling.

`TRState` owns the tensors one decoding loop needs (the adjacency matrices,
the loop state, the KV cache of the verification layer, the per-step outputs
and the workspaces) and calls the libtr ABI on the current stream.  It does
no arithmetic itself.  A step is

    state.verify(Q, Kt, Vt)          # tree attention for the current tree
    ... the target produces logits (or hidden states) for state.tree_tok ...
    state.finish(logits=...)         # top-K, accept, update, KV commit, next tree

Every call is asynchronous and allocation-free after construction, so whole
loops can be captured in a CUDA graph.
"""
from __future__ import annotations

import torch

from . import (TR_INIT_INHERIT, TR_UPD_ALL, Tree, make_step_args, tr_get_status, tr_init_matrix, tr_retrieve,
               tr_step, tr_step_sampled, tr_step_workspace_bytes, tr_verify_attn, tr_verify_attn_workspace_bytes,
               workspace)


class TRState:
    def __init__(self, tree: Tree, B: int, V: int, m_dtype=torch.int64, Hq=0, Hkv=0, d=128, cap=0,
                 logits_dtype=torch.float32, D=0, device="cuda"):
        self.tree = tree
        self.B, self.V, self.K, self.N = B, V, tree.K, tree.N
        self.Dmax = tree.max_depth
        self.device = device
        self.logits_dtype = logits_dtype
        self.D = D
        dev = dict(device=device)
        self.M = torch.zeros(B, V, tree.K, dtype=m_dtype, **dev)
        self.root = torch.zeros(B, dtype=torch.int32, **dev)
        self.L = torch.zeros(B, dtype=torch.int32, **dev)
        self.tree_tok = torch.zeros(B, self.N, dtype=torch.int32, **dev)
        self.ids = torch.zeros(B * self.N, tree.K, dtype=torch.int32, **dev)
        self.vals = torch.zeros(B * self.N, tree.K, dtype=torch.float32, **dev)
        self.acc_len = torch.zeros(B, dtype=torch.int32, **dev)
        self.path = torch.zeros(B, self.Dmax + 1, dtype=torch.int32, **dev)
        self.committed = torch.zeros(B, self.Dmax + 1, dtype=torch.int32, **dev)
        self.attention = Hq > 0
        if self.attention:
            self.Hq, self.Hkv, self.d, self.cap = Hq, Hkv, d, cap
            self.Kc = torch.zeros(B, Hkv, cap, d, dtype=torch.bfloat16, **dev)
            self.Vc = torch.zeros_like(self.Kc)
            self.O = torch.zeros(B, self.N, Hq, d, dtype=torch.float32, **dev)
            self.ws_attn = workspace(tr_verify_attn_workspace_bytes(B, Hq, Hkv, d, cap, tree), device)
            self.scale = d ** -0.5
        self._args = make_step_args(tree, self.M, self.tree_tok, self.ids, self.vals, self.acc_len, self.path,
                                    self.committed, self.root, self.L,
                                    logits=torch.empty(1, V, dtype=logits_dtype, **dev) if D == 0 else None,
                                    H=torch.empty(1, max(D, 64), dtype=torch.bfloat16, **dev) if D else None,
                                    Wt=torch.empty(1, max(D, 64), dtype=torch.bfloat16, **dev) if D else None)
        self.ws_step = workspace(tr_step_workspace_bytes(self._args), device)

    def start(self, root, L, M_src=None, mode=TR_INIT_INHERIT, seed=0):
        """Set the roots and cache lengths, initialise M, retrieve the first tree.

        M_src [B, V, K] is copied in as it is; M_src [V, K] is inherited by
        every sequence (tr_init_matrix INHERIT); without M_src, ``mode`` is
        TR_INIT_ZERO or TR_INIT_RANDOM (at ``seed``), or None to keep M as it
        already is."""
        self.root.copy_(torch.as_tensor(root, dtype=torch.int32))
        self.L.copy_(torch.as_tensor(L, dtype=torch.int32))
        if M_src is not None and M_src.dim() == 3:
            self.M.copy_(M_src)
        elif mode is not None:
            tr_init_matrix(self.M, mode, M_src, seed)
        tr_retrieve(self.M, self.tree, self.root, self.tree_tok)

    def verify(self, Q, Kt, Vt):
        tr_verify_attn(Q, Kt, Vt, self.Kc, self.Vc, self.L, self.tree, self.O, self.scale, self.ws_attn)
        return self.O

    def finish(self, logits=None, H=None, Wt=None, Kt=None, Vt=None, mode=TR_UPD_ALL, temperature=None, U=None):
        """Everything after the target's forward pass: tr_step, or tr_step_sampled
        at ``temperature`` with the uniforms U [B, N, K+1]."""
        a = make_step_args(self.tree, self.M, self.tree_tok, self.ids, self.vals, self.acc_len, self.path,
                           self.committed, self.root, self.L, logits=logits, H=H, Wt=Wt,
                           Kt=Kt if self.attention else None, Vt=Vt if self.attention else None,
                           Kc=self.Kc if self.attention else None, Vc=self.Vc if self.attention else None,
                           mode=mode, ws=self.ws_step)
        if temperature is None:
            tr_step(a)
        else:
            tr_step_sampled(a, temperature, U)

    def status(self):
        return tr_get_status()
