"""Device-side synthetic target for GPU runs (tests, benchmark, smoke).

Thin wrappers over libtr's trsyn_* generators, which implement the same
definitions as the numpy functions of ``synth`` (a GPU test compares them bit
for bit).  Nothing here is Token Recycling arithmetic.
"""
from __future__ import annotations

import torch

import free_speculative_decoding_gb300 as tr
import synth


class DeviceTarget:
    """Produces a step's target outputs for the state's current tree on the GPU."""

    def __init__(self, w: synth.Workload, tree, device="cuda"):
        self.w = w
        self.tree = tree
        self.device = device
        B, N = w.B, tree.N
        if w.logits == "lmhead":
            self.Wt = torch.empty(w.V, w.D, dtype=torch.bfloat16, device=device)
            tr.trsyn_lm_weight(w.seed, self.Wt)
            self.H = torch.empty(B * N, w.D, dtype=torch.bfloat16, device=device)
        else:
            dt = torch.bfloat16 if w.logits == "bf16" else torch.float32
            self.logits = torch.empty(B * N, w.V, dtype=dt, device=device)

    def logits_for(self, state, out=None):
        out = self.logits if out is None else out
        tr.trsyn_logits(self.w.seed, self.tree, state.tree_tok, state.L, out, V=self.w.V)
        return out

    def hidden_for(self, state, out=None):
        out = self.H if out is None else out
        tr.trsyn_lm_hidden(self.w.seed, self.tree, state.tree_tok, state.L, out)
        return out


def step_qkv(w: synth.Workload, step, N, device="cuda", out=None):
    """Q [B,N,Hq,d], Kt/Vt [B,N,Hkv,d] of one step, generated on the device."""
    if out is None:
        q = torch.empty(w.B, N, w.Hq, w.d, dtype=torch.bfloat16, device=device)
        kt = torch.empty(w.B, N, w.Hkv, w.d, dtype=torch.bfloat16, device=device)
        vt = torch.empty_like(kt)
    else:
        q, kt, vt = out
    tr.trsyn_rows_bf16(w.seed, synth.TAG_Q, step, q)
    tr.trsyn_rows_bf16(w.seed, synth.TAG_KT, step, kt)
    tr.trsyn_rows_bf16(w.seed, synth.TAG_VT, step, vt)
    return q, kt, vt


def fill_cache(w: synth.Workload, state):
    """Prefix K/V of every sequence into the state's cache (positions < L)."""
    L0 = torch.as_tensor(w.prefix_lengths(), dtype=torch.int32, device=state.L.device)
    tr.trsyn_cache_bf16(w.seed, synth.TAG_KC, L0, state.Kc)
    tr.trsyn_cache_bf16(w.seed, synth.TAG_VC, L0, state.Vc)


def warm_matrices(w: synth.Workload, state):
    tr.trsyn_warm_matrix(w.seed, state.M)
