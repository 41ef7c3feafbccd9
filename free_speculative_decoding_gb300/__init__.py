"""Python binding of libtr, the sm_103a hot path of Token Recycling.

Argument marshalling only: every function takes torch tensors that already
live on the current CUDA device, checks their dtypes and shapes, and hands raw
pointers and the current stream to the C ABI declared in ``include/tr.h``.
All arithmetic runs in libtr's CUDA kernels; there is no fallback.  Importing
the package works without a GPU (the library loads lazily), but every call
raises if ``libtr.so`` has not been built or the device is not an sm_103 GPU.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtr.so")

TR_OK, TR_E_INVAL, TR_E_UNSUPPORTED, TR_E_CUDA, TR_E_DEVICE, TR_E_TIMEOUT = range(6)
TR_DEV_BAD_TOKEN, TR_DEV_CACHE_FULL, TR_DEV_BAD_LENGTH, TR_DEV_TIMEOUT = 1, 2, 4, 8
TR_I32, TR_I64 = 0, 1
TR_F32, TR_BF16 = 0, 1
TR_INIT_ZERO, TR_INIT_RANDOM, TR_INIT_INHERIT = 0, 1, 2
TR_UPD_ALL, TR_UPD_ACCEPTED = 0, 1

_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_sz = ctypes.c_size_t
_f = ctypes.c_float


class TRError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__("%s failed: %s" % (fn, msg))
        self.code = code


class tr_step_args(ctypes.Structure):
    _fields_ = [
        ("B", _i), ("V", _i64), ("K", _i), ("tree", _p),
        ("M", _p), ("mtype", _i),
        ("logits", _p), ("ltype", _i), ("ld", _i64),
        ("H", _p), ("Wt", _p), ("D", _i),
        ("tree_tok", _p), ("ids", _p), ("vals", _p), ("acc_len", _p), ("path", _p), ("committed", _p),
        ("root", _p), ("L", _p),
        ("Kt", _p), ("Vt", _p), ("Kc", _p), ("Vc", _p), ("cap", _i), ("Hkv", _i), ("d", _i),
        ("mode", _i), ("ws", _p), ("ws_bytes", _sz),
    ]


# name -> (restype, argtypes)
_SIGS = {
    "tr_tree_create": (_i, [_p, _i, _i, ctypes.POINTER(_p)]),
    "tr_tree_destroy": (_i, [_p]),
    "tr_tree_info": (_i, [_p, _p, _p, _p, _p, _p]),
    "tr_init_matrix": (_i, [_p, _i, _i, _i64, _i, _i, _p, _u64, _p]),
    "tr_retrieve": (_i, [_p, _i, _i, _i64, _i, _p, _p, _p, _p]),
    "tr_verify_attn": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _f, _p, _p, _p, _sz, _p]),
    "tr_verify_attn_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _p]),
    "tr_topk": (_i, [_p, _i, _i64, _i64, _i64, _i, _p, _p, _p, _sz, _p]),
    "tr_topk_workspace_bytes": (_sz, [_i64, _i64, _i]),
    "tr_topk_noalloc": (_i, [_p, _i, _i64, _i64, _i64, _i, _p, _p, _p]),
    "tr_topk_softmax": (_i, [_p, _i, _i64, _i64, _i64, _i, _f, _p, _p, _p, _p, _p, _sz, _p]),
    "tr_softmax_steps": (_i, [_i64, _i]),
    "tr_accept_sampled": (_i, [_p, _i, _p, _p, _i, _p, _i, _i64, _i64, _p, _p, _f, _p, _p, _p, _p, _p, _p]),
    "tr_step_sampled": (_i, [ctypes.POINTER(tr_step_args), _f, _p, _p]),
    "tr_lmhead_topk": (_i, [_p, _p, _i64, _i, _i64, _i, _p, _p, _p, _sz, _p]),
    "tr_lmhead_topk_workspace_bytes": (_sz, [_i64, _i, _i64, _i]),
    "tr_accept": (_i, [_p, _i, _p, _p, _i, _p, _p, _p, _p, _p]),
    "tr_update": (_i, [_p, _i, _i, _i64, _i, _p, _p, _p, _i, _p, _p, _p]),
    "tr_kv_commit": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _p, _p, _p, _p, _sz, _p]),
    "tr_kv_commit_workspace_bytes": (_sz, [_i]),
    "tr_step": (_i, [ctypes.POINTER(tr_step_args), _p]),
    "tr_step_workspace_bytes": (_sz, [ctypes.POINTER(tr_step_args)]),
    "tr_get_status": (_i, [ctypes.POINTER(ctypes.c_int32), _p]),
    "tr_workspace_clear": (_i, [_p, _sz, _p]),
    "tr_set_wait_limit_ns": (_i, [_u64, ctypes.POINTER(_u64)]),
    "tr_status_string": (ctypes.c_char_p, [_i]),
    "trsyn_logits": (_i, [_u64, _i, _i64, _p, _p, _p, _i, _p, _i64, _p]),
    "trsyn_rows_bf16": (_i, [_u64, _i, _i64, _i, _i, _i, _i, _p, _p]),
    "trsyn_cache_bf16": (_i, [_u64, _i, _i, _i, _i, _i, _p, _p, _p]),
    "trsyn_lm_hidden": (_i, [_u64, _i, _i, _p, _p, _p, _p, _p]),
    "trsyn_lm_weight": (_i, [_u64, _i64, _i, _p, _p]),
    "trsyn_warm_matrix": (_i, [_u64, _i, _i64, _i, _i, _p, _p]),
    "trsyn_uniforms": (_i, [_u64, _i64, _i, _i, _i, _p, _p]),
}

ABI_SYMBOLS = tuple(_SIGS)
_LIB = None


def lib():
    """The loaded libtr (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libtr.so is not built: run __graft_entry__.build() "
                              "(or python free_speculative_decoding_gb300/build.py)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(fn, rc):
    if rc != TR_OK:
        raise TRError(fn, rc, lib().tr_status_string(rc).decode())


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on the CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _itype(M):
    if M.dtype == torch.int64:
        return TR_I64
    if M.dtype == torch.int32:
        return TR_I32
    raise ValueError("M must be int32 or int64")


def _ftype(x):
    if x.dtype == torch.float32:
        return TR_F32
    if x.dtype == torch.bfloat16:
        return TR_BF16
    raise ValueError("logits must be float32 or bfloat16")


def _i32(t, name):
    if t is not None and t.dtype != torch.int32:
        raise ValueError("%s must be int32" % name)


class Tree:
    """A static draft-tree plan (host memory; copied into each launch)."""

    def __init__(self, child_counts, K):
        counts = (ctypes.c_int32 * len(child_counts))(*[int(c) for c in child_counts])
        h = ctypes.c_void_p()
        _check("tr_tree_create", lib().tr_tree_create(counts, len(child_counts), int(K), ctypes.byref(h)))
        self._h = h
        self.K = int(K)
        n, dmax = ctypes.c_int(), ctypes.c_int()
        par = (ctypes.c_int32 * len(child_counts))()
        rank = (ctypes.c_int32 * len(child_counts))()
        depth = (ctypes.c_int32 * len(child_counts))()
        _check("tr_tree_info", lib().tr_tree_info(h, ctypes.byref(n), ctypes.byref(dmax), par, rank, depth))
        self.N = n.value
        self.max_depth = dmax.value
        self.parent = list(par)
        self.rank = list(rank)
        self.depth = list(depth)

    @property
    def handle(self):
        return self._h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _LIB is not None:
            _LIB.tr_tree_destroy(h)
            self._h = None


def tr_tree_create(child_counts, K):
    return Tree(child_counts, K)


def workspace(nbytes, device=None):
    """A zeroed byte workspace (every libtr call leaves its counters at zero again)."""
    return torch.zeros(max(int(nbytes), 1), dtype=torch.uint8, device=device or "cuda")


def tr_init_matrix(M, mode, src=None, seed=0):
    B, V, K = M.shape
    if src is not None and src.dtype != M.dtype:
        raise ValueError("src must have M's dtype")
    _check("tr_init_matrix", lib().tr_init_matrix(_ptr(M), _itype(M), B, V, K, mode, _ptr(src), seed, _stream()))


def tr_retrieve(M, tree, root, tree_tok):
    B, V, K = M.shape
    _i32(root, "root")
    _i32(tree_tok, "tree_tok")
    _check("tr_retrieve", lib().tr_retrieve(_ptr(M), _itype(M), B, V, K, tree.handle, _ptr(root), _ptr(tree_tok),
                                            _stream()))


def tr_verify_attn_workspace_bytes(B, Hq, Hkv, d, cap, tree):
    return lib().tr_verify_attn_workspace_bytes(B, Hq, Hkv, d, cap, tree.handle)


def tr_verify_attn(Q, Kt, Vt, Kc, Vc, L, tree, O, scale, ws):
    B, N, Hq, d = Q.shape
    Hkv, cap = Kc.shape[1], Kc.shape[2]
    for t, name in ((Q, "Q"), (Kt, "Kt"), (Vt, "Vt"), (Kc, "Kc"), (Vc, "Vc")):
        if t.dtype != torch.bfloat16:
            raise ValueError("%s must be bfloat16" % name)
    if O.dtype != torch.float32:
        raise ValueError("O must be float32")
    _i32(L, "L")
    _check("tr_verify_attn", lib().tr_verify_attn(_ptr(Q), _ptr(Kt), _ptr(Vt), _ptr(Kc), _ptr(Vc), _ptr(L), cap, B,
                                                  Hq, Hkv, d, float(scale), tree.handle, _ptr(O), _ptr(ws),
                                                  ws.numel(), _stream()))


def tr_topk_workspace_bytes(rows, V, K):
    return lib().tr_topk_workspace_bytes(rows, V, K)


def tr_topk(logits, K, ids, vals, ws, V=None):
    rows, ld = logits.shape
    V = ld if V is None else V
    _i32(ids, "ids")
    _check("tr_topk", lib().tr_topk(_ptr(logits), _ftype(logits), rows, V, ld, K, _ptr(ids), _ptr(vals),
                                    _ptr(ws) if ws is not None else None, ws.numel() if ws is not None else 0,
                                    _stream()))


TR_TOPK_NOALLOC_SCRATCH_BYTES = 4 << 20


def tr_topk_noalloc(logits, K, ids, vals, V=None):
    """tr_topk without a workspace: the library's static device scratch is used.

    For callers that cannot allocate device memory.  Calls on one device share
    the scratch, so they must not overlap on the GPU."""
    rows, ld = logits.shape
    V = ld if V is None else V
    _i32(ids, "ids")
    _check("tr_topk_noalloc", lib().tr_topk_noalloc(_ptr(logits), _ftype(logits), rows, V, ld, K, _ptr(ids),
                                                    _ptr(vals), _stream()))


def tr_softmax_steps(V, dtype):
    return lib().tr_softmax_steps(V, TR_F32 if dtype == torch.float32 else TR_BF16)


def tr_topk_softmax(logits, K, temperature, ids, vals, stats, step_stats, ws, V=None):
    """tr_topk plus stats [rows, 2] = (row max, sum of exp((x - max) / T)) and
    step_stats [rows, tr_softmax_steps(V, dtype), 2], the same pair per 8 KB step."""
    rows, ld = logits.shape
    V = ld if V is None else V
    _i32(ids, "ids")
    if stats.dtype != torch.float32 or step_stats.dtype != torch.float32:
        raise ValueError("stats must be float32")
    if step_stats.numel() < rows * tr_softmax_steps(V, logits.dtype) * 2:
        raise ValueError("step_stats too small")
    _check("tr_topk_softmax", lib().tr_topk_softmax(_ptr(logits), _ftype(logits), rows, V, ld, K, float(temperature),
                                                    _ptr(ids), _ptr(vals), _ptr(stats), _ptr(step_stats),
                                                    _ptr(ws) if ws is not None else None,
                                                    ws.numel() if ws is not None else 0, _stream()))


def tr_accept_sampled(tree, tree_tok, ids, logits, stats, step_stats, temperature, U, acc_len, path, committed,
                      bonus, V=None):
    B = tree_tok.shape[0]
    K = ids.shape[-1]
    V = logits.shape[1] if V is None else V
    if U.dtype != torch.float32 or stats.dtype != torch.float32 or step_stats.dtype != torch.float32:
        raise ValueError("U and the statistics must be float32")
    _check("tr_accept_sampled", lib().tr_accept_sampled(
        tree.handle, B, _ptr(tree_tok), _ptr(ids), K, _ptr(logits), _ftype(logits), V, logits.shape[1], _ptr(stats),
        _ptr(step_stats), float(temperature), _ptr(U), _ptr(acc_len), _ptr(path), _ptr(committed), _ptr(bonus),
        _stream()))


def tr_lmhead_topk_workspace_bytes(rows, D, V, K):
    return lib().tr_lmhead_topk_workspace_bytes(rows, D, V, K)


def tr_lmhead_topk(H, Wt, K, ids, vals, ws):
    rows, D = H.shape
    V = Wt.shape[0]
    if H.dtype != torch.bfloat16 or Wt.dtype != torch.bfloat16:
        raise ValueError("H and Wt must be bfloat16")
    _check("tr_lmhead_topk", lib().tr_lmhead_topk(_ptr(H), _ptr(Wt), rows, D, V, K, _ptr(ids), _ptr(vals), _ptr(ws),
                                                  ws.numel(), _stream()))


def tr_accept(tree, tree_tok, ids, acc_len, path, committed, bonus):
    B = tree_tok.shape[0]
    K = ids.shape[-1]
    _check("tr_accept", lib().tr_accept(tree.handle, B, _ptr(tree_tok), _ptr(ids), K, _ptr(acc_len), _ptr(path),
                                        _ptr(committed), _ptr(bonus), _stream()))


def tr_update(M, tree, tree_tok, ids, mode=TR_UPD_ALL, path=None, acc_len=None):
    B, V, K = M.shape
    _check("tr_update", lib().tr_update(_ptr(M), _itype(M), B, V, K, tree.handle, _ptr(tree_tok), _ptr(ids), mode,
                                        _ptr(path), _ptr(acc_len), _stream()))


def tr_kv_commit(Kt, Vt, Kc, Vc, L, tree, path, acc_len, ws):
    B, Hkv, cap, d = Kc.shape
    _check("tr_kv_commit", lib().tr_kv_commit(_ptr(Kt), _ptr(Vt), _ptr(Kc), _ptr(Vc), _ptr(L), cap, B, Hkv, d,
                                              tree.handle, _ptr(path), _ptr(acc_len), _ptr(ws), ws.numel(),
                                              _stream()))


def tr_kv_commit_workspace_bytes(B):
    return lib().tr_kv_commit_workspace_bytes(B)


def make_step_args(tree, M, tree_tok, ids, vals, acc_len, path, committed, root, L, logits=None, H=None, Wt=None,
                   Kt=None, Vt=None, Kc=None, Vc=None, mode=TR_UPD_ALL, ws=None):
    """Fill a tr_step_args structure from tensors (keeps no references)."""
    B, V, K = M.shape
    a = tr_step_args()
    a.B, a.V, a.K, a.tree = B, V, K, tree.handle
    a.M, a.mtype = _ptr(M), _itype(M)
    if logits is not None:
        a.logits, a.ltype, a.ld = _ptr(logits), _ftype(logits), logits.shape[1]
    if H is not None:
        a.H, a.Wt, a.D = _ptr(H), _ptr(Wt), H.shape[1]
    a.tree_tok, a.ids, a.vals = _ptr(tree_tok), _ptr(ids), _ptr(vals)
    a.acc_len, a.path, a.committed, a.root, a.L = _ptr(acc_len), _ptr(path), _ptr(committed), _ptr(root), _ptr(L)
    if Kt is not None:
        a.Kt, a.Vt, a.Kc, a.Vc = _ptr(Kt), _ptr(Vt), _ptr(Kc), _ptr(Vc)
        a.Hkv, a.cap, a.d = Kc.shape[1], Kc.shape[2], Kc.shape[3]
    a.mode = mode
    if ws is not None:
        a.ws, a.ws_bytes = _ptr(ws), ws.numel()
    return a


def tr_step_workspace_bytes(args):
    return lib().tr_step_workspace_bytes(ctypes.byref(args))


def tr_step(args):
    _check("tr_step", lib().tr_step(ctypes.byref(args), _stream()))


def tr_step_sampled(args, temperature, U):
    if U.dtype != torch.float32:
        raise ValueError("U must be float32")
    _check("tr_step_sampled", lib().tr_step_sampled(ctypes.byref(args), float(temperature), _ptr(U), _stream()))


def tr_set_wait_limit_ns(ns):
    """Sets the limit of every bounded device wait for later launches; returns the previous one."""
    prev = _u64()
    _check("tr_set_wait_limit_ns", lib().tr_set_wait_limit_ns(int(ns), ctypes.byref(prev)))
    return prev.value


def tr_workspace_clear(ws):
    _check("tr_workspace_clear", lib().tr_workspace_clear(_ptr(ws), ws.numel() * ws.element_size(), _stream()))


def tr_get_status():
    """Waits for the current stream, returns and clears the device status word."""
    v = ctypes.c_int32()
    rc = lib().tr_get_status(ctypes.byref(v), _stream())
    if rc not in (TR_OK, TR_E_DEVICE):
        _check("tr_get_status", rc)
    return v.value


# ---------------------------------------------------------------------------
# synthetic workload on the device (target-model stand-in, not the method)
# ---------------------------------------------------------------------------

def trsyn_logits(seed, tree, tree_tok, L, out, V=None):
    rows, ld = out.shape
    B = tree_tok.shape[0]
    V = ld if V is None else V
    _check("trsyn_logits", lib().trsyn_logits(seed, B, V, tree.handle, _ptr(tree_tok), _ptr(L), _ftype(out),
                                              _ptr(out), ld, _stream()))


def trsyn_rows_bf16(seed, tag, step, out):
    n0, n1, n2, d = out.shape
    _check("trsyn_rows_bf16", lib().trsyn_rows_bf16(seed, tag, step, n0, n1, n2, d, _ptr(out), _stream()))


def trsyn_cache_bf16(seed, tag, L, out):
    B, H, cap, d = out.shape
    _check("trsyn_cache_bf16", lib().trsyn_cache_bf16(seed, tag, B, H, cap, d, _ptr(L), _ptr(out), _stream()))


def trsyn_lm_hidden(seed, tree, tree_tok, L, out):
    B = tree_tok.shape[0]
    D = out.shape[1]
    _check("trsyn_lm_hidden", lib().trsyn_lm_hidden(seed, B, D, tree.handle, _ptr(tree_tok), _ptr(L), _ptr(out),
                                                    _stream()))


def trsyn_lm_weight(seed, out):
    V, D = out.shape
    _check("trsyn_lm_weight", lib().trsyn_lm_weight(seed, V, D, _ptr(out), _stream()))


def trsyn_uniforms(seed, step, out):
    B, N, K1 = out.shape
    _check("trsyn_uniforms", lib().trsyn_uniforms(seed, step, B, N, K1, _ptr(out), _stream()))


def trsyn_warm_matrix(seed, M):
    B, V, K = M.shape
    _check("trsyn_warm_matrix", lib().trsyn_warm_matrix(seed, B, V, K, _itype(M), _ptr(M), _stream()))
