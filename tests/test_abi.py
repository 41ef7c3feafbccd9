"""The C ABI without a GPU: the library loads, exports every declared symbol,
rejects bad arguments on the host, and builds the same tree plans as the oracle."""
import ctypes
import glob
import os
import re

import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from free_speculative_decoding_gb300 import build as b
    b.build()
    import free_speculative_decoding_gb300 as tr
    return tr.lib()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:int|size_t|const char\s*\*)\s*(\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    import free_speculative_decoding_gb300 as tr
    names = _declared()
    assert {"tr_retrieve", "tr_verify_attn", "tr_topk", "tr_lmhead_topk", "tr_accept", "tr_update",
            "tr_step", "tr_init_matrix", "tr_get_status"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(tr.ABI_SYMBOLS)


def test_tree_plan_matches_oracle(lib):
    import free_speculative_decoding_gb300 as tr
    for counts in (synth.TREE_T80, synth.TREE_T128, synth.chain_tree(5), (0,), (3, 2, 1, 0, 0, 0, 0)):
        t = tr.Tree(counts, 8)
        p = oracle.TreePlan(counts, 8)
        assert t.N == p.N and t.max_depth == p.max_depth
        assert t.parent == p.parent and t.rank == p.rank and t.depth == p.depth


@pytest.mark.parametrize("counts,K", [((4, 0, 0), 8), ((1, 0, 1), 8), ((9,) + (0,) * 9, 8), ((), 8),
                                      ((0,) * 129, 8), ((1, 0), 0), ((1, 0), 33)])
def test_tree_rejects_bad_specs(lib, counts, K):
    import free_speculative_decoding_gb300 as tr
    with pytest.raises(tr.TRError) as e:
        tr.Tree(counts, K)
    assert e.value.code == tr.TR_E_INVAL


def test_host_validation_before_any_launch(lib):
    import free_speculative_decoding_gb300 as tr
    p = ctypes.c_void_p(16)   # never dereferenced: validation fails first
    ws = ctypes.c_void_p(0)
    assert lib.tr_topk(p, tr.TR_F32, 4, 10, 10, 11, p, None, ws, 0, None) == tr.TR_E_INVAL      # K > V
    assert lib.tr_topk(p, tr.TR_F32, 4, 10, 8, 3, p, None, ws, 0, None) == tr.TR_E_INVAL       # ld < V
    assert lib.tr_topk(p, 7, 4, 10, 10, 3, p, None, ws, 0, None) == tr.TR_E_INVAL               # dtype
    assert lib.tr_topk(None, tr.TR_F32, 0, 10, 10, 3, None, None, ws, 0, None) == tr.TR_OK       # empty
    assert lib.tr_lmhead_topk(p, p, 4, 100, 10, 3, p, None, ws, 0, None) == tr.TR_E_UNSUPPORTED  # D % 64
    assert lib.tr_init_matrix(None, tr.TR_I64, 1, 10, 3, 0, None, 0, None) == tr.TR_E_INVAL
    assert lib.tr_init_matrix(p, tr.TR_I64, 1, 10, 3, tr.TR_INIT_INHERIT, None, 0, None) == tr.TR_E_INVAL
    t = tr.Tree(synth.TREE_T80, 8)
    assert lib.tr_retrieve(p, tr.TR_I64, 1, 100, 4, t.handle, p, p, None) == tr.TR_E_INVAL       # K mismatch
    assert lib.tr_verify_attn(p, p, p, p, p, p, 64, 1, 6, 4, 128, 0.1, t.handle, p, p, 1 << 30,
                              None) == tr.TR_E_INVAL                                               # Hq % Hkv
    assert lib.tr_verify_attn(p, p, p, p, p, p, 64, 1, 4, 4, 64, 0.1, t.handle, p, p, 1 << 30,
                              None) == tr.TR_E_UNSUPPORTED                                         # d != 128
    for bad_scale in (0.0, -0.1, float("inf"), float("nan")):
        assert lib.tr_verify_attn(p, p, p, p, p, p, 64, 1, 4, 4, 128, bad_scale, t.handle, p, p, 1 << 30,
                                  None) == tr.TR_E_INVAL                                           # scale
    assert lib.tr_update(p, tr.TR_I64, 1, 100, 8, t.handle, p, p, tr.TR_UPD_ACCEPTED, None, None,
                         None) == tr.TR_E_INVAL
    assert lib.tr_get_status(None, None) == tr.TR_E_INVAL
    assert lib.tr_status_string(tr.TR_E_CUDA).startswith(b"TR_E_CUDA")


def test_workspace_sizes(lib):
    import free_speculative_decoding_gb300 as tr
    # rows of at most one 8 KB unit (2048 fp32 elements) are never split and
    # need no workspace; longer rows need a K-key list slot per unit (8-byte
    # keys, 16 units for a 32000-entry fp32 row) and a counter per row
    assert lib.tr_topk_workspace_bytes(10, 2048, 8) == 0
    assert lib.tr_topk_workspace_bytes(10, 2049, 8) > 0
    assert lib.tr_topk_workspace_bytes(1280, 32000, 8) >= 1280 * 16 * 8 * 8 + 1280 * 4
    assert lib.tr_topk_workspace_bytes(1024, 128256, 8) >= 1024 * 63 * 8 * 8 + 1024 * 4
    assert lib.tr_topk_workspace_bytes(33, 20000, 16) >= 33 * 10 * 16 * 8 + 33 * 4
    t = tr.Tree(synth.TREE_T80, 8)
    assert lib.tr_verify_attn_workspace_bytes(16, 32, 32, 128, 5888, t.handle) > 0
    assert lib.tr_kv_commit_workspace_bytes(16) >= 64


def test_step_and_noalloc_validation_before_any_launch(lib):
    # every case is refused on the host, before the device is touched
    import free_speculative_decoding_gb300 as tr
    t = tr.Tree(synth.TREE_T80, 8)
    p = 16  # an address that is never dereferenced

    def args(**kw):
        a = tr.tr_step_args(B=2, V=1000, K=8, tree=t.handle, M=p, mtype=tr.TR_I64, logits=p, ltype=tr.TR_F32,
                            ld=1000, tree_tok=p, ids=p, acc_len=p, path=p, committed=p, root=p, L=p,
                            mode=tr.TR_UPD_ALL)
        a.ws, a.ws_bytes = p, 1 << 40
        for k, v in kw.items():
            setattr(a, k, v)
        return a

    step = lambda a: lib.tr_step(ctypes.byref(a), None)
    assert lib.tr_step(None, None) == tr.TR_E_INVAL
    assert step(args(K=4)) == tr.TR_E_INVAL                       # K differs from the tree's
    assert step(args(mtype=9)) == tr.TR_E_INVAL
    assert step(args(mode=9)) == tr.TR_E_INVAL
    assert step(args(logits=None)) == tr.TR_E_INVAL               # neither logits nor H and Wt
    assert step(args(M=None)) == tr.TR_E_INVAL
    assert step(args(Kt=p, Vt=None, Kc=p, Vc=p, cap=64, Hkv=2, d=128)) == tr.TR_E_INVAL   # Kt without Vt
    assert step(args(Kt=p, Vt=p, Kc=p + 8, Vc=p, cap=64, Hkv=2, d=128)) == tr.TR_E_INVAL  # misaligned cache
    assert step(args(Kt=p, Vt=p, Kc=p, Vc=p, cap=64, Hkv=2, d=100)) == tr.TR_E_INVAL      # d % 8
    a = args()
    a.ws_bytes = 0
    assert step(a) == tr.TR_E_INVAL                                  # workspace too small
    assert lib.tr_step_workspace_bytes(ctypes.byref(args())) > 0
    # the allocation-free top-K refuses what its static scratch cannot hold
    assert lib.tr_topk_noalloc(p, tr.TR_F32, 4, 10, 10, 11, p, None, None) == tr.TR_E_INVAL          # K > V
    assert lib.tr_topk_noalloc(p, tr.TR_F32, 70000, 10, 10, 3, p, None, None) == tr.TR_E_UNSUPPORTED  # rows
    assert lib.tr_topk_noalloc(p, tr.TR_BF16, 60000, 128256, 128256, 8, p, None,
                               None) == tr.TR_E_UNSUPPORTED                                           # scratch


def test_wait_limit_is_host_state(lib):
    """tr_set_wait_limit_ns only records the limit later launches take (no GPU needed)."""
    import free_speculative_decoding_gb300 as tr
    prev = ctypes.c_uint64()
    assert lib.tr_set_wait_limit_ns(0, ctypes.byref(prev)) == tr.TR_E_INVAL
    assert lib.tr_set_wait_limit_ns(61_000_000_000, None) == tr.TR_E_INVAL
    assert tr.tr_set_wait_limit_ns(5000) == 2_000_000_000
    assert tr.tr_set_wait_limit_ns(2_000_000_000) == 5000
