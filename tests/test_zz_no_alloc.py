"""The allocation-free top-K entry point against the oracle and the workspace one (GB300 only).

tr_topk_noalloc exists for callers that cannot allocate device memory (a
plugin whose host framework owns every buffer, a serving loop that must not
call cudaMalloc, a foreign-function caller without an allocator).  It must
give exactly the oracle's top-K, and so what tr_topk gives -- top-K IDs are
integers and the values are copied logits, so the comparison is exact, as in
every top-K test here -- on
two calls in a row, which also shows that the shared static scratch carries no
state from one call to the next.  This file is collected last so a
stop-at-first-failure run has already run everything else; it also passes
alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tr():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from free_speculative_decoding_gb300 import build as b
    b.build()
    import free_speculative_decoding_gb300 as m
    return m


def _both(tr, x, K):
    rows, V = x.shape
    ids_a = torch.full((rows, K), -7, dtype=torch.int32, device="cuda")
    vals_a = torch.zeros(rows, K, dtype=torch.float32, device="cuda")
    tr.tr_topk(x, K, ids_a, vals_a, tr.workspace(tr.tr_topk_workspace_bytes(rows, V, K)))
    ids_b = torch.full((rows, K), -7, dtype=torch.int32, device="cuda")
    vals_b = torch.zeros(rows, K, dtype=torch.float32, device="cuda")
    # straight through the C ABI
    rc = tr.lib().tr_topk_noalloc(ctypes.c_void_p(x.data_ptr()),
                                  tr.TR_F32 if x.dtype == torch.float32 else tr.TR_BF16, rows, V, V, K,
                                  ctypes.c_void_p(ids_b.data_ptr()), ctypes.c_void_p(vals_b.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == tr.TR_OK
    torch.cuda.synchronize()
    return (ids_a.cpu().numpy(), vals_a.cpu().numpy()), (ids_b.cpu().numpy(), vals_b.cpu().numpy())


@pytest.mark.parametrize("rows,V,K,dtype", [(640, 32000, 8, torch.float32), (96, 128256, 8, torch.bfloat16),
                                            (33, 20000, 16, torch.float32)])
def test_noalloc_matches_workspace_topk_twice(tr, rows, V, K, dtype):
    g = torch.Generator().manual_seed(rows + V)
    for call in range(2):
        x = (torch.round(torch.randn(rows, V, generator=g) * 8) / 8).to(dtype).cuda()   # ties included
        (ia, va), (ib, vb) = _both(tr, x, K)
        ids_ref, vals_ref = oracle.topk_rows(x.float().cpu().numpy(), K)
        assert np.array_equal(ib, ids_ref), "ids differ from the oracle on call %d" % call
        assert np.array_equal(vb, vals_ref.astype(np.float32)), "values differ from the oracle on call %d" % call
        assert np.array_equal(ia, ib), "ids differ on call %d" % call
        assert np.array_equal(va, vb), "values differ on call %d" % call
        assert (ia >= 0).all()
    assert tr.tr_get_status() == 0


def test_noalloc_binding_and_size_limit(tr):
    x = torch.randn(40, 30000, device="cuda")
    ids = torch.zeros(40, 8, dtype=torch.int32, device="cuda")
    tr.tr_topk_noalloc(x, 8, ids, None)
    ref = torch.zeros_like(ids)
    tr.tr_topk(x, 8, ref, None, tr.workspace(tr.tr_topk_workspace_bytes(40, 30000, 8)))
    assert torch.equal(ids, ref)
    # scratch beyond the static maximum is refused before any launch
    rows = 60000
    assert tr.tr_topk_workspace_bytes(rows, 128256, 8) > tr.TR_TOPK_NOALLOC_SCRATCH_BYTES
    rc = tr.lib().tr_topk_noalloc(ctypes.c_void_p(x.data_ptr()), tr.TR_F32, rows, 128256, 128256, 8,
                                  ctypes.c_void_p(ids.data_ptr()), None, None)
    assert rc == tr.TR_E_UNSUPPORTED
