"""The paged prefill entry point that needs no caller-provided workspace.

Callers that cannot allocate device memory (their runtime owns all of it, or
an allocation's device synchronisation is not acceptable where they run) use
gdn_chunk_gated_delta_rule_paged_static_workspace, whose workspace is a fixed
array inside the library.  These tests call it through the C ABI and compare
it with gdn_chunk_gated_delta_rule_paged (caller workspace) on the same
inputs, twice in a row with different shapes, so the second call runs on the
array the first one left behind.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import gated_deltanet_paged_gb300 as gdn
from gated_deltanet_paged_gb300 import workloads
from gpu_util import O_TOL, S_TOL, SCALE, rel_fro_rows

FN = "gdn_chunk_gated_delta_rule_paged_static_workspace"


def _fn():
    lib = gdn.library()
    f = getattr(lib, FN)
    P, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    f.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f32, P, i32, P, P, i32, P, P, P, P]
    f.restype = ctypes.c_int
    return f


def _static_call(f, c, pool, o):
    T, H = c.q.shape[0], c.q.shape[1]
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = f(p(c.q), p(c.k), p(c.v), p(c.g), p(c.beta), p(o), p(c.cu_seqlens), c.cu_seqlens.numel() - 1, T, H,
           128, 128, SCALE, p(pool), pool.shape[0], p(c.page_indices), p(c.page_indptr), c.page_size,
           p(c.last_page_len), None, None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, gdn.gdn_status_string(rc)


def _compare_pools(a, b):
    """Rows equal bit for bit, or (rows the calls wrote) within the state tolerance."""
    same = (a.view(torch.int32) == b.view(torch.int32)).flatten(1).all(dim=1)
    diff = torch.nonzero(~same).flatten()
    if diff.numel():
        ga, gb = a[diff].cpu().numpy(), b[diff].cpu().numpy()
        assert np.isfinite(gb).all()
        assert rel_fro_rows(gb, ga).max() <= S_TOL


@pytest.mark.gpu
def test_static_workspace_matches_caller_workspace_two_calls():
    f = _fn()
    w = workloads.worked_example("cuda")
    pool_ref, pool_st = w.pool.clone(), w.pool.clone()
    for c in w.calls:  # 2048-token prefix call, then the 452-token call
        o_ref = gdn.gdn_chunk_gated_delta_rule_paged(c.q, c.k, c.v, c.g, c.beta, c.cu_seqlens, pool_ref,
                                                     c.page_indices, c.page_indptr, c.page_size, c.last_page_len,
                                                     scale=SCALE)
        o_st = torch.empty_like(o_ref)
        _static_call(f, c, pool_st, o_st)
        torch.cuda.synchronize()
        d = (o_st.float() - o_ref.float()).abs().max().item()
        assert np.isfinite(d) and d <= O_TOL
        _compare_pools(pool_ref, pool_st)


@pytest.mark.gpu
def test_static_workspace_rejects_calls_beyond_its_size():
    f = _fn()
    fake = ctypes.c_void_p(0x10000)
    # 2^26 tokens x 32 heads need ~4 GB of workspace: refused before any device work
    rc = f(*([fake] * 7), 1, 1 << 26, 32, 128, 128, 0.0, fake, 8, fake, fake, 64, fake, None, None, None)
    assert rc == -2
