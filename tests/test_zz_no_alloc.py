"""The paged prefill entry point that needs no caller-provided workspace.

Callers that cannot allocate device memory (their runtime owns all of it, or
an allocation's device synchronisation is not acceptable where they run) use
gdn_chunk_gated_delta_rule_paged_static_workspace, whose workspace is a fixed
array inside the library.  These tests call it through the C ABI and compare
it with gdn_chunk_gated_delta_rule_paged (caller workspace) on the same
inputs, twice in a row with different shapes, so the second call runs on the
array the first one left behind; the results must be identical bit for bit and
match the oracle.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import gated_deltanet_paged_gb300 as gdn
from gated_deltanet_paged_gb300 import workloads
import oracle
from conftest import bf16_bits, f32, i32
from gpu_util import SCALE, Errors, check_o, check_pool

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


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


@pytest.mark.gpu
def test_static_workspace_matches_caller_workspace_two_calls():
    """Both calls run the same kernels, which do no atomic or order-dependent
    arithmetic and write every workspace entry they read, so the outputs and
    the whole pool must agree bit for bit, also on the second call, which runs
    over what the first one left in the array.  The static-workspace results
    are also checked against the oracle directly."""
    f = _fn()
    w = workloads.worked_example("cuda")
    pool_ref, pool_st = w.pool.clone(), w.pool.clone()
    pool_ora = w.pool.cpu().numpy().copy()
    errs = Errors()
    for c in w.calls:  # 2048-token prefix call, then the 452-token call
        o_ref = gdn.gdn_chunk_gated_delta_rule_paged(c.q, c.k, c.v, c.g, c.beta, c.cu_seqlens, pool_ref,
                                                     c.page_indices, c.page_indptr, c.page_size, c.last_page_len,
                                                     scale=SCALE)
        o_st = torch.full_like(o_ref, float("nan"))
        before = pool_st.clone()
        _static_call(f, c, pool_st, o_st)
        torch.cuda.synchronize()
        assert torch.equal(_bits(o_st), _bits(o_ref))
        assert torch.equal(_bits(pool_st), _bits(pool_ref))
        o_ora, written = oracle.chunk_gated_delta_rule_paged(
            bf16_bits(c.q), bf16_bits(c.k), bf16_bits(c.v), f32(c.g), f32(c.beta), i32(c.cu_seqlens), pool_ora,
            i32(c.page_indices), i32(c.page_indptr), c.page_size, i32(c.last_page_len), SCALE)
        check_o(o_st, o_ora, errs)
        check_pool(pool_st, before, pool_ora, written, errs)
    print("static workspace, worked example: %r" % errs)


@pytest.mark.gpu
def test_static_workspace_rejects_calls_beyond_its_size():
    """2^26 tokens x 32 heads need about 4 GB of workspace: refused before any
    device work.  Every array pointer is NULL, so that a call which got past
    the size check would stop at the host's argument check (-1) and could not
    launch anything."""
    f = _fn()
    rc = f(*([None] * 7), 1, 1 << 26, 32, 128, 128, 0.0, None, 8, None, None, 64, None, None, None, None)
    assert rc == -2
