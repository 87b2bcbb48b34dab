"""GPU parity of the pool row utilities (gdn_pool_copy_rows, gdn_pool_zero_rows)
against their definition in the oracle package: bit-exact, fp32 and bf16
pools, -1 skips, rows outside the pool reported and skipped, and a
copy-on-write fork of a shared page followed by prefills that continue from
it ("gdn-prefix-cache", §The fix)."""
import numpy as np
import pytest
import torch

import gated_deltanet_paged_gb300 as gdn
import oracle
from gated_deltanet_paged_gb300 import workloads
from conftest import bf16_bits, f32, i32
from gpu_util import SCALE, Errors, bf16_pool_pair, check_o, check_pool

pytestmark = pytest.mark.gpu

GDN_DEVERR_PAGE_ID = 1


def _pools(pool, pool_dtype):
    """(GPU pool, oracle pool) of the same bits."""
    if pool_dtype == "bfloat16":
        g, o = bf16_pool_pair(pool)
        return g.cuda(), o
    return pool.cuda(), pool.numpy().copy()


def _bits(p):
    return p.view(torch.int16 if p.element_size() == 2 else torch.int32).cpu().numpy()


def _ora_bits(p):
    return p.view(np.int16) if p.dtype == np.uint16 else p.view(np.int32)


def _rows(x):
    return torch.tensor(x, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("pool_dtype", ["float32", "bfloat16"])
def test_copy_and_zero_rows_bit_exact(pool_dtype):
    H = 4
    pool = workloads.sentinel_pool(12, H, "cpu")  # NaN rows, each with its own payload
    workloads.fill_rows(pool, [1, 2, 5], torch.Generator().manual_seed(21))
    pool[2, 0, 0, :4] = torch.tensor([-0.0, float("inf"), -float("inf"), 1e-40])
    pg, po = _pools(pool, pool_dtype)
    src, dst = [1, -1, 2, 5, 7], [8, 3, 9, -1, 10]
    gdn.gdn_pool_copy_rows(pg, _rows(src), _rows(dst))
    oracle.pool_copy_rows(po, src, dst)
    torch.cuda.synchronize()
    assert (_bits(pg) == _ora_bits(po)).all()
    zero = [3, -1, 11, 8]
    gdn.gdn_pool_zero_rows(pg, _rows(zero))
    oracle.pool_zero_rows(po, zero)
    torch.cuda.synchronize()
    assert (_bits(pg) == _ora_bits(po)).all()
    assert (_bits(pg)[[3, 8, 11]] == 0).all()


def test_rows_outside_the_pool_are_reported_and_skipped():
    H = 2
    pool = workloads.sentinel_pool(8, H, "cpu")
    pg, po = _pools(pool, "float32")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_pool_copy_rows(pg, _rows([0, 99, 1]), _rows([5, 6, 7]), err_word=err)
    oracle.pool_copy_rows(po, [0, 99, 1], [5, 6, 7])
    torch.cuda.synchronize()
    assert int(err.item()) == (GDN_DEVERR_PAGE_ID << 24) | 1
    assert (_bits(pg) == _ora_bits(po)).all()
    err.zero_()
    gdn.gdn_pool_zero_rows(pg, _rows([8, 2]), err_word=err)
    oracle.pool_zero_rows(po, [8, 2])
    torch.cuda.synchronize()
    assert int(err.item()) == (GDN_DEVERR_PAGE_ID << 24) | 0
    assert (_bits(pg) == _ora_bits(po)).all()


@pytest.mark.parametrize("pool_dtype", ["float32", "bfloat16"])
def test_copy_on_write_fork_then_prefill(pool_dtype):
    """Two sequences share a 2000-token prefix in pages [7, 3] (page 3 holds the
    state after token 2000, 976 tokens into it).  Sequence B forks page 3 into
    page 13 before appending, so that its new tokens never touch the shared
    page; then both sequences prefill new tokens in one call, A into [7, 3, 12],
    B into [7, 13, 14].  Pages 7 and 3 keep their bits except that A writes its
    own boundary state to page 3."""
    H, ps = 2, 1024
    gen = torch.Generator().manual_seed(31)
    pool = workloads.sentinel_pool(16, H, "cpu")
    pg, po = _pools(pool, pool_dtype)
    errs = Errors()
    # the shared prefix: 2000 tokens into pages [7, 3]
    q, k, v, g, b = workloads.draw_tokens(gen, 2000, H, "cpu")
    ip, pi, lpl = workloads.page_table([2000], [7, 3], ps, "cpu")
    call = workloads.PrefillCall(q, k, v, g, b, torch.tensor([0, 2000], dtype=torch.int32), ip, pi, lpl, ps)
    _prefill(call, pg, po, errs)
    # fork: B's copy of the shared last page
    gdn.gdn_pool_copy_rows(pg, _rows([3]), _rows([13]))
    oracle.pool_copy_rows(po, [3], [13])
    torch.cuda.synchronize()
    assert (_bits(pg)[13] == _bits(pg)[3]).all()
    # both continue: A 300 new tokens on [7, 3, 12], B 700 on [7, 13, 14]
    lens = [300, 700]
    q, k, v, g, b = workloads.draw_tokens(gen, sum(lens), H, "cpu")
    ip, pi, lpl = workloads.page_table([2300, 2700], [7, 3, 12, 7, 13, 14], ps, "cpu")
    cu = torch.tensor([0, 300, 1000], dtype=torch.int32)
    before7 = _bits(pg)[7].copy()
    _, written = _prefill(workloads.PrefillCall(q, k, v, g, b, cu, ip, pi, lpl, ps), pg, po, errs)
    assert sorted(np.flatnonzero(written).tolist()) == [3, 12, 13, 14]
    assert (_bits(pg)[7] == before7).all()
    print("fork + prefill (%s pool): %r" % (pool_dtype, errs))


def _prefill(call, pg, po, errs):
    dev = lambda t: t.cuda().contiguous()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = pg.clone()
    o = gdn.gdn_chunk_gated_delta_rule_paged(dev(call.q), dev(call.k), dev(call.v), dev(call.g), dev(call.beta),
                                             dev(call.cu_seqlens), pg, dev(call.page_indices), dev(call.page_indptr),
                                             call.page_size, dev(call.last_page_len), scale=SCALE, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_ref, written = oracle.chunk_gated_delta_rule_paged(
        bf16_bits(call.q), bf16_bits(call.k), bf16_bits(call.v), f32(call.g), f32(call.beta), i32(call.cu_seqlens),
        po, i32(call.page_indices), i32(call.page_indptr), call.page_size, i32(call.last_page_len), SCALE)
    check_o(o, o_ref, errs)
    check_pool(pg, before, po, written, errs)
    return o, written
