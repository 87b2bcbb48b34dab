"""GPU parity at the full workload sizes: the 256-sequence decode batch, the
64-sequence mixed prefill through the general slot API, and the 4 x 65,536
token long-context prefill followed by 128 decode steps.  The oracle runs on
every (sequence, head) chain of each; rows outside the write sets must keep
their bits."""
import numpy as np
import pytest
import torch

import gated_deltanet_paged_gb300 as gdn
import oracle
from gated_deltanet_paged_gb300 import workloads
from conftest import bf16_bits, f32, i32
from gpu_util import SCALE, Errors, bits_equal, check_o, check_pool, rel_fro_rows, S_TOL, S_TOL_BF16, O_TOL

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.mark.parametrize("pool_dtype", ["float32", "bfloat16"])
def test_decode_batch_full_size(pool_dtype):
    """The full decode batch (B = 256, H = 32) on its 10,000-row pool, fp32 or
    bf16 (the same values cut to bf16)."""
    w = workloads.decode_batch("cuda")
    call = w.calls[0]
    pool = w.pool if pool_dtype == "float32" else (w.pool.view(torch.int32) >> 16).to(torch.int16).view(torch.bfloat16)
    ip, pi, lpl = (i32(t) for t in (call.page_indptr, call.page_indices, call.last_page_len))
    s = oracle.decode_slots(ip, pi, lpl, call.page_size)
    slots = gdn.gdn_paged_decode_slots(call.page_indptr, call.page_indices, call.last_page_len)
    for k in s:
        assert (slots[k].cpu().numpy() == s[k]).all()
    rows = sorted(set(s["initial_state_indices"].tolist()) | set(s["output_state_indices"].tolist()))
    rows = [r for r in rows if r >= 0]
    remap = {r: i for i, r in enumerate(rows)}
    local = pool[torch.tensor(rows, device="cuda")].cpu()
    local = local.view(torch.int16).numpy().view(np.uint16).copy() if pool_dtype == "bfloat16" else local.numpy()
    before = pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = gdn.gdn_gated_delta_rule_decode_paged(call.q, call.k, call.v, call.g, call.beta, pool, call.page_indices,
                                              call.page_indptr, call.last_page_len, scale=SCALE, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    o_ref, written = oracle.gated_delta_rule_decode(
        bf16_bits(call.q), bf16_bits(call.k), bf16_bits(call.v), f32(call.g), f32(call.beta), local,
        [remap.get(r, -1) for r in s["initial_state_indices"].tolist()],
        [remap[r] for r in s["output_state_indices"].tolist()], SCALE)
    errs = Errors()
    check_o(o, o_ref, errs)
    wrows = [rows[i] for i in np.flatnonzero(written)]
    got = pool[torch.tensor(wrows, device="cuda")].float().cpu().numpy()
    ref = local[np.flatnonzero(written)]
    if pool_dtype == "bfloat16":
        ref = (ref.astype(np.uint32) << 16).view(np.float32)
    e = rel_fro_rows(got, ref)
    errs.state = float(e.max())
    assert e.max() <= (S_TOL_BF16 if pool_dtype == "bfloat16" else S_TOL)
    keep = torch.ones(pool.shape[0], dtype=torch.bool, device="cuda")
    keep[torch.tensor(wrows, device="cuda")] = False
    assert bits_equal(pool[keep], before[keep])
    print("decode batch B=256 H=32 %s pool: %r" % (pool_dtype, errs))


def _checkpoint_layout(prefix, lens, N):
    """Checkpoint count per sequence, (prefix + len) // N - prefix // N
    ("Slot arguments"), laid out densely: (cu_starts, total)."""
    counts = (prefix + lens) // N - prefix // N
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int32)
    return starts, int(counts.sum())


def test_mixed_prefill_general_api_full_size():
    w = workloads.mixed_prefill("cpu")
    call = w.calls[0]
    N = w.checkpoint_every
    P, L = w.prefix_lens.numpy(), w.seq_lens.numpy()
    ccs, total = _checkpoint_layout(P, L, N)
    dev = lambda t: torch.as_tensor(t).cuda()
    cu, ip, pi, lpl = dev(call.cu_seqlens), dev(call.page_indptr), dev(call.page_indices), dev(call.last_page_len)
    slots = gdn.gdn_paged_prefill_slots(cu, ip, pi, lpl, call.page_size)
    ref = oracle.prefill_slots(i32(call.cu_seqlens), i32(call.page_indptr), i32(call.page_indices),
                               i32(call.last_page_len), call.page_size)
    for k in ref:
        assert (slots[k].cpu().numpy() == ref[k]).all(), k
    assert (ref["prefix_lens"] == P).all()
    cki = np.arange(total, dtype=np.int32)
    ck = workloads.sentinel_pool(total, w.H, "cpu")
    pool_g, ck_g = w.pool.cuda(), ck.cuda()
    pb, cb = pool_g.clone(), ck_g.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = gdn.gdn_chunk_gated_delta_rule(
        dev(call.q), dev(call.k), dev(call.v), dev(call.g), dev(call.beta), cu, scale=SCALE, initial_state=pool_g,
        state_indices=slots["state_indices"], output_state=pool_g,
        output_state_indices=slots["output_state_indices"], state_checkpoints=ck_g,
        checkpoint_state_indices=dev(cki), checkpoint_cu_starts=dev(ccs), prefix_lens=slots["prefix_lens"],
        checkpoint_every_n_tokens=N, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    # without the error word: the same bits
    pool_f, ck_f = pb.clone(), cb.clone()
    o_f = gdn.gdn_chunk_gated_delta_rule(
        dev(call.q), dev(call.k), dev(call.v), dev(call.g), dev(call.beta), cu, scale=SCALE, initial_state=pool_f,
        state_indices=slots["state_indices"], output_state=pool_f,
        output_state_indices=slots["output_state_indices"], state_checkpoints=ck_f,
        checkpoint_state_indices=dev(cki), checkpoint_cu_starts=dev(ccs), prefix_lens=slots["prefix_lens"],
        checkpoint_every_n_tokens=N)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_f.view(torch.int16)), "outputs differ without the error word"
    assert bits_equal(pool_g, pool_f) and bits_equal(ck_g, ck_f), "states differ without the error word"
    del o_f, pool_f, ck_f
    pool_o, ck_o = w.pool.numpy().copy(), ck.numpy().copy()
    o_ref, w_out, w_ck = oracle.chunk_gated_delta_rule(
        bf16_bits(call.q), bf16_bits(call.k), bf16_bits(call.v), f32(call.g), f32(call.beta), i32(call.cu_seqlens),
        SCALE, initial_state=pool_o, state_indices=ref["state_indices"], output_state=pool_o,
        output_state_indices=ref["output_state_indices"], state_checkpoints=ck_o, checkpoint_state_indices=cki,
        checkpoint_cu_starts=ccs, prefix_lens=P, checkpoint_every_n_tokens=N)
    errs = Errors()
    check_o(o, o_ref, errs)
    check_pool(pool_g, pb, pool_o, w_out, errs, "pool")
    check_pool(ck_g, cb, ck_o, w_ck, errs, "checkpoints")
    assert w_ck.all()
    print("mixed prefill S=64 H=16 (T=%d, %d checkpoints): %r" % (call.q.shape[0], total, errs))


def test_long_context_prefill_then_decode():
    """The long-context workload in full: the 4 x 65,536-token prefill with
    H = 32 (128 (sequence, head) chains, 57 state stores each), then 128 decode
    steps on the same pool, every chain against the oracle.  Outputs are
    compared element by element, every written state row by row, and every
    other pool row bit for bit.  The oracle runs one sequence (32 chains) at a
    time so that its fp64 outputs stay a few GB."""
    w = workloads.long_context("cuda")
    pre, decs = w.calls[0], w.calls[1:]
    pool = w.pool
    before = pool.clone()
    pool_ora = pool.cpu().numpy().copy()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = gdn.gdn_chunk_gated_delta_rule_paged(pre.q, pre.k, pre.v, pre.g, pre.beta, pre.cu_seqlens, pool,
                                             pre.page_indices, pre.page_indptr, pre.page_size, pre.last_page_len,
                                             scale=SCALE, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    # the same call without the error word (the kernels without the device
    # checks, the ones the benchmark times) gives the same bits
    pool_fast = before.clone()
    o_fast = gdn.gdn_chunk_gated_delta_rule_paged(pre.q, pre.k, pre.v, pre.g, pre.beta, pre.cu_seqlens, pool_fast,
                                                  pre.page_indices, pre.page_indptr, pre.page_size,
                                                  pre.last_page_len, scale=SCALE)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_fast.view(torch.int16)), "outputs differ without the error word"
    assert bits_equal(pool, pool_fast), "pool differs without the error word"
    del o_fast, pool_fast

    cu = pre.cu_seqlens.cpu().numpy()
    ip = pre.page_indptr.cpu().numpy()
    pages = pre.page_indices.cpu().numpy()
    lpl = i32(pre.last_page_len)
    errs = Errors()
    written = np.zeros(pool.shape[0], bool)
    for b in range(len(cu) - 1):
        sl = slice(int(cu[b]), int(cu[b + 1]))
        ids = pages[ip[b]:ip[b + 1]]
        o_ref, w_b = oracle.chunk_gated_delta_rule_paged(
            bf16_bits(pre.q[sl]), bf16_bits(pre.k[sl]), bf16_bits(pre.v[sl]), f32(pre.g[sl]), f32(pre.beta[sl]),
            [0, sl.stop - sl.start], pool_ora, ids, [0, len(ids)], pre.page_size, lpl[b:b + 1], SCALE)
        assert w_b[ids].all() and w_b.sum() == len(ids)  # 57 pages, each written once
        check_o(o[sl], o_ref, errs)
        del o_ref
        written |= w_b.astype(bool)
    check_pool(pool, before, pool_ora, written, errs, "prefill")

    # 128 decode steps on the same pool (in place; last_page_len 1025 .. 1152),
    # each side continuing from its own fp32 pool
    before = pool.clone()
    written = np.zeros(pool.shape[0], bool)
    for step, call in enumerate(decs):
        o_d = gdn.gdn_gated_delta_rule_decode_paged(call.q, call.k, call.v, call.g, call.beta, pool,
                                                    call.page_indices, call.page_indptr, call.last_page_len,
                                                    scale=SCALE, err_word=err)
        o_ref, w_d = oracle.gated_delta_rule_decode_paged(
            bf16_bits(call.q), bf16_bits(call.k), bf16_bits(call.v), f32(call.g), f32(call.beta), pool_ora,
            i32(call.page_indices), i32(call.page_indptr), i32(call.last_page_len), call.page_size, SCALE)
        check_o(o_d, o_ref, errs)
        written |= w_d.astype(bool)
    torch.cuda.synchronize()
    assert err.item() == 0
    check_pool(pool, before, pool_ora, written, errs, "decode")
    print("long context 4 x 65536, H=32, then 128 decode steps, all chains: %r" % errs)


def test_prefill_and_decode_are_deterministic():
    """The kernels do no atomic or order-dependent arithmetic, so repeating a
    call on the same inputs gives the same bits.  Runs the prefill of a
    multi-chunk, multi-page workload (4 x 16,384 tokens, H = 32: many chunk-local
    work items per CTA, page-boundary stores, every warp role of the chain busy)
    and the full decode batch three times each; any race between the kernels'
    warp roles or CTAs would show as a difference between the repeats."""
    w = workloads.long_context("cuda", L=16384, decode_steps=0)
    pre = w.calls[0]
    outs, pools = [], []
    for rep in range(8):  # three with the error word, five without (the benchmark's kernels)
        pool = w.pool.clone()
        err = torch.zeros(1, dtype=torch.int32, device="cuda") if rep < 3 else None
        o = gdn.gdn_chunk_gated_delta_rule_paged(pre.q, pre.k, pre.v, pre.g, pre.beta, pre.cu_seqlens, pool,
                                                 pre.page_indices, pre.page_indptr, pre.page_size,
                                                 pre.last_page_len, scale=SCALE, err_word=err)
        torch.cuda.synchronize()
        assert err is None or err.item() == 0
        outs.append(o)
        pools.append(pool)
    for r in range(1, 8):
        assert torch.equal(outs[0].view(torch.int16), outs[r].view(torch.int16)), "prefill outputs differ"
        assert bits_equal(pools[0], pools[r]), "prefill states differ"
    del outs, pools

    wd = workloads.decode_batch("cuda")  # 21 GB pool: one extra copy at a time
    dc = wd.calls[0]
    first = None
    for _ in range(3):
        dpool = wd.pool.clone()
        od = gdn.gdn_gated_delta_rule_decode_paged(dc.q, dc.k, dc.v, dc.g, dc.beta, dpool, dc.page_indices,
                                                   dc.page_indptr, dc.last_page_len, scale=SCALE)
        torch.cuda.synchronize()
        if first is None:
            first = (od, dpool)
        else:
            assert torch.equal(first[0].view(torch.int16), od.view(torch.int16)), "decode outputs differ"
            assert bits_equal(first[1], dpool), "decode states differ"
        del dpool
