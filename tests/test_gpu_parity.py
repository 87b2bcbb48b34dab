"""GPU parity of the CUDA library against the fp64 oracle on small cases:
the tiny two-sequence workload, the worked 2500-token example, ragged
prefixes / lengths around the 64-token chunk, the general slot API with -1
rows, and device-side validation."""
import numpy as np
import pytest
import torch

import gated_deltanet_paged_gb300 as gdn
import oracle
from gated_deltanet_paged_gb300 import workloads
from conftest import bf16_bits, f32, i32
from gpu_util import (SCALE, Errors, bf16_pool_pair, bits_equal, check_o, check_pool, decode_paged_both,
                      prefill_paged_both)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("use_slots", [False, True])
@pytest.mark.parametrize("decay", [1.0, 0.01])
def test_tiny_workload(decay, use_slots):
    w = workloads.tiny("cpu", decay)
    pool_gpu, pool_ora = w.pool.cuda(), w.pool.numpy().copy()
    errs = Errors()
    for call in w.calls:
        if call.kind == "prefill":
            prefill_paged_both(call, pool_gpu, pool_ora, errs, use_slots)
        else:
            decode_paged_both(call, pool_gpu, pool_ora, errs, use_slots)
    print("tiny decay=%g slots=%s: %r" % (decay, use_slots, errs))


@pytest.mark.parametrize("decay", [1.0, 0.01])
def test_bf16_pool_tiny_workload(decay):
    """The tiny workload (prefill from empty and non-empty prefixes, then
    decode) on a bf16 state pool, through the paged prefill and decode calls."""
    w = workloads.tiny("cpu", decay)
    pool_gpu, pool_ora = bf16_pool_pair(w.pool)
    pool_gpu = pool_gpu.cuda()
    errs = Errors()
    for call in w.calls:
        if call.kind == "prefill":
            prefill_paged_both(call, pool_gpu, pool_ora, errs)
        else:
            decode_paged_both(call, pool_gpu, pool_ora, errs, use_slots=True)
    print("tiny decay=%g bf16 pool: %r" % (decay, errs))


@pytest.mark.parametrize("decay", [1.0, 0.01])
def test_bf16_pool_worked_example(decay):
    """The worked 2500-token example on a bf16 pool: page 12 written, pages 7
    and 3 bit-unchanged by the second call."""
    w = workloads.worked_example("cpu", decay)
    pool_gpu, pool_ora = bf16_pool_pair(w.pool)
    pool_gpu = pool_gpu.cuda()
    errs = Errors()
    prefill_paged_both(w.calls[0], pool_gpu, pool_ora, errs)
    kept = pool_gpu[[7, 3]].clone()
    _, written = prefill_paged_both(w.calls[1], pool_gpu, pool_ora, errs)
    assert np.flatnonzero(written).tolist() == [12]
    assert bits_equal(pool_gpu[[7, 3]], kept)
    print("worked example decay=%g bf16 pool: %r" % (decay, errs))


@pytest.mark.parametrize("decay", [1.0, 0.01])
def test_worked_example(decay):
    """2048 cached tokens in pages [7, 3], 452 new with page 12: the second
    call reads page 3, writes page 12 and leaves 7 and 3 bit-unchanged."""
    w = workloads.worked_example("cpu", decay)
    pool_gpu, pool_ora = w.pool.cuda(), w.pool.numpy().copy()
    errs = Errors()
    prefill_paged_both(w.calls[0], pool_gpu, pool_ora, errs)
    kept = pool_gpu[[7, 3]].clone()
    _, written = prefill_paged_both(w.calls[1], pool_gpu, pool_ora, errs)
    assert np.flatnonzero(written).tolist() == [12]
    assert bits_equal(pool_gpu[[7, 3]], kept)
    print("worked example decay=%g: %r" % (decay, errs))


def _ragged_case(seed, ps, lens, prefixes, H=2, decay=1.0):
    gen = torch.Generator().manual_seed(seed)
    ctx = [l + p for l, p in zip(lens, prefixes)]
    npages = sum(max(1, -(-c // ps)) for c in ctx)
    ids = torch.randperm(npages + 3, generator=gen)
    ip, pi, lpl = workloads.page_table(ctx, ids, ps, "cpu")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q, k, v, g, b = workloads.draw_tokens(gen, int(sum(lens)), H, "cpu", decay)
    pool = workloads.sentinel_pool(npages + 3, H, "cpu")
    s = oracle.prefill_slots(i32(cu), i32(ip), i32(pi), i32(lpl), ps)
    workloads.fill_rows(pool, [r for r in s["state_indices"].tolist() if r >= 0], gen)
    return workloads.PrefillCall(q, k, v, g, b, cu, ip, pi, lpl, ps), pool


RAGGED = [
    (64, [1, 5, 63, 64, 65, 127, 128, 200], [0, 0, 0, 0, 0, 0, 0, 0]),
    (64, [1, 5, 63, 64, 65, 127, 128, 200], [1, 63, 64, 65, 127, 128, 129, 191]),
    (128, [3, 61, 64, 70, 129, 250, 0, 300], [60, 4, 128, 58, 1, 6, 77, 255]),
    (192, [500, 1, 191, 192, 193], [191, 383, 1, 0, 64]),
]


@pytest.mark.parametrize("decay", [1.0, 0.01])
@pytest.mark.parametrize("case", range(len(RAGGED)))
def test_ragged_prefixes_and_tails(case, decay):
    ps, lens, prefixes = RAGGED[case]
    call, pool = _ragged_case(100 + case, ps, lens, prefixes, decay=decay)
    errs = Errors()
    prefill_paged_both(call, pool.cuda(), pool.numpy().copy(), errs)
    print("ragged case %d decay=%g: %r" % (case, decay, errs))


def test_long_ragged_sequences():
    """Long chains next to short ones: 188 and 313 chunks (prefixes 0 and 129,
    so the second starts with a partial chunk), 47 chunks and 2 chunks, with a
    page store every 10 chunks."""
    call, pool = _ragged_case(7, 640, [12000, 3000, 20000, 100], [0, 70, 129, 5])
    errs = Errors()
    prefill_paged_both(call, pool.cuda(), pool.numpy().copy(), errs)
    print("long ragged sequences: %r" % errs)


@pytest.mark.parametrize("H", [1, 3, 5, 64])
def test_head_counts_that_are_not_powers_of_two(H):
    """The chunk-local kernel's work items (chunk pair x head) and the chain's
    grid (sequence x head) both map through H; odd head counts (and one head)
    run the ragged prefixes / lengths of the page_size 128 case; 64 heads make
    the token rows 16 KB wide."""
    ps, lens, prefixes = RAGGED[2]
    call, pool = _ragged_case(200 + H, ps, lens, prefixes, H=H)
    errs = Errors()
    prefill_paged_both(call, pool.cuda(), pool.numpy().copy(), errs)
    print("H=%d ragged case 2: %r" % (H, errs))


def test_split_prompt_matches_single_call_on_gpu():
    """Chunked prefill can split a prompt at any token: a 173 + 527 split on the
    GPU equals one 700-token GPU call within the state tolerance."""
    ps, H, L, split = 128, 2, 700, 173
    gen = torch.Generator().manual_seed(5)
    q, k, v, g, b = workloads.draw_tokens(gen, L, H, "cpu", 0.01)
    ids = torch.tensor([3, 8, 1, 12, 6, 10], dtype=torch.int32)
    full = workloads.PrefillCall(q, k, v, g, b, torch.tensor([0, L], dtype=torch.int32),
                                 *workloads.page_table([L], ids, ps, "cpu"), ps)
    part1 = workloads.PrefillCall(q[:split], k[:split], v[:split], g[:split], b[:split],
                                  torch.tensor([0, split], dtype=torch.int32),
                                  *workloads.page_table([split], ids, ps, "cpu"), ps)
    part2 = workloads.PrefillCall(q[split:], k[split:], v[split:], g[split:], b[split:],
                                  torch.tensor([0, L - split], dtype=torch.int32),
                                  *workloads.page_table([L], ids, ps, "cpu"), ps)
    base = workloads.sentinel_pool(16, H, "cpu")
    errs = Errors()
    p1, r1 = base.cuda(), base.numpy().copy()
    o_full, _ = prefill_paged_both(full, p1, r1, errs)
    p2, r2 = base.cuda(), base.numpy().copy()
    o_a, _ = prefill_paged_both(part1, p2, r2, errs)
    o_b, _ = prefill_paged_both(part2, p2, r2, errs)
    d = (torch.cat([o_a, o_b]).float() - o_full.float()).abs().max().item()
    assert d <= 1e-2
    e = (p2[ids.long()] - p1[ids.long()]).flatten(1).norm(dim=1) / p1[ids.long()].flatten(1).norm(dim=1)
    assert e.max().item() <= 1e-3


@pytest.mark.parametrize("pool_dtype", ["float32", "bfloat16"])
def test_general_slot_api_minus_one_rows(pool_dtype):
    """Read row -1 = zero state; write and checkpoint rows of -1 are skipped
    (fp32 and bf16 pools)."""
    H, N = 2, 64
    lens = [150, 90, 200]
    prefixes = [0, 30, 64]
    gen = torch.Generator().manual_seed(9)
    q, k, v, g, b = workloads.draw_tokens(gen, sum(lens), H, "cpu")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    pool = workloads.sentinel_pool(6, H, "cpu")
    workloads.fill_rows(pool, [1, 2], gen)
    si = torch.tensor([-1, 1, 2], dtype=torch.int32)
    osi = torch.tensor([3, -1, 4], dtype=torch.int32)
    P = torch.tensor(prefixes, dtype=torch.int32)
    counts = [(p + l) // N - p // N for p, l in zip(prefixes, lens)]
    ccs = torch.tensor(np.concatenate([[0], np.cumsum(counts)[:-1]]), dtype=torch.int32)
    cki = torch.arange(sum(counts), dtype=torch.int32)
    cki[1] = -1
    cki[-1] = -1
    ck = workloads.sentinel_pool(sum(counts), H, "cpu")
    dev = lambda t: t.cuda()
    if pool_dtype == "bfloat16":
        (pool_g, pool_o), (ck_g, ck_o) = bf16_pool_pair(pool), bf16_pool_pair(ck)
        pool_g, ck_g = pool_g.cuda(), ck_g.cuda()
    else:
        pool_g, ck_g = pool.cuda(), ck.cuda()
        pool_o, ck_o = pool.numpy().copy(), ck.numpy().copy()
    pb, cb = pool_g.clone(), ck_g.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = gdn.gdn_chunk_gated_delta_rule(dev(q), dev(k), dev(v), dev(g), dev(b), dev(cu), scale=SCALE,
                                       initial_state=pool_g, state_indices=dev(si), output_state=pool_g,
                                       output_state_indices=dev(osi), state_checkpoints=ck_g,
                                       checkpoint_state_indices=dev(cki), checkpoint_cu_starts=dev(ccs),
                                       prefix_lens=dev(P), checkpoint_every_n_tokens=N, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    o_ref, w_out, w_ck = oracle.chunk_gated_delta_rule(
        bf16_bits(q), bf16_bits(k), bf16_bits(v), f32(g), f32(b), i32(cu), SCALE, initial_state=pool_o,
        state_indices=i32(si), output_state=pool_o, output_state_indices=i32(osi), state_checkpoints=ck_o,
        checkpoint_state_indices=i32(cki), checkpoint_cu_starts=i32(ccs), prefix_lens=i32(P),
        checkpoint_every_n_tokens=N)
    errs = Errors()
    check_o(o, o_ref, errs)
    check_pool(pool_g, pb, pool_o, w_out, errs, "pool")
    check_pool(ck_g, cb, ck_o, w_ck, errs, "checkpoints")
    assert w_ck[1] == 0 and w_ck[-1] == 0


def test_device_validation_skips_bad_sequences():
    """With err_word, a page id outside the pool is reported and that sequence
    is skipped; the others still match the oracle."""
    call, pool = _ragged_case(7, 64, [100, 80], [10, 0])
    bad = call.page_indices.clone()
    n0 = int(call.page_indptr[1])
    bad[0] = 10_000                               # sequence 0 reads a page outside the pool
    call_bad = workloads.PrefillCall(call.q, call.k, call.v, call.g, call.beta, call.cu_seqlens, call.page_indptr,
                                     bad, call.last_page_len, call.page_size)
    pool_g = pool.cuda()
    before = pool_g.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda t: t.cuda()
    o = torch.zeros(call.q.shape[0], 2, 128, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_chunk_gated_delta_rule_paged(dev(call.q), dev(call.k), dev(call.v), dev(call.g), dev(call.beta),
                                         dev(call.cu_seqlens), pool_g, dev(bad), dev(call.page_indptr), 64,
                                         dev(call.last_page_len), scale=SCALE, o=o, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == (1 << 24) | 0
    # sequence 0 wrote nothing; sequence 1 matches the oracle
    assert bits_equal(pool_g[bad[:n0][bad[:n0] < pool.shape[0]].long()], before[bad[:n0][bad[:n0] < pool.shape[0]].long()])
    assert (o[:100] == 0).all()
    pool_o = pool.numpy().copy()
    o_ref, written = oracle.chunk_gated_delta_rule_paged(
        bf16_bits(call.q), bf16_bits(call.k), bf16_bits(call.v), f32(call.g), f32(call.beta), i32(call.cu_seqlens),
        pool_o, i32(call.page_indices), i32(call.page_indptr), 64, i32(call.last_page_len), SCALE,
        chains=np.array([[0, 0], [1, 1]], bool))
    errs = Errors()
    check_o(o[100:], o_ref[100:], errs)


@pytest.mark.parametrize("value", [1.0e6, 300.0])
@pytest.mark.parametrize("tensor", ["q", "k", "v"])
def test_value_beyond_fp16_range_is_reported(tensor, value):
    """The prefill's tensor-core operands are fp16: with err_word, a q, k or v
    element beyond +-65504 (here about 1e6, planted in sequence 1) is reported
    as GDN_DEVERR_RANGE for its sequence, while a large value inside the range
    whose products stay finite (300) is not.  (A k element near the limit,
    such as 60,000, makes k.k and the factors built from it overflow fp16; the
    stored states then turn non-finite, which is reported too.)  The other
    sequence still matches the oracle."""
    call, pool = _ragged_case(7, 64, [100, 80], [10, 0])
    t = getattr(call, tensor).clone()
    t[120, 1, 5] = value  # token 20 of sequence 1, head 1
    args = {n: getattr(call, n) for n in ("q", "k", "v")}
    args[tensor] = t
    call = workloads.PrefillCall(args["q"], args["k"], args["v"], call.g, call.beta, call.cu_seqlens,
                                 call.page_indptr, call.page_indices, call.last_page_len, call.page_size)
    pool_g = pool.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda x: x.cuda()
    o = gdn.gdn_chunk_gated_delta_rule_paged(dev(call.q), dev(call.k), dev(call.v), dev(call.g), dev(call.beta),
                                             dev(call.cu_seqlens), pool_g, dev(call.page_indices),
                                             dev(call.page_indptr), 64, dev(call.last_page_len), scale=SCALE,
                                             err_word=err)
    torch.cuda.synchronize()
    if value > 65504:
        assert int(err.item()) == (5 << 24) | 1
    else:
        assert int(err.item()) == 0
        assert torch.isfinite(o.float()).all()
    pool_o = pool.numpy().copy()
    o_ref, written = oracle.chunk_gated_delta_rule_paged(
        bf16_bits(call.q), bf16_bits(call.k), bf16_bits(call.v), f32(call.g), f32(call.beta), i32(call.cu_seqlens),
        pool_o, i32(call.page_indices), i32(call.page_indptr), 64, i32(call.last_page_len), SCALE,
        chains=np.array([[1, 1], [0, 0]], bool))
    errs = Errors()
    check_o(o[:100], o_ref[:100], errs)
    n0 = int(call.page_indptr[1])
    rows = call.page_indices[:n0].long()
    got = pool_g[rows.cuda()].cpu().numpy()
    from gpu_util import rel_fro_rows, S_TOL
    assert rel_fro_rows(got, pool_o[rows.numpy()]).max() <= S_TOL


def test_wait_that_runs_out_is_reported():
    """A bounded wait that runs out: with the test hook enabled, the state
    chain's first wait is on a barrier that nothing completes.  It gives up
    after about 1 ms, before any copy or tensor-core operation is in flight,
    records GDN_DEVERR_TIMEOUT and returns; the call then has written no output
    and no pool row, and the next call (hook disabled) runs normally on the
    same context and matches the oracle."""
    w = workloads.tiny("cpu")
    call = w.calls[0]
    dev = lambda t: t.cuda()
    pool_g = w.pool.cuda()
    before = pool_g.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.full((call.q.shape[0], w.H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_debug_set_wait_stall(True)
    try:
        gdn.gdn_chunk_gated_delta_rule_paged(dev(call.q), dev(call.k), dev(call.v), dev(call.g), dev(call.beta),
                                             dev(call.cu_seqlens), pool_g, dev(call.page_indices),
                                             dev(call.page_indptr), call.page_size, dev(call.last_page_len),
                                             scale=SCALE, o=o, err_word=err)
        torch.cuda.synchronize()
    finally:
        gdn.gdn_debug_set_wait_stall(False)
    assert int(err.item()) >> 24 == 15
    assert bits_equal(pool_g, before)
    assert torch.isnan(o.float()).all()
    errs = Errors()
    prefill_paged_both(call, pool_g, w.pool.numpy().copy(), errs)


def test_prefill_slots_refuse_a_last_page_len_outside_a_page():
    """The slot kernel skips (rows -1, prefix 0) the sequences the prefill
    kernels skip: a last page holding no token or more than page_size tokens;
    a valid neighbour keeps its rows (prefix 125 at page_size 64: read its
    page 1, write its page 1, first checkpoint entry 4 + 1)."""
    t = lambda x: torch.tensor(x, dtype=torch.int32, device="cuda")
    slots = gdn.gdn_paged_prefill_slots(t([0, 3, 5, 8]), t([0, 2, 4, 6]), t([5, 6, 7, 8, 9, 10]), t([0, 65, 64]),
                                        64)
    assert slots["state_indices"].tolist() == [-1, -1, 10]
    assert slots["output_state_indices"].tolist() == [-1, -1, 10]
    assert slots["prefix_lens"].tolist() == [0, 0, 125]
    assert slots["checkpoint_cu_starts"].tolist() == [0, 2, 5]


def test_empty_and_all_zero_length_batches():
    H = 2
    pool = workloads.sentinel_pool(4, H, "cuda")
    before = pool.clone()
    z = torch.zeros(0, H, 128, dtype=torch.bfloat16, device="cuda")
    zg = torch.zeros(0, H, device="cuda")
    ip = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    pi = torch.tensor([1, 3], dtype=torch.int32, device="cuda")
    lpl = torch.tensor([5, 64], dtype=torch.int32, device="cuda")
    cu = torch.zeros(3, dtype=torch.int32, device="cuda")
    gdn.gdn_chunk_gated_delta_rule_paged(z, z, z, zg, zg, cu, pool, pi, ip, 64, lpl, scale=SCALE)
    torch.cuda.synchronize()
    assert bits_equal(pool, before)
    slots = gdn.gdn_paged_prefill_slots(cu, ip, pi, lpl, 64)
    assert slots["output_state_indices"].tolist() == [-1, -1]
    assert slots["state_indices"].tolist() == [1, 3]


def test_decode_padding_and_scratch_rows():
    """A padded decode sequence on its own scratch page (last_page_len >= 2)
    updates only that page; explicit -1 write rows skip the store."""
    H = 2
    gen = torch.Generator().manual_seed(3)
    q, k, v, g, b = workloads.draw_tokens(gen, 3, H, "cpu")
    ip = torch.tensor([0, 2, 3, 4], dtype=torch.int32)
    pi = torch.tensor([5, 0, 2, 7], dtype=torch.int32)
    lpl = torch.tensor([1, 2, 9], dtype=torch.int32)
    call = workloads.DecodeCall(q, k, v, g, b, ip, pi, lpl, 64)
    pool = workloads.sentinel_pool(8, H, "cpu")
    workloads.fill_rows(pool, [5, 2, 7], gen)
    errs = Errors()
    decode_paged_both(call, pool.cuda(), pool.numpy().copy(), errs, use_slots=True)
    # explicit rows with a skipped write
    pool_g = pool.cuda()
    before = pool_g.clone()
    slots = {"initial_state_indices": torch.tensor([5, -1, 7], dtype=torch.int32, device="cuda"),
             "output_state_indices": torch.tensor([-1, 1, 7], dtype=torch.int32, device="cuda")}
    o = gdn.gdn_gated_delta_rule_decode_paged(q.cuda(), k.cuda(), v.cuda(), g.cuda(), b.cuda(), pool_g, pi.cuda(),
                                              ip.cuda(), lpl.cuda(), scale=SCALE, slots=slots)
    pool_o = pool.numpy().copy()
    o_ref, written = oracle.gated_delta_rule_decode(bf16_bits(q), bf16_bits(k), bf16_bits(v), f32(g), f32(b),
                                                    pool_o, [5, -1, 7], [-1, 1, 7], SCALE)
    torch.cuda.synchronize()
    check_o(o, o_ref, errs)
    check_pool(pool_g, before, pool_o, written, errs)
    print("decode padding: %r" % errs)
