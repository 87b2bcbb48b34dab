"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: worked
examples printed on the pages (tests/golden), closed forms of the recurrence,
brute force with explicit matrices, and cross-call invariants.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_paged_gb300 import workloads
from conftest import bf16_bits, bits_to_f64, ints, load_golden

SCALE = 128 ** -0.5


def draw(T, H, seed, decay=1.0, K=128, V=128):
    gen = torch.Generator().manual_seed(seed)
    q, k, v, g, b = workloads.draw_tokens(gen, T, H, "cpu", decay, K=K, V=V)
    return bf16_bits(q), bf16_bits(k), bf16_bits(v), g.numpy(), b.numpy()


def sentinel(rows, H, K=128, V=128):
    r = np.arange(rows, dtype=np.uint32).reshape(rows, 1, 1, 1)
    return np.ascontiguousarray(np.broadcast_to(r | 0x7FC00000, (rows, H, V, K))).view(np.float32).copy()


def rel_fro(a, b):
    return np.linalg.norm((a.astype(np.float64) - b.astype(np.float64)).ravel()) / max(
        np.linalg.norm(b.astype(np.float64).ravel()), 1e-300)


# ---------------------------------------------------------------------------
# CSR page tables (drill hint page, sections ①-③ and ⑥)
# ---------------------------------------------------------------------------

def test_csr_three_sequence_example():
    ex = load_golden("csr_worked_examples.txt")["three_sequences"]
    ps = int(ex["page_size"])
    table = np.array([ints(r) for r in ex["block_table"].split(";")])
    indptr, indices, last = oracle.block_table_to_csr(table, ints(ex["ctx"]), ps)
    assert indptr.tolist() == ints(ex["indptr"]).tolist()
    assert indices.tolist() == ints(ex["indices"]).tolist()
    assert last.tolist() == ints(ex["last_page_len"]).tolist()
    assert np.diff(indptr).tolist() == ints(ex["num_pages"]).tolist()
    back, ctx = oracle.csr_to_block_table(indptr, indices, last, ps, table.shape[1])
    assert back.tolist() == table.tolist()
    assert ctx.tolist() == ints(ex["ctx"]).tolist()


def test_csr_self_test_full_last_page():
    ex = load_golden("csr_worked_examples.txt")["self_test_1"]
    ps, ctx = int(ex["page_size"]), ints(ex["ctx"])
    table = np.arange(100, 100 + 4 * 8).reshape(4, 8)
    indptr, indices, last = oracle.block_table_to_csr(table, ctx, ps)
    assert indptr.tolist() == ints(ex["indptr"]).tolist()
    assert last.tolist() == ints(ex["last_page_len"]).tolist()
    assert [oracle.csr.pages_for(int(c), ps) for c in ctx] == ints(ex["num_pages"]).tolist()


def test_csr_zero_page_sequence_rejected():
    ex = load_golden("csr_worked_examples.txt")["self_test_2"]
    indptr = ints(ex["indptr"])
    with pytest.raises(ValueError, match="sequence %s owns no page" % ex["zero_page_sequence"]):
        oracle.csr_to_block_table(indptr, np.arange(5), np.array([1, 1, 1]), 16, 4)
    with pytest.raises(ValueError):
        oracle.prefill_slots([0, 1, 1, 2], indptr, np.arange(5), [1, 1, 1], 16)


# ---------------------------------------------------------------------------
# Page semantics ("flashinfer.gdn_paged": §Page table and the example)
# ---------------------------------------------------------------------------

def test_worked_prefill_example_rows():
    ex = load_golden("paged_prefill_2500.txt")[""]
    ps = int(ex["page_size"])
    s = oracle.prefill_slots(ints(ex["cu_seqlens"]), ints(ex["page_indptr"]), ints(ex["page_indices"]),
                             ints(ex["last_page_len"]), ps)
    assert s["state_indices"].tolist() == [int(ex["read_row"])]
    assert s["output_state_indices"].tolist() == ints(ex["written_rows"]).tolist()
    assert s["prefix_lens"].tolist() == [int(ex["total_tokens"]) - 452]

    H = 2
    q, k, v, g, b = draw(452, H, 7)
    pool = sentinel(16, H)
    pool[3] = np.random.default_rng(0).standard_normal((H, 128, 128)).astype(np.float32)
    before = pool.copy()
    o, written = oracle.chunk_gated_delta_rule_paged(
        q, k, v, g, b, ints(ex["cu_seqlens"]), pool, ints(ex["page_indices"]), ints(ex["page_indptr"]),
        ps, ints(ex["last_page_len"]), SCALE)
    assert np.flatnonzero(written).tolist() == ints(ex["written_rows"]).tolist()
    for r in range(16):
        if r in ints(ex["written_rows"]).tolist():
            assert np.isfinite(pool[r]).all()
        else:  # pages 7 and 3 (and every other row) keep their exact bits
            assert (pool[r].view(np.uint32) == before[r].view(np.uint32)).all(), r
    assert np.isfinite(o).all()


def test_state_after_table():
    """Page p holds the state after its last token: a 2500-token prefill from
    an empty prefix stores, in pages 7, 3, 12, the final states of prefills of
    the first 1024, 2048 and 2500 tokens."""
    ex = load_golden("paged_prefill_2500.txt")[""]
    ps, H = int(ex["page_size"]), 1
    q, k, v, g, b = draw(2500, H, 11)
    pool = sentinel(16, H)
    oracle.chunk_gated_delta_rule_paged(q, k, v, g, b, [0, 2500], pool, [7, 3, 12], [0, 3], ps, [452], SCALE)
    for item in ex["state_after"].split():
        page, count = (int(x) for x in item.split(":"))
        ref = sentinel(4, H)
        oracle.chunk_gated_delta_rule(q[:count], k[:count], v[:count], g[:count], b[:count], [0, count], SCALE,
                                      output_state=ref, output_state_indices=[2])
        assert (pool[page].view(np.uint32) == ref[2].view(np.uint32)).all(), page


@pytest.mark.parametrize("N", [64, 128])
def test_checkpoint_count_formula(N):
    """'Slot arguments': sequence i has (prefix + len) // N - prefix // N
    checkpoints, taken after new token n when (prefix + n) % N == 0."""
    H, K, V = 1, 1, 1
    lens = np.arange(0, 201)
    q, k, v, g, b = draw(int(lens.sum()), H, 3, K=K, V=V)
    cu = np.concatenate([[0], np.cumsum(lens)])
    slots_per_seq = 8
    for P in range(0, 201, 7):
        prefix = np.full(len(lens), P)
        cu_starts = np.arange(len(lens)) * slots_per_seq
        ck = np.zeros((len(lens) * slots_per_seq, H, V, K), np.float32)
        _, _, written = oracle.chunk_gated_delta_rule(
            q, k, v, g, b, cu, SCALE, state_checkpoints=ck,
            checkpoint_state_indices=np.arange(len(lens) * slots_per_seq), checkpoint_cu_starts=cu_starts,
            prefix_lens=prefix, checkpoint_every_n_tokens=N)
        got = written.reshape(len(lens), slots_per_seq).sum(1)
        assert got.tolist() == ((P + lens) // N - P // N).tolist()


def test_checkpoint_values_equal_truncated_runs():
    """The j-th checkpoint is the state after absolute position
    (P // N + j + 1) * N, i.e. the final state of a call that stops there."""
    H, N, P, L = 2, 64, 37, 300
    q, k, v, g, b = draw(L, H, 5)
    rng = np.random.default_rng(1)
    init = rng.standard_normal((1, H, 128, 128)).astype(np.float32)
    count = (P + L) // N - P // N
    ck = sentinel(count, H)
    oracle.chunk_gated_delta_rule(q, k, v, g, b, [0, L], SCALE, initial_state=init, state_indices=[0],
                                  state_checkpoints=ck, checkpoint_state_indices=np.arange(count),
                                  checkpoint_cu_starts=[0], prefix_lens=[P], checkpoint_every_n_tokens=N)
    for j in range(count):
        stop = (P // N + j + 1) * N - P
        fin = sentinel(1, H)
        oracle.chunk_gated_delta_rule(q[:stop], k[:stop], v[:stop], g[:stop], b[:stop], [0, stop], SCALE,
                                      initial_state=init, state_indices=[0], output_state=fin,
                                      output_state_indices=[0])
        assert (fin[0].view(np.uint32) == ck[j].view(np.uint32)).all(), j


def test_checkpoint_rows_minus_one_skip():
    H, N, L = 1, 64, 200
    q, k, v, g, b = draw(L, H, 9)
    ck = sentinel(3, H)
    before = ck.copy()
    _, _, written = oracle.chunk_gated_delta_rule(
        q, k, v, g, b, [0, L], SCALE, state_checkpoints=ck, checkpoint_state_indices=[-1, 1, -1],
        checkpoint_cu_starts=[0], prefix_lens=[0], checkpoint_every_n_tokens=N)
    assert written.tolist() == [0, 1, 0]
    assert (ck[0].view(np.uint32) == before[0].view(np.uint32)).all()
    assert (ck[2].view(np.uint32) == before[2].view(np.uint32)).all()


def test_padded_pool_rows():
    """Pools whose rows are padded (row stride > H*V*K, slot arguments
    paragraph: "the row stride may be padded") give the states of a dense pool
    in the first H*V*K elements of each row and never touch the padding."""
    H, N, P, L = 2, 64, 30, 170
    q, k, v, g, b = draw(L, H, 15)
    rng = np.random.default_rng(3)
    n, pad = H * 128 * 128, 24
    dense = sentinel(4, H)
    dense[1] = rng.standard_normal((H, 128, 128)).astype(np.float32)
    padded = np.empty((4, n + pad), np.float32)
    padded[:, :n] = dense.reshape(4, n)
    padded[:, n:] = (np.arange(4, dtype=np.uint32).reshape(4, 1) | 0x7FA00000).view(np.float32)
    before = padded.copy()
    kw = dict(state_indices=[1], output_state_indices=[3], checkpoint_state_indices=[0, 2, 0],
              checkpoint_cu_starts=[0], prefix_lens=[P], checkpoint_every_n_tokens=N)
    o1, w1, c1 = oracle.chunk_gated_delta_rule(q, k, v, g, b, [0, L], SCALE, initial_state=dense,
                                               output_state=dense, state_checkpoints=dense, **kw)
    o2, w2, c2 = oracle.chunk_gated_delta_rule(q, k, v, g, b, [0, L], SCALE, initial_state=padded,
                                               output_state=padded, state_checkpoints=padded, **kw)
    assert (o1 == o2).all() and (w1 == w2).all() and (c1 == c2).all()
    assert w1.tolist() == [0, 0, 0, 1] and c1.tolist() == [1, 0, 1, 0]
    assert (padded[:, :n].view(np.uint32) == dense.reshape(4, n).view(np.uint32)).all()
    assert (padded[:, n:].view(np.uint32) == before[:, n:].view(np.uint32)).all()
    with pytest.raises(ValueError):  # rows shorter than one state
        oracle.chunk_gated_delta_rule(q, k, v, g, b, [0, L], SCALE, initial_state=padded[:, : n - 8].copy(), **kw)


def _random_table(rng, S, ps, allow_empty=True):
    lens = rng.integers(0 if allow_empty else 1, 3 * ps, S)
    pre = rng.integers(0, 4 * ps, S)
    pre[(lens + pre) == 0] = 1
    ctx = lens + pre
    npages = [oracle.csr.pages_for(int(c), ps) for c in ctx]
    ids = rng.permutation(sum(npages) + 5)
    indptr, indices, last = oracle.csr_from_lengths(ctx, ids, ps)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return cu, indptr, indices, last, lens, pre


@pytest.mark.parametrize("ps", [64, 128, 1024])
def test_prefill_slots_match_position_arithmetic(ps):
    """Position-walking slots equal the division forms that follow from the
    page table: read = page (P-1)//ps, final = last page, first checkpoint page
    at index P//ps, prefix = ctx - len."""
    rng = np.random.default_rng(ps)
    for _ in range(20):
        cu, indptr, indices, last, lens, pre = _random_table(rng, 9, ps)
        s = oracle.prefill_slots(cu, indptr, indices, last, ps)
        for bb in range(len(lens)):
            P, L = int(pre[bb]), int(lens[bb])
            assert s["prefix_lens"][bb] == P
            assert s["state_indices"][bb] == (indices[indptr[bb] + (P - 1) // ps] if P > 0 else -1)
            assert s["output_state_indices"][bb] == (indices[indptr[bb + 1] - 1] if L > 0 else -1)
            assert s["checkpoint_cu_starts"][bb] == indptr[bb] + P // ps


def test_decode_slots_rule():
    """Decode paragraph: lpl == 1 reads the previous page and writes the new
    one; otherwise the last page is read and written in place."""
    rng = np.random.default_rng(2)
    ps = 64
    ctx = rng.integers(2, 10 * ps, 200)
    ctx[::4] = rng.integers(1, 9, 50) * ps + 1
    indptr, indices, last = oracle.csr_from_lengths(ctx, rng.permutation(5000), ps)
    s = oracle.decode_slots(indptr, indices, last, ps)
    for bb in range(len(ctx)):
        lastp = indices[indptr[bb + 1] - 1]
        assert s["output_state_indices"][bb] == lastp
        if last[bb] == 1:
            assert s["initial_state_indices"][bb] == indices[indptr[bb + 1] - 2]
        else:
            assert s["initial_state_indices"][bb] == lastp
    # decode rows are the prefill rows of a one-token call
    p = oracle.prefill_slots(np.arange(len(ctx) + 1), indptr, indices, last, ps)
    assert (p["state_indices"] == s["initial_state_indices"]).all()
    assert (p["output_state_indices"] == s["output_state_indices"]).all()


@pytest.mark.parametrize("lpl", [0, -3, 65, 1000])
def test_last_page_len_outside_a_page_is_rejected(lpl):
    """Page table section: the last page of a sequence holds between one token
    and a full page, so a last_page_len outside 1..page_size names no token
    position and both slot derivations refuse the table (rather than walk past
    the sequence's page list)."""
    indptr = np.array([0, 2], np.int32)
    indices = np.array([4, 7], np.int32)
    last = np.array([lpl], np.int32)
    with pytest.raises(ValueError):
        oracle.prefill_slots(np.array([0, 1], np.int32), indptr, indices, last, 64)
    with pytest.raises(ValueError):
        oracle.decode_slots(indptr, indices, last, 64)
    # the bounds themselves are valid
    for ok in (1, 64):
        s = oracle.prefill_slots(np.array([0, 1], np.int32), indptr, indices, np.array([ok], np.int32), 64)
        assert s["output_state_indices"].tolist() == [7]


def test_zero_length_sequences_leave_pool_unchanged():
    """A zero-length sequence (and a padded one: no new tokens, one scratch
    page) writes nothing; its neighbours are unaffected."""
    ps, H = 64, 2
    lens = [50, 0, 70, 0]
    pre = [10, 100, 0, 1]
    ctx = [a + b for a, b in zip(lens, pre)]
    indptr, indices, last = oracle.csr_from_lengths(ctx, np.random.default_rng(3).permutation(12), ps)
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, b = draw(sum(lens), H, 4)
    pool = sentinel(12, H)
    for r in indices:
        pool[r] = np.random.default_rng(int(r)).standard_normal((H, 128, 128)).astype(np.float32)
    before = pool.copy()
    o, written = oracle.chunk_gated_delta_rule_paged(q, k, v, g, b, cu, pool, indices, indptr, ps, last, SCALE)
    own = lambda s: set(indices[indptr[s]:indptr[s + 1]].tolist())
    assert not (set(np.flatnonzero(written).tolist()) & (own(1) | own(3)))
    for r in own(1) | own(3):
        assert (pool[r].view(np.uint32) == before[r].view(np.uint32)).all()
    # the batch with the empty sequences removed gives the same result
    keep = [0, 2]
    ip2 = np.concatenate([[0], np.cumsum([indptr[s + 1] - indptr[s] for s in keep])])
    ix2 = np.concatenate([indices[indptr[s]:indptr[s + 1]] for s in keep])
    pool2 = before.copy()
    o2, _ = oracle.chunk_gated_delta_rule_paged(q, k, v, g, b, [0, 50, 120], pool2, ix2, ip2, ps,
                                                last[keep], SCALE)
    assert (pool2.view(np.uint32) == pool.view(np.uint32)).all()
    assert (o2 == o).all()


# ---------------------------------------------------------------------------
# The recurrence: brute force and closed forms
# ---------------------------------------------------------------------------

def test_brute_force_householder_form():
    """S_t = S_{t-1} e_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T with explicit
    matrices, on a non-square state (K=5, V=3) so a transposed operand shows."""
    K, V, T, H = 5, 3, 9, 2
    q, k, v, g, b = draw(T, H, 21, K=K, V=V)
    rng = np.random.default_rng(5)
    init = rng.standard_normal((1, H, V, K)).astype(np.float32)
    out = np.zeros((1, H, V, K), np.float32)
    o, _, _ = oracle.chunk_gated_delta_rule(q, k, v, g, b, [0, T], 0.3, initial_state=init,
                                            state_indices=[0], output_state=out, output_state_indices=[0])
    qd, kd, vd = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    for h in range(H):
        S = init[0, h].astype(np.float64)
        for t in range(T):
            e = np.exp(np.float64(g[t, h]))
            kk = kd[t, h][:, None]
            S = S @ (e * (np.eye(K) - np.float64(b[t, h]) * (kk @ kk.T))) + np.float64(b[t, h]) * np.outer(vd[t, h], kd[t, h])
            np.testing.assert_allclose(o[t, h], 0.3 * S @ qd[t, h], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(out[0, h], S.astype(np.float32), rtol=1e-6, atol=1e-7)


def test_scalar_state_by_hand():
    """K = V = 1: s' = e s + beta (v - e s k) k, o = scale s' q, worked by hand
    for exactly representable inputs: s=2, g=0 (e=1), beta=0.5, k=1, v=4,
    q=0.5 -> s' = 2 + 0.5 * (4 - 2) = 3, o = 0.25 * 3 * 0.5 = 0.375."""
    bits = lambda x: np.array([[[x]]], np.float32).view(np.uint32).astype(np.uint32) >> 16
    q, k, v = (bits(x).astype(np.uint16) for x in (0.5, 1.0, 4.0))
    init = np.array([[[[2.0]]]], np.float32)
    out = np.zeros_like(init)
    o, _, _ = oracle.chunk_gated_delta_rule(q, k, v, np.zeros((1, 1), np.float32), np.full((1, 1), 0.5, np.float32),
                                            [0, 1], 0.25, initial_state=init, state_indices=[0],
                                            output_state=out, output_state_indices=[0])
    assert out[0, 0, 0, 0] == 3.0
    assert o[0, 0, 0] == 0.375


def test_beta_zero_is_pure_decay():
    """beta = 0: S_T = exp(sum g) S_0 and o_t = scale exp(G_t) S_0 q_t."""
    T, H = 40, 2
    q, k, v, g, _ = draw(T, H, 31)
    b = np.zeros((T, H), np.float32)
    rng = np.random.default_rng(6)
    init = rng.standard_normal((1, H, 128, 128)).astype(np.float32)
    out = np.zeros_like(init)
    o, _, _ = oracle.chunk_gated_delta_rule(q, k, v, g, b, [0, T], SCALE, initial_state=init, state_indices=[0],
                                            output_state=out, output_state_indices=[0])
    G = np.cumsum(g.astype(np.float64), axis=0)
    for h in range(H):
        S0 = init[0, h].astype(np.float64)
        for t in range(T):
            np.testing.assert_allclose(o[t, h], SCALE * np.exp(G[t, h]) * (S0 @ bits_to_f64(q)[t, h]), rtol=1e-10,
                                       atol=1e-14)
        np.testing.assert_allclose(out[0, h], (np.exp(G[-1, h]) * S0).astype(np.float32), rtol=2e-7, atol=1e-30)


def test_unit_key_overwrites_column():
    """g = 0, beta = 1, k = e_i: the delta rule replaces column i of S by v and
    leaves the rest (exact with small-integer values)."""
    K = V = 128
    H, T = 1, 4
    rng = np.random.default_rng(7)
    init = rng.integers(-8, 8, (1, H, V, K)).astype(np.float32)
    cols = [3, 77, 3, 127]
    kk = np.zeros((T, H, K), np.float32)
    for t, c in enumerate(cols):
        kk[t, 0, c] = 1.0
    vv = rng.integers(-5, 5, (T, H, V)).astype(np.float32)
    qq = rng.integers(-2, 3, (T, H, K)).astype(np.float32)
    to_bits = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)
    out = np.zeros_like(init)
    o, _, _ = oracle.chunk_gated_delta_rule(to_bits(qq), to_bits(kk), to_bits(vv), np.zeros((T, H), np.float32),
                                            np.ones((T, H), np.float32), [0, T], 1.0, initial_state=init,
                                            state_indices=[0], output_state=out, output_state_indices=[0])
    S = init[0, 0].astype(np.float64).copy()
    for t, c in enumerate(cols):
        S[:, c] = vv[t, 0]
        assert (o[t, 0] == S @ qq[t, 0]).all()
    assert (out[0, 0] == S).all()


def test_full_forgetting_stores_outer_product():
    """exp(g) underflowing to 0 (g = -1e4) forgets S: S = beta v k^T."""
    T, H = 5, 2
    q, k, v, _, b = draw(T, H, 41)
    g = np.full((T, H), -1e4, np.float32)
    init = np.random.default_rng(8).standard_normal((1, H, 128, 128)).astype(np.float32)
    out = np.zeros_like(init)
    oracle.chunk_gated_delta_rule(q, k, v, g, b, [0, T], SCALE, initial_state=init, state_indices=[0],
                                  output_state=out, output_state_indices=[0])
    for h in range(H):
        ref = np.outer(np.float64(b[-1, h]) * bits_to_f64(v)[-1, h], bits_to_f64(k)[-1, h])
        assert (out[0, h] == ref.astype(np.float32)).all()


def test_zero_state_is_literal_zeros():
    """A read row of -1 starts from zeros; a NaN-filled pool is never read."""
    T, H = 20, 2
    q, k, v, g, b = draw(T, H, 51)
    pool = sentinel(3, H)
    o1, _, _ = oracle.chunk_gated_delta_rule(q, k, v, g, b, [0, T], SCALE, initial_state=pool, state_indices=[-1],
                                             output_state=pool, output_state_indices=[2])
    zeros = np.zeros((1, H, 128, 128), np.float32)
    out = np.zeros_like(zeros)
    o2, _, _ = oracle.chunk_gated_delta_rule(q, k, v, g, b, [0, T], SCALE, initial_state=zeros, state_indices=[0],
                                             output_state=out, output_state_indices=[0])
    assert np.isfinite(o1).all() and (o1 == o2).all()
    assert (pool[2] == out[0]).all()


# ---------------------------------------------------------------------------
# Cross-call invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("decay", [1.0, 0.01])
def test_resume_from_page_equals_recompute(decay):
    """A hit that resumes from the last shared full page equals the cold run
    (gaudi-cookbook gdn-prefix-cache, §Verify: cold and hit agree)."""
    ps, H, L = 128, 2, 700
    q, k, v, g, b = draw(L, H, 61, decay)
    ids = np.array([9, 2, 14, 5, 0, 11], np.int32)
    ip = np.array([0, 6], np.int32)
    last = np.array([L - 5 * ps], np.int32)
    cold = sentinel(16, H)
    o_cold, _ = oracle.chunk_gated_delta_rule_paged(q, k, v, g, b, [0, L], cold, ids, ip, ps, last, SCALE)
    for hit_pages in (1, 3, 5):
        P = hit_pages * ps
        hot = sentinel(16, H)
        hot[ids[:hit_pages]] = cold[ids[:hit_pages]]
        o_hot, _ = oracle.chunk_gated_delta_rule_paged(q[P:], k[P:], v[P:], g[P:], b[P:], [0, L - P], hot, ids, ip,
                                                       ps, last, SCALE)
        np.testing.assert_allclose(o_hot, o_cold[P:], rtol=1e-5, atol=1e-6)
        for r in ids[hit_pages:]:
            assert rel_fro(hot[r], cold[r]) < 1e-6


@pytest.mark.parametrize("decay", [1.0, 0.01])
@pytest.mark.parametrize("split", [1, 63, 64, 173, 256, 699])
def test_split_prompt_at_any_token(split, decay):
    """Chunked prefill can split a prompt at any token: two calls (the second
    continuing a partial page in place) equal one call."""
    ps, H, L = 128, 2, 700
    q, k, v, g, b = draw(L, H, 71, decay)
    ids = np.array([3, 8, 1, 12, 6, 10], np.int32)
    one = sentinel(16, H)
    o_one, _ = oracle.chunk_gated_delta_rule_paged(q, k, v, g, b, [0, L], one, ids, [0, 6], ps, [L - 5 * ps], SCALE)
    two = sentinel(16, H)
    n1 = oracle.csr.pages_for(split, ps)
    o_a, _ = oracle.chunk_gated_delta_rule_paged(q[:split], k[:split], v[:split], g[:split], b[:split], [0, split],
                                                 two, ids[:n1], [0, n1], ps, [split - (n1 - 1) * ps], SCALE)
    o_b, _ = oracle.chunk_gated_delta_rule_paged(q[split:], k[split:], v[split:], g[split:], b[split:],
                                                 [0, L - split], two, ids, [0, 6], ps, [L - 5 * ps], SCALE)
    np.testing.assert_allclose(np.concatenate([o_a, o_b]), o_one, rtol=1e-5, atol=1e-6)
    for r in ids:
        assert rel_fro(two[r], one[r]) < 1e-6


@pytest.mark.parametrize("ctx", [2, 65, 100, 129])
def test_decode_equals_one_token_prefill(ctx):
    ps, H = 64, 2
    q, k, v, g, b = draw(1, H, 81)
    ids = np.array([4, 1, 7], np.int32)
    n = oracle.csr.pages_for(ctx, ps)
    ip, last = np.array([0, n], np.int32), np.array([ctx - (n - 1) * ps], np.int32)
    base = sentinel(8, H)
    for r in ids[:n]:
        base[r] = np.random.default_rng(int(r)).standard_normal((H, 128, 128)).astype(np.float32)
    p1, p2 = base.copy(), base.copy()
    o_dec, w1 = oracle.gated_delta_rule_decode_paged(q, k, v, g, b, p1, ids[:n], ip, last, ps, SCALE)
    o_pre, w2 = oracle.chunk_gated_delta_rule_paged(q, k, v, g, b, [0, 1], p2, ids[:n], ip, ps, last, SCALE)
    assert (o_dec.reshape(-1) == o_pre.reshape(-1)).all()
    assert (w1 == w2).all() and (p1.view(np.uint32) == p2.view(np.uint32)).all()


def test_heads_are_independent():
    T, H = 90, 3
    q, k, v, g, b = draw(T, H, 91)
    perm = [2, 0, 1]
    init = np.random.default_rng(9).standard_normal((1, H, 128, 128)).astype(np.float32)
    out1, out2 = np.zeros_like(init), np.zeros_like(init)
    o1, _, _ = oracle.chunk_gated_delta_rule(q, k, v, g, b, [0, T], SCALE, initial_state=init, state_indices=[0],
                                             output_state=out1, output_state_indices=[0])
    o2, _, _ = oracle.chunk_gated_delta_rule(q[:, perm], k[:, perm], v[:, perm], g[:, perm], b[:, perm], [0, T],
                                             SCALE, initial_state=np.ascontiguousarray(init[:, perm]),
                                             state_indices=[0], output_state=out2, output_state_indices=[0])
    assert (o2 == o1[:, perm]).all()
    assert (out2 == out1[:, perm]).all()


def test_value_rows_are_independent():
    """Row v of S and component v of every output depend on v only through
    v_t[v] and row v of the initial state (the recurrence is applied row by
    row): changing the values and initial state of row 5 changes row 5 of the
    state and component 5 of the outputs, bit for bit nothing else.  A
    transposed state or a q / k swap breaks this."""
    T, H = 70, 2
    q, k, v, g, b = draw(T, H, 93)
    rng = np.random.default_rng(19)
    init = rng.standard_normal((1, H, 128, 128)).astype(np.float32)
    init2 = init.copy()
    init2[:, :, 5, :] = rng.standard_normal((H, 128)).astype(np.float32)
    v2 = v.copy()
    v2[:, :, 5] = bf16_bits(torch.randn(T, H, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16))
    outs = []
    for vv, ii in ((v, init), (v2, init2)):
        out = np.zeros_like(init)
        o, _, _ = oracle.chunk_gated_delta_rule(q, k, vv, g, b, [0, T], SCALE, initial_state=ii, state_indices=[0],
                                                output_state=out, output_state_indices=[0])
        outs.append((o, out))
    (o1, s1), (o2, s2) = outs
    others = [i for i in range(128) if i != 5]
    assert (o1[:, :, others] == o2[:, :, others]).all() and (s1[:, :, others] == s2[:, :, others]).all()
    assert (o1[:, :, 5] != o2[:, :, 5]).any() and (s1[:, :, 5] != s2[:, :, 5]).any()


def test_rows_outside_write_set_keep_their_bits():
    """NaN-poisoned pool after a mixed batch: exactly the rows the oracle
    reports as written changed; every other row is bit-identical."""
    rng = np.random.default_rng(10)
    ps, H = 64, 2
    cu, indptr, indices, last, lens, pre = _random_table(rng, 6, ps)
    q, k, v, g, b = draw(int(lens.sum()), H, 101)
    rows = int(indices.max()) + 4
    pool = sentinel(rows, H)
    s = oracle.prefill_slots(cu, indptr, indices, last, ps)
    for r in s["state_indices"]:
        if r >= 0:
            pool[r] = rng.standard_normal((H, 128, 128)).astype(np.float32)
    before = pool.copy()
    _, written = oracle.chunk_gated_delta_rule_paged(q, k, v, g, b, cu, pool, indices, indptr, ps, last, SCALE)
    changed = (pool.view(np.uint32) != before.view(np.uint32)).reshape(rows, -1).any(1)
    assert (changed == written.astype(bool)).all()
    expect = set()
    for bb in range(len(lens)):
        P, L = int(pre[bb]), int(lens[bb])
        for j in range(P // ps, (P + L + ps - 1) // ps if L else P // ps):
            expect.add(int(indices[indptr[bb] + j]))
    assert set(np.flatnonzero(written).tolist()) == expect


# ---------------------------------------------------------------------------
# bf16 state pools: states rounded to the nearest bf16 value, ties to even.
# ---------------------------------------------------------------------------

def _bf16_from_bits(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def test_bf16_rounding_by_hand():
    """The store rounding, on values whose nearest bf16 (8 significant bits,
    ties to even) is worked out by hand: ties go to the even significand,
    anything past a tie goes up, the fp32 exponent range with a 2^-133 quantum
    below 2^-126, overflow to infinity past the largest finite value."""
    cases = [
        (1.0, 0x3F80),
        (1 + 2.0 ** -8, 0x3F80),                 # tie between 1 and 1 + 2^-7: even is 1
        (1 + 3 * 2.0 ** -8, 0x3F82),             # tie between 1 + 2^-7 and 1 + 2^-6: even is the latter
        (1 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),    # just past the tie
        (-(1 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (1.5 * 2.0 ** -130, 0x000C),             # 12 quanta of 2^-133
        (2.0 ** -134, 0x0000),                   # half a quantum: tie to the even 0
        (3 * 2.0 ** -134, 0x0002),               # 1.5 quanta: tie to 2
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),  # the largest finite bf16
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),  # its tie with 2^128 rounds to even: infinity
        (float("inf"), 0x7F80),
    ]
    for x, want in cases:
        assert oracle.double_to_bf16_bits(x) == want, (x, hex(oracle.double_to_bf16_bits(x)), hex(want))


def test_bf16_pool_keeps_a_state_it_does_not_change():
    """beta = 0 and g = 0 leave S as it is, so a bf16 pool row read, updated and
    written back keeps its bits (bf16 -> fp64 -> bf16 is exact), in place and to
    another row, and o = scale S q from those values."""
    H, K, V = 2, 128, 128
    rng = np.random.default_rng(11)
    pool = (rng.standard_normal((3, H, V, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q, k, v, _, _ = draw(1, H, 12)
    zeros = np.zeros((1, H), np.float32)
    before = pool.copy()
    o, written = oracle.gated_delta_rule_decode(q, k, v, zeros, zeros, pool, [0], [2], SCALE)
    assert written.tolist() == [0, 0, 1]
    assert (pool[2] == before[0]).all() and (pool[:2] == before[:2]).all()
    S = _bf16_from_bits(before[0]).astype(np.float64)
    qd = bits_to_f64(q[0])
    for h in range(H):
        assert np.allclose(o[0, h], SCALE * S[h] @ qd[h], rtol=0, atol=1e-12)


def test_bf16_pool_stores_the_nearest_value():
    """g = 0, beta = 1, k = e_i writes v into column i; with v = 1 + 2^-8 and
    1 + 3 2^-8 (bf16 ties) the bf16 pool holds 1 and 1 + 2^-6, while an fp32
    pool holds the values exactly."""
    K = V = 128
    H, T = 1, 1
    kk = np.zeros((T, H, K), np.float32)
    kk[0, 0, 5] = 1.0
    vv = np.zeros((T, H, V), np.float32)
    vv[0, 0, 0::2] = 1 + 2.0 ** -8
    vv[0, 0, 1::2] = 1 + 3 * 2.0 ** -8
    to_bits = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)
    # v is passed as bf16 bits; 1 + 2^-8 is not a bf16 value, so feed it through
    # the state instead: start from S with column 5 equal to those values and
    # apply beta = 0 (S unchanged) into a bf16 pool.
    S0 = np.zeros((1, H, V, K), np.float32)
    S0[0, 0, :, 5] = vv[0, 0]
    f32_pool = S0.copy()
    bf_pool = np.zeros((1, H, V, K), np.uint16)
    zeros = np.zeros((T, H), np.float32)
    q = to_bits(np.zeros((T, H, K), np.float32))
    oracle.chunk_gated_delta_rule(q, to_bits(kk), q[:, :, :V], zeros, zeros, [0, T], SCALE,
                                  initial_state=f32_pool, state_indices=[0], output_state=f32_pool,
                                  output_state_indices=[0])
    assert (f32_pool[0, 0, :, 5] == vv[0, 0]).all()
    # same state, bf16 pool as the output (the read pool is the fp32 one)
    with pytest.raises(TypeError):
        oracle.chunk_gated_delta_rule(q, to_bits(kk), q[:, :, :V], zeros, zeros, [0, T], SCALE,
                                      initial_state=S0, state_indices=[0], output_state=bf_pool,
                                      output_state_indices=[0])
    # a bf16 pool both read (zero row -1) and written: column 5 = beta v with
    # beta = 1 + 2^-8 and v = 1 gives 1 + 2^-8 -> 1 (tie, even), with beta =
    # 1 + 3 2^-8 it gives 1 + 2^-6
    for beta, want in ((1 + 2.0 ** -8, 0x3F80), (1 + 3 * 2.0 ** -8, 0x3F82)):
        bf_pool[:] = 0
        ones_v = to_bits(np.ones((T, H, V), np.float32))
        oracle.chunk_gated_delta_rule(q, to_bits(kk), ones_v, zeros, np.full((T, H), beta, np.float32), [0, T],
                                      SCALE, initial_state=bf_pool, state_indices=[-1], output_state=bf_pool,
                                      output_state_indices=[0])
        assert (bf_pool[0, 0, :, 5] == want).all()
        assert (np.delete(bf_pool[0, 0], 5, axis=1) == 0).all()


def test_row_copies_keep_every_bit():
    """The row utilities' reference is their definition: rows move whole and bit
    for bit (NaN payloads, -0.0 and bf16 bit patterns included), -1 skips, a row
    outside the pool skips, and pairs run in order."""
    pool = np.arange(6 * 8, dtype=np.uint32).reshape(6, 8) | np.uint32(0x7FC00000)
    pool[1, 0] = np.float32(-0.0).view(np.uint32)
    before = pool.copy()
    oracle.pool_copy_rows(pool, [1, -1, 2, 9], [4, 3, 5, 0])
    assert (pool[4] == before[1]).all() and (pool[5] == before[2]).all()
    assert (pool[[0, 1, 2, 3]] == before[[0, 1, 2, 3]]).all()
    bf = np.arange(4 * 4, dtype=np.uint16).reshape(4, 4) | np.uint16(0x7F80)
    bref = bf.copy()
    oracle.pool_zero_rows(bf, [2, -1, 7])
    assert (bf[2] == 0).all() and (bf[[0, 1, 3]] == bref[[0, 1, 3]]).all()
