"""GPU parity of the general slot-argument call in its full generality
("flashinfer.gdn_paged", §Slot arguments of chunk_gated_delta_rule): int64
slot arrays, a padded pool row stride, and one selected checkpoint per
sequence given by -1 in every other entry; int64 entries outside the int32
range are reported and their sequence skipped."""
import numpy as np
import pytest
import torch

import gated_deltanet_paged_gb300 as gdn
import oracle
from gated_deltanet_paged_gb300 import workloads
from conftest import bf16_bits, f32, i32
from gpu_util import SCALE, Errors, bf16_pool_pair, bits_equal, check_o, check_pool

pytestmark = pytest.mark.gpu

GDN_DEVERR_INDEX_RANGE = 4
PAD = 40  # elements after each row: 160 B (fp32) or 80 B (bf16), rows stay 16-byte aligned


def _padded(pool):
    """[rows, H*V*K + PAD] fp32 with pool's rows in front and a per-row NaN
    pattern (0x7FA00000 | row) in the padding."""
    rows, n = pool.shape[0], pool[0].numel()
    full = torch.empty(rows, n + PAD, dtype=torch.float32)
    full[:, :n] = pool.reshape(rows, n)
    full[:, n:] = (torch.arange(rows, dtype=torch.int32) | 0x7FA00000).view(rows, 1).expand(rows, PAD).view(
        torch.float32)
    return full


def _gpu_and_oracle(full, pool_dtype):
    if pool_dtype == "bfloat16":
        g, o = bf16_pool_pair(full)
        return g.cuda(), o
    return full.cuda(), full.numpy().copy()


def _rows_view(full_g, H):
    n = H * 128 * 128
    return full_g[:, :n].view(full_g.shape[0], H, 128, 128)


def _ora_rows(full_o, H):
    n = H * 128 * 128
    return full_o[:, :n].reshape(full_o.shape[0], H, 128, 128)


def _case(seed, lens, prefixes, H, N):
    gen = torch.Generator().manual_seed(seed)
    q, k, v, g, b = workloads.draw_tokens(gen, sum(lens), H, "cpu")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    counts = [(p + l) // N - p // N for p, l in zip(prefixes, lens)]
    return gen, (q, k, v, g, b), cu, counts


@pytest.mark.parametrize("pool_dtype", ["float32", "bfloat16"])
def test_int64_slots_padded_rows_one_selected_checkpoint(pool_dtype):
    """int64 slot arrays, pools with padded rows (the padding never touched),
    and for each sequence one selected checkpoint (all other entries -1)."""
    H, N = 2, 64
    lens, prefixes = [300, 130, 200, 0], [0, 70, 64, 5]
    gen, (q, k, v, g, b), cu, counts = _case(13, lens, prefixes, H, N)
    pool = workloads.sentinel_pool(8, H, "cpu")
    workloads.fill_rows(pool, [1, 2, 6], gen)
    ck = workloads.sentinel_pool(10, H, "cpu")
    si = [-1, 1, 2, 6]
    osi = [3, 4, 5, 7]
    ccs = np.concatenate([[0], np.cumsum(counts)[:-1]]).tolist()
    cki = [-1] * sum(counts)
    for s, c in enumerate(counts):  # the middle checkpoint of each sequence, to row 2 s + 1
        if c:
            cki[ccs[s] + c // 2] = 2 * s + 1
    full_p, full_c = _padded(pool), _padded(ck)
    pg, po = _gpu_and_oracle(full_p, pool_dtype)
    cg, co = _gpu_and_oracle(full_c, pool_dtype)
    pb, cb = pg.clone(), cg.clone()
    i64 = lambda x: torch.tensor(x, dtype=torch.int64, device="cuda")
    dev = lambda t: t.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = gdn.gdn_chunk_gated_delta_rule(dev(q), dev(k), dev(v), dev(g), dev(b), dev(cu), scale=SCALE,
                                       initial_state=_rows_view(pg, H), state_indices=i64(si),
                                       output_state=_rows_view(pg, H), output_state_indices=i64(osi),
                                       state_checkpoints=_rows_view(cg, H), checkpoint_state_indices=i64(cki),
                                       checkpoint_cu_starts=i64(ccs), prefix_lens=i64(prefixes),
                                       checkpoint_every_n_tokens=N, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    # the oracle takes the same values as int32 and the padded rows as [rows, stride] arrays
    o_ref, w_out, w_ck = oracle.chunk_gated_delta_rule(
        bf16_bits(q), bf16_bits(k), bf16_bits(v), f32(g), f32(b), i32(cu), SCALE, initial_state=po,
        state_indices=np.array(si, np.int32), output_state=po, output_state_indices=np.array(osi, np.int32),
        state_checkpoints=co, checkpoint_state_indices=np.array(cki, np.int32),
        checkpoint_cu_starts=np.array(ccs, np.int32), prefix_lens=np.array(prefixes, np.int32),
        checkpoint_every_n_tokens=N)
    errs = Errors()
    check_o(o, o_ref, errs)
    check_pool(_rows_view(pg, H), _rows_view(pb, H), _ora_rows(po, H), w_out, errs, "pool")
    check_pool(_rows_view(cg, H), _rows_view(cb, H), _ora_rows(co, H), w_ck, errs, "checkpoints")
    n = H * 128 * 128
    assert bits_equal(pg[:, n:], pb[:, n:]) and bits_equal(cg[:, n:], cb[:, n:]), "row padding changed"
    assert sorted(np.flatnonzero(w_ck).tolist()) == [2 * s + 1 for s, c in enumerate(counts) if c]
    print("int64 slots, padded rows (%s): %r" % (pool_dtype, errs))


@pytest.mark.parametrize("bad", ["final_row", "checkpoint_row", "read_row", "checkpoint_start"])
def test_int64_entry_outside_int32_is_reported(bad):
    """One sequence with an int64 entry no int32 row can hold is skipped and
    reported; the others match the oracle and nothing else changes."""
    H, N = 2, 64
    lens, prefixes = [150, 200, 90], [10, 0, 64]
    gen, (q, k, v, g, b), cu, counts = _case(17, lens, prefixes, H, N)
    pool = workloads.sentinel_pool(6, H, "cpu")
    workloads.fill_rows(pool, [0, 1, 2], gen)
    ck = workloads.sentinel_pool(sum(counts), H, "cpu")
    si, osi = [0, 1, 2], [3, 4, 5]
    ccs = np.concatenate([[0], np.cumsum(counts)[:-1]]).tolist()
    cki = list(range(sum(counts)))
    si64, osi64, cki64, ccs64 = list(si), list(osi), list(cki), list(ccs)
    if bad == "final_row":
        osi64[1] = (1 << 32) + 4      # would wrap to row 4 as int32
    elif bad == "checkpoint_row":
        cki64[ccs[1] + 1] = -2
    elif bad == "read_row":
        si64[1] = -(1 << 33)
    else:
        ccs64[1] = 1 << 31
    pg, cg = pool.cuda(), ck.cuda()
    pb, cb = pg.clone(), cg.clone()
    po, co = pool.numpy().copy(), ck.numpy().copy()
    i64 = lambda x: torch.tensor(x, dtype=torch.int64, device="cuda")
    dev = lambda t: t.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.zeros(sum(lens), H, 128, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_chunk_gated_delta_rule(dev(q), dev(k), dev(v), dev(g), dev(b), dev(cu), scale=SCALE, initial_state=pg,
                                   state_indices=i64(si64), output_state=pg, output_state_indices=i64(osi64),
                                   state_checkpoints=cg, checkpoint_state_indices=i64(cki64),
                                   checkpoint_cu_starts=i64(ccs64), prefix_lens=i64(prefixes),
                                   checkpoint_every_n_tokens=N, o=o, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == (GDN_DEVERR_INDEX_RANGE << 24) | 1
    chains = np.ones((3, H), bool)
    chains[1] = False                 # the oracle leaves sequence 1 out entirely
    o_ref, w_out, w_ck = oracle.chunk_gated_delta_rule(
        bf16_bits(q), bf16_bits(k), bf16_bits(v), f32(g), f32(b), i32(cu), SCALE, initial_state=po,
        state_indices=np.array(si, np.int32), output_state=po, output_state_indices=np.array(osi, np.int32),
        state_checkpoints=co, checkpoint_state_indices=np.array(cki, np.int32),
        checkpoint_cu_starts=np.array(ccs, np.int32), prefix_lens=np.array(prefixes, np.int32),
        checkpoint_every_n_tokens=N, chains=chains)
    assert w_out[4] == 0 and not any(w_ck[ccs[1]:ccs[1] + counts[1]])
    errs = Errors()
    check_o(o, o_ref, errs)           # sequence 1: zeros on both sides
    check_pool(pg, pb, po, w_out, errs, "pool")
    check_pool(cg, cb, co, w_ck, errs, "checkpoints")
