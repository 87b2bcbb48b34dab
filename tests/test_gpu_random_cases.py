"""Seeded random batches against the oracle: page sizes, head counts,
lengths, prefixes, decay, pool dtype and with or without precomputed slots all
drawn at random, then a paged prefill followed by two decode steps on the same
pool ("flashinfer.gdn_paged", §Page table and the decode paragraph).  Each case
is small enough for the oracle and spans several chunks and a ragged tail."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_paged_gb300 import workloads
from conftest import i32
from gpu_util import Errors, bf16_pool_pair, decode_paged_both, prefill_paged_both

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(seed)
    ps = 64 * int(rng.integers(1, 9))
    H = int(rng.choice([1, 2, 3, 4]))
    S = int(rng.integers(1, 7))
    lens = [int(x) for x in rng.integers(0, 700, S)]
    prefixes = [int(x) for x in rng.integers(0, 1200, S)]
    for i in range(S):
        if rng.random() < 0.2:
            prefixes[i] = ps * int(rng.integers(0, 3))      # prefix on a page boundary
        if lens[i] + prefixes[i] == 0:
            prefixes[i] = 1
    decay = float(rng.choice([1.0, 0.01]))
    bf16 = bool(rng.random() < 0.4)
    use_slots = bool(rng.random() < 0.5)
    gen = torch.Generator().manual_seed(5000 + seed)
    ctx = [l + p for l, p in zip(lens, prefixes)]
    # each sequence's own pages, with room for two decode tokens after the prefill
    need = [-(-(c + 2) // ps) for c in ctx]
    ids = torch.randperm(sum(need) + 4, generator=gen).tolist()
    owned = [ids[sum(need[:i]):sum(need[:i + 1])] for i in range(S)]
    ip, pi, lpl = _table(ctx, owned, ps)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q, k, v, g, b = workloads.draw_tokens(gen, int(sum(lens)), H, "cpu", decay)
    pool = workloads.sentinel_pool(sum(need) + 4, H, "cpu")
    s = oracle.prefill_slots(i32(cu), i32(ip), i32(pi), i32(lpl), ps)
    workloads.fill_rows(pool, [r for r in s["state_indices"].tolist() if r >= 0], gen)
    call = workloads.PrefillCall(q, k, v, g, b, cu, ip, pi, lpl, ps)
    return dict(ps=ps, H=H, lens=lens, prefixes=prefixes, decay=decay, bf16=bf16, use_slots=use_slots, gen=gen,
                call=call, pool=pool, ctx=ctx, owned=owned)


def _table(ctx, owned, ps):
    """CSR page table of sequences with ctx[b] tokens on the first pages of owned[b]."""
    flat = sum((owned[b][: -(-c // ps)] for b, c in enumerate(ctx)), [])
    return workloads.page_table(ctx, torch.tensor(flat), ps, "cpu")


@pytest.mark.parametrize("seed", range(10))
def test_random_batch(seed):
    c = _case(seed)
    if c["bf16"]:
        pg, po = bf16_pool_pair(c["pool"])
        pg = pg.cuda()
    else:
        pg, po = c["pool"].cuda(), c["pool"].numpy().copy()
    errs = Errors()
    prefill_paged_both(c["call"], pg, po, errs, use_slots=c["use_slots"])
    # two decode steps for every sequence that holds at least one token
    ctx = list(c["ctx"])
    ps = c["ps"]
    for step in range(2):
        ctx = [x + 1 for x in ctx]
        keep = [i for i, x in enumerate(ctx) if x >= 2]
        if not keep:
            break
        # the prefill's pages in the same order, one more where the token opens a page
        ip, pi, lpl = _table([ctx[i] for i in keep], [c["owned"][i] for i in keep], ps)
        q, k, v, g, b = workloads.draw_tokens(c["gen"], len(keep), c["H"], "cpu", c["decay"])
        decode_paged_both(workloads.DecodeCall(q, k, v, g, b, ip, pi, lpl, ps), pg, po, errs,
                          use_slots=c["use_slots"])
    print("random case %d (ps=%d H=%d S=%d %s slots=%s decay=%g): %r" % (
        seed, ps, c["H"], len(c["lens"]), "bf16" if c["bf16"] else "fp32", c["use_slots"], c["decay"], errs))
