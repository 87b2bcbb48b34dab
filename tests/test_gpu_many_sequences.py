"""Large batches against the oracle: thousands of short prefill sequences
(many chains in several waves, zero-length sequences, prefixes inside and at
the ends of pages) and a decode batch of 8,192 sequences, on fp32 and bf16
pools ("flashinfer.gdn_paged", §Page table and the decode paragraph)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_paged_gb300 import workloads
from conftest import i32
from gpu_util import Errors, bf16_pool_pair, decode_paged_both, prefill_paged_both

pytestmark = pytest.mark.gpu


def _pools(pool, pool_dtype):
    if pool_dtype == "bfloat16":
        g, o = bf16_pool_pair(pool)
        return g.cuda(), o
    return pool.cuda(), pool.numpy().copy()


def _short_sequences_case(S, H, ps, seed, use_slots):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 81, S)
    lens[rng.random(S) < 0.1] = 0
    prefixes = rng.integers(0, 301, S)
    edge = rng.random(S) < 0.1
    prefixes[edge] = ps * rng.integers(0, 3, int(edge.sum()))  # prefixes that end a page (or are empty)
    prefixes[(lens + prefixes) == 0] = 1
    gen = torch.Generator().manual_seed(seed + 1)
    ctx = (lens + prefixes).tolist()
    npages = sum(-(-c // ps) for c in ctx)
    ids = torch.randperm(npages + 3, generator=gen)
    ip, pi, lpl = workloads.page_table(ctx, ids, ps, "cpu")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q, k, v, g, b = workloads.draw_tokens(gen, int(lens.sum()), H, "cpu")
    pool = workloads.sentinel_pool(npages + 3, H, "cpu")
    s = oracle.prefill_slots(i32(cu), i32(ip), i32(pi), i32(lpl), ps)
    workloads.fill_rows(pool, [r for r in s["state_indices"].tolist() if r >= 0], gen)
    errs = Errors()
    prefill_paged_both(workloads.PrefillCall(q, k, v, g, b, cu, ip, pi, lpl, ps), pool.cuda(), pool.numpy().copy(),
                       errs, use_slots=use_slots)
    print("%d sequences, %d tokens: %r" % (S, int(lens.sum()), errs))


@pytest.mark.parametrize("use_slots", [False, True])
def test_two_thousand_short_sequences(use_slots):
    _short_sequences_case(2000, 2, 128, 71, use_slots)


def test_more_than_4096_sequences():
    """4,500 sequences: the state chain then takes sequence b = CTA / H in batch
    order (below 4,096 sequences it orders them by length first)."""
    _short_sequences_case(4500, 1, 64, 81, False)


@pytest.mark.parametrize("pool_dtype", ["float32", "bfloat16"])
def test_decode_batch_of_8192(pool_dtype):
    st = workloads.decode_layers("cpu", L=1, B=8192, H=1, page_size=64, max_ctx=300, seed=73, sentinel=True)
    pg, po = _pools(st.pools[0], pool_dtype)
    errs = Errors()
    decode_paged_both(st.calls[0], pg, po, errs, use_slots=pool_dtype == "float32")
    print("decode B=8192 (%s): %r" % (pool_dtype, errs))
