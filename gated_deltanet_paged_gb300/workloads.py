"""Seeded synthetic workloads for paged GDN prefill and decode.

This module only draws inputs: token counts, page tables, q/k/v/g/beta and
initial pool contents.  It holds none of the method's arithmetic and is the one
piece that the CUDA path's callers (tests, bench, smoke) and the oracle's
callers share.

Input recipe (the same for every workload):
  - q, k: N(0, 1) fp32, L2-normalised per (token, head), rounded to bf16;
  - v: N(0, 1) rounded to bf16;
  - g: -softplus(N(0, 1)) fp32 (times ``decay_scale``; 0.01 gives slow decay);
  - beta: sigmoid(N(0, 1)) fp32;
  - pool rows owned by a sequence: N(0, 1) fp32; every other row holds a NaN
    whose payload is its row number, so a stray read or write shows up.
Draw order: lengths -> page permutation -> q, k, v, g, beta (per call, in call
order) -> pool.  One torch.Generator on ``device`` seeded with 1234 + index;
generation on "cuda" is for the large workloads, whose oracle inputs are
copied back to the host.

Page tables follow "flashinfer.gdn_paged" §Page table: a sequence with ctx
tokens after the call owns ceil(ctx / page_size) pages (ids from a random
permutation, in any order) and last_page_len = ctx - (pages - 1) * page_size.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

K_DIM = 128
V_DIM = 128


@dataclass
class PrefillCall:
    """One prefill call.  q, k: bf16 [T, H, K]; v: bf16 [T, H, V]; g, beta:
    fp32 [T, H]; page table int32 (page_indptr [S+1], page_indices,
    last_page_len [S]); cu_seqlens int32 [S+1]."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    cu_seqlens: torch.Tensor
    page_indptr: torch.Tensor
    page_indices: torch.Tensor
    last_page_len: torch.Tensor
    page_size: int
    kind: str = "prefill"


@dataclass
class DecodeCall:
    """One decode step.  q, k: bf16 [B, H, K]; v: bf16 [B, H, V]; g, beta:
    fp32 [B, H]; page table after the decoded token."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    page_indptr: torch.Tensor
    page_indices: torch.Tensor
    last_page_len: torch.Tensor
    page_size: int
    kind: str = "decode"


@dataclass
class Workload:
    name: str
    H: int
    page_size: int
    num_pages: int
    pool: torch.Tensor                     # fp32 [num_pages, H, V, K], initial contents
    calls: List[object] = field(default_factory=list)
    checkpoint_every: int = 0              # >0: the prefill calls use a separate checkpoint buffer
    seq_lens: Optional[torch.Tensor] = None    # new tokens per sequence (int64, host)
    prefix_lens: Optional[torch.Tensor] = None  # tokens before them (int64, host)
    K: int = K_DIM
    V: int = V_DIM


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_tokens(gen, T: int, H: int, device, decay_scale: float = 1.0, K: int = K_DIM, V: int = V_DIM):
    """q, k, v (bf16) and g, beta (fp32) for T tokens of H heads."""
    q = torch.randn(T, H, K, generator=gen, device=device)
    k = torch.randn(T, H, K, generator=gen, device=device)
    q = (q / q.norm(dim=-1, keepdim=True).clamp_min(1e-6)).to(torch.bfloat16)
    k = (k / k.norm(dim=-1, keepdim=True).clamp_min(1e-6)).to(torch.bfloat16)
    v = torch.randn(T, H, V, generator=gen, device=device).to(torch.bfloat16)
    g = -torch.nn.functional.softplus(torch.randn(T, H, generator=gen, device=device)) * decay_scale
    beta = torch.sigmoid(torch.randn(T, H, generator=gen, device=device))
    return q.contiguous(), k.contiguous(), v.contiguous(), g.float().contiguous(), beta.float().contiguous()


def sentinel_pool(num_pages: int, H: int, device, K: int = K_DIM, V: int = V_DIM) -> torch.Tensor:
    """Pool whose row r is filled with the quiet-NaN bit pattern 0x7FC00000 | r."""
    rows = torch.arange(num_pages, device=device, dtype=torch.int32)
    bits = (rows | 0x7FC00000).view(num_pages, 1, 1, 1).expand(num_pages, H, V, K).contiguous()
    return bits.view(torch.float32)


def fill_rows(pool: torch.Tensor, rows, gen) -> None:
    """Give the listed rows N(0, 1) contents (in the order listed)."""
    rows = torch.as_tensor(rows, dtype=torch.int64).tolist()
    for r in rows:
        pool[r] = torch.randn(pool.shape[1:], generator=gen, device=pool.device)


def page_table(ctx, page_ids, page_size: int, device):
    """CSR page table for sequences of ctx[b] tokens, taking page ids in order
    from page_ids.  Returns int32 (indptr, indices, last_page_len)."""
    ctx = [int(c) for c in torch.as_tensor(ctx).tolist()]
    ids = [int(p) for p in torch.as_tensor(page_ids).tolist()]
    indptr, indices, last = [0], [], []
    for c in ctx:
        n = max(1, -(-c // page_size))
        indices.extend(ids[indptr[-1]:indptr[-1] + n])
        if len(indices) != indptr[-1] + n:
            raise ValueError("not enough page ids")
        last.append(c - (n - 1) * page_size)
        indptr.append(indptr[-1] + n)
    t = lambda x: torch.tensor(x, dtype=torch.int32, device=device)
    return t(indptr), t(indices), t(last)


def _cu(lens, device):
    out = [0]
    for n in lens:
        out.append(out[-1] + int(n))
    return torch.tensor(out, dtype=torch.int32, device=device)


# --------------------------------------------------------------------------
# The five workloads.
# --------------------------------------------------------------------------

def tiny(device="cpu", decay_scale: float = 1.0, seed: int = 1234) -> Workload:
    """2 sequences, H=2, page_size 64.  A prior call prefills sequence 1's
    64-token prefix into its first page; the main call adds [100, 37] new tokens
    (prefixes [0, 64]); then one decode step per sequence.  16-page pool."""
    H, ps, npool = 2, 64, 16
    gen = _gen(seed, device)
    perm = torch.randperm(npool, generator=gen, device=device).tolist()
    pages0, pages1 = perm[0:2], perm[2:4]
    pool = sentinel_pool(npool, H, device)
    calls = []
    q, k, v, g, b = draw_tokens(gen, 64, H, device, decay_scale)
    ip, pi, lpl = page_table([64], pages1[:1], ps, device)
    calls.append(PrefillCall(q, k, v, g, b, _cu([64], device), ip, pi, lpl, ps))
    q, k, v, g, b = draw_tokens(gen, 137, H, device, decay_scale)
    ip, pi, lpl = page_table([100, 101], pages0 + pages1, ps, device)
    calls.append(PrefillCall(q, k, v, g, b, _cu([100, 37], device), ip, pi, lpl, ps))
    q, k, v, g, b = draw_tokens(gen, 2, H, device, decay_scale)
    ip, pi, lpl = page_table([101, 102], pages0 + pages1, ps, device)
    calls.append(DecodeCall(q, k, v, g, b, ip, pi, lpl, ps))
    return Workload("tiny: 2 seqs H=2 ps=64, prefix [0,64] + new [100,37], 1 decode step",
                    H, ps, npool, pool, calls,
                    seq_lens=torch.tensor([100, 37]), prefix_lens=torch.tensor([0, 64]))


def worked_example(device="cpu", decay_scale: float = 1.0, seed: int = 1235) -> Workload:
    """One 2500-token sequence, page_size 1024, H=16, 32-page pool.  A prior
    call prefills the 2048-token prefix into pages [7, 3]; the main call adds
    452 tokens with pages [7, 3, 12] and last_page_len 452."""
    H, ps, npool = 16, 1024, 32
    gen = _gen(seed, device)
    pool = sentinel_pool(npool, H, device)
    calls = []
    q, k, v, g, b = draw_tokens(gen, 2048, H, device, decay_scale)
    ip, pi, lpl = page_table([2048], [7, 3], ps, device)
    calls.append(PrefillCall(q, k, v, g, b, _cu([2048], device), ip, pi, lpl, ps))
    q, k, v, g, b = draw_tokens(gen, 452, H, device, decay_scale)
    ip, pi, lpl = page_table([2500], [7, 3, 12], ps, device)
    calls.append(PrefillCall(q, k, v, g, b, _cu([452], device), ip, pi, lpl, ps))
    return Workload("worked example: 1 seq, 2048 cached + 452 new, ps=1024, H=16",
                    H, ps, npool, pool, calls,
                    seq_lens=torch.tensor([452]), prefix_lens=torch.tensor([2048]))


def decode_batch(device="cuda", B: int = 256, H: int = 32, page_size: int = 1024,
                 num_pages: int = 10000, max_ctx: int = 32768, seed: int = 1236,
                 decay_scale: float = 1.0, steps: int = 1) -> Workload:
    """B sequences with ctx ~ U{2..max_ctx} tokens after the decoded one; a
    quarter (seeded) forced to ctx = m * page_size + 1 (the token opens a new
    page).  Page ids from a permutation of the pool.  ``steps`` decode calls
    with fresh inputs, all on the same page table (for timing)."""
    gen = _gen(seed, device)
    ctx = torch.randint(2, max_ctx + 1, (B,), generator=gen, device=device)
    forced = torch.randperm(B, generator=gen, device=device)[: B // 4]
    m = torch.randint(1, max_ctx // page_size, (B // 4,), generator=gen, device=device)
    ctx[forced] = m * page_size + 1
    perm = torch.randperm(num_pages, generator=gen, device=device)
    ip, pi, lpl = page_table(ctx.cpu(), perm.cpu(), page_size, device)
    calls = []
    for _ in range(steps):
        q, k, v, g, b = draw_tokens(gen, B, H, device, decay_scale)
        calls.append(DecodeCall(q, k, v, g, b, ip, pi, lpl, page_size))
    pool = sentinel_pool(num_pages, H, device)
    fill_rows(pool, pi.cpu(), gen)
    return Workload("decode batch: B=%d H=%d ps=%d ctx U{2..%d}, 25%% open a page, %d-page pool"
                    % (B, H, page_size, max_ctx, num_pages), H, page_size, num_pages, pool, calls)


def mixed_prefill(device="cpu", S: int = 64, H: int = 16, page_size: int = 896,
                  max_len: int = 8192, max_prefix: int = 16384, seed: int = 1237,
                  decay_scale: float = 1.0) -> Workload:
    """S sequences, new lengths floor(exp(U(0, ln(max_len+1)))) - 1 (4 forced
    to 0), prefixes U{0..max_prefix} (4 forced to multiples of 64, 2 to
    multiples of page_size, 2 to 0), plus the last sequence a padded one (no
    new tokens, one scratch page, last_page_len 1).  Checkpoints every
    page_size tokens go to a separate buffer (the caller lays it out)."""
    gen = _gen(seed, device)
    u = torch.rand(S, generator=gen, device=device, dtype=torch.float64)
    L = (torch.exp(u * math.log(max_len + 1)).floor() - 1).clamp(0, max_len).long()
    P = torch.randint(0, max_prefix + 1, (S,), generator=gen, device=device)
    order = torch.randperm(S - 1, generator=gen, device=device).tolist()
    for i in order[0:4]:
        L[i] = 0
    for i in order[4:8]:
        P[i] = 64 * int(torch.randint(0, max_prefix // 64 + 1, (1,), generator=gen, device=device))
    for i in order[8:10]:
        P[i] = page_size * int(torch.randint(0, max_prefix // page_size + 1, (1,), generator=gen, device=device))
    for i in order[10:12]:
        P[i] = 0
    L[S - 1], P[S - 1] = 0, 1                        # the padded sequence
    for i in range(S):                               # a page table holds >= 1 token per sequence
        if int(L[i]) + int(P[i]) == 0:
            P[i] = 1
    L, P = L.cpu(), P.cpu()
    ctx = (L + P).tolist()
    npages_needed = sum(max(1, -(-c // page_size)) for c in ctx)
    num_pages = npages_needed + 64
    perm = torch.randperm(num_pages, generator=gen, device=device)
    ip, pi, lpl = page_table(ctx, perm.cpu(), page_size, device)
    q, k, v, g, b = draw_tokens(gen, int(L.sum()), H, device, decay_scale)
    calls = [PrefillCall(q, k, v, g, b, _cu(L.tolist(), device), ip, pi, lpl, page_size)]
    pool = sentinel_pool(num_pages, H, device)
    fill_rows(pool, pi.cpu(), gen)
    return Workload("mixed prefill: %d seqs H=%d ps=%d, log-uniform new lengths, ragged prefixes"
                    % (S, H, page_size), H, page_size, num_pages, pool, calls,
                    checkpoint_every=page_size, seq_lens=L, prefix_lens=P)


def long_context(device="cuda", S: int = 4, L: int = 65536, H: int = 32, page_size: int = 1152,
                 num_pages: int = 256, decode_steps: int = 128, seed: int = 1238,
                 decay_scale: float = 1.0) -> Workload:
    """S sequences of L new tokens from an empty prefix (state stored at every
    page boundary), then ``decode_steps`` decode steps on the same pool."""
    gen = _gen(seed, device)
    perm = torch.randperm(num_pages, generator=gen, device=device).cpu()
    ip, pi, lpl = page_table([L] * S, perm, page_size, device)
    q, k, v, g, b = draw_tokens(gen, S * L, H, device, decay_scale)
    calls = [PrefillCall(q, k, v, g, b, _cu([L] * S, device), ip, pi, lpl, page_size)]
    for step in range(decode_steps):
        ipd, pid, lpld = page_table([L + step + 1] * S, perm, page_size, device)
        q, k, v, g, b = draw_tokens(gen, S, H, device, decay_scale)
        calls.append(DecodeCall(q, k, v, g, b, ipd, pid, lpld, page_size))
    pool = sentinel_pool(num_pages, H, device)
    return Workload("long context: %d seqs x %d new tokens, H=%d, ps=%d, then %d decode steps"
                    % (S, L, H, page_size, decode_steps), H, page_size, num_pages, pool, calls,
                    seq_lens=torch.tensor([L] * S), prefix_lens=torch.zeros(S, dtype=torch.int64))


@dataclass
class LayerStep:
    """One model step through L GDN layers ("flashinfer.gdn_paged", §Page
    table: the rows depend only on the batch, so one slots call per step serves
    every layer).  Every layer has its own state pool, pools[l] = fp32
    [num_pages, H, V, K], and its own inputs, calls[l]; the page table is the
    same for all layers."""
    name: str
    H: int
    page_size: int
    pools: torch.Tensor            # fp32 [L, num_pages, H, V, K]
    calls: List[object]


def decode_layers(device="cuda", L: int = 32, B: int = 256, H: int = 32, page_size: int = 1024,
                  max_ctx: int = 32768, seed: int = 1241, sentinel: bool = False) -> LayerStep:
    """B sequences decode one token through L layers.  ctx ~ U{2..max_ctx}, a
    quarter (seeded) forced to ctx = m * page_size + 1 (the token opens a new
    page), as in decode_batch.  All pages of a sequence but its last two are
    full prefix pages shared by every sequence (ids 0 .. n_shared - 1; decode
    never reads or writes them); the last two are its own (n_shared + 2b,
    n_shared + 2b + 1), so a layer's pool holds n_shared + 2B rows.  Pools:
    with ``sentinel`` the usual NaN rows with N(0, 1) in the rows a sequence
    owns; otherwise (timing) layer 0's rows N(0, 1), copied to every layer."""
    gen = _gen(seed, device)
    ctx = torch.randint(2, max_ctx + 1, (B,), generator=gen, device=device)
    forced = torch.randperm(B, generator=gen, device=device)[: B // 4]
    m = torch.randint(1, max_ctx // page_size, (B // 4,), generator=gen, device=device)
    ctx[forced] = m * page_size + 1
    ctx = ctx.cpu().tolist()
    n_shared = max(0, max(math.ceil(c / page_size) for c in ctx) - 2)
    indptr, indices, last = [0], [], []
    for b, c in enumerate(ctx):
        n = math.ceil(c / page_size)
        own = [n_shared + 2 * b, n_shared + 2 * b + 1][2 - min(n, 2):]
        indices += list(range(n - len(own))) + own
        indptr.append(len(indices))
        last.append(c - (n - 1) * page_size)
    as_t = lambda x: torch.tensor(x, dtype=torch.int32, device=device)
    ip, pi, lpl = as_t(indptr), as_t(indices), as_t(last)
    num_pages = n_shared + 2 * B
    calls = []
    for _ in range(L):
        q, k, v, g, b_ = draw_tokens(gen, B, H, device)
        calls.append(DecodeCall(q, k, v, g, b_, ip, pi, lpl, page_size))
    if sentinel:
        pools = torch.stack([sentinel_pool(num_pages, H, device) for _ in range(L)])
        for l in range(L):
            fill_rows(pools[l], range(n_shared, num_pages), gen)
    else:
        pools = torch.empty(L, num_pages, H, V_DIM, K_DIM, device=device)
        pools[0] = torch.randn(num_pages, H, V_DIM, K_DIM, generator=gen, device=device)
        pools[1:] = pools[0]
    return LayerStep("decode step: %d layers, B=%d, H=%d, ps=%d, ctx U{2..%d} (25%% open a page), "
                     "last two pages per sequence own, the rest shared" % (L, B, H, page_size, max_ctx),
                     H, page_size, pools, calls)


def prefill_layers(device="cuda", L: int = 32, S: int = 4, T_seq: int = 8192, H: int = 32,
                   page_size: int = 1152, seed: int = 1242, sentinel: bool = False) -> LayerStep:
    """S sequences of T_seq new tokens from an empty prefix through L layers
    (state stored at every page end).  Layer 0's tokens are drawn as usual;
    layer l's are layer 0's rolled by l * 997 tokens (distinct buffers and
    contents).  Pools: sentinel NaN rows with ``sentinel``, else zeros (an
    empty prefix reads no row)."""
    gen = _gen(seed, device)
    num_pages = S * math.ceil(T_seq / page_size)
    perm = torch.randperm(num_pages, generator=gen, device=device).cpu()
    ip, pi, lpl = page_table([T_seq] * S, perm, page_size, device)
    q0, k0, v0, g0, b0 = draw_tokens(gen, S * T_seq, H, device)
    cu = _cu([T_seq] * S, device)
    calls = []
    for l in range(L):
        r = lambda t: torch.roll(t, l * 997, dims=0).contiguous()
        calls.append(PrefillCall(r(q0), r(k0), r(v0), r(g0), r(b0), cu, ip, pi, lpl, page_size))
    if sentinel:
        pools = torch.stack([sentinel_pool(num_pages, H, device) for _ in range(L)])
    else:
        pools = torch.zeros(L, num_pages, H, V_DIM, K_DIM, device=device)
    return LayerStep("prefill step: %d layers, %d seqs x %d new tokens, H=%d, ps=%d"
                     % (L, S, T_seq, H, page_size), H, page_size, pools, calls)


WORKLOADS = {0: tiny, 1: worked_example, 2: decode_batch, 3: mixed_prefill, 4: long_context}
