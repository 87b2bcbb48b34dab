"""Block table <-> CSR page table, written as plain loops.

TEST INFRASTRUCTURE ONLY (part of the oracle package).

Follows "F1 提示与讲解 · FlashInfer 的 CSR 分页格式与 plan / run"
(kzhou003.github.io/gpu-kernel-drills/hints/f1_flashinfer_paged.html),
sections ① (the three CSR arrays and ctx = (pages - 1) * page_size +
last_page_len), ② (block table -> CSR; a full last page has length page_size,
not 0) and ③ (CSR -> block table), and "flashinfer.gdn_paged" §Page table.
"""
from __future__ import annotations

import numpy as np


def pages_for(ctx: int, page_size: int) -> int:
    """Number of pages a sequence of ctx >= 1 tokens fills, counted by filling
    pages one token at a time."""
    if ctx < 1:
        raise ValueError("a sequence in a page table holds at least one token")
    pages, fill = 1, 0
    for _ in range(ctx):
        if fill == page_size:
            pages += 1
            fill = 0
        fill += 1
    return pages


def block_table_to_csr(block_table, ctx, page_size):
    """Padded per-sequence block table [B, max_blocks] + token counts [B] ->
    (indptr [B+1], indices [sum pages], last_page_len [B]), all int32.

    Sequence b keeps the first pages_for(ctx[b]) entries of its row, in order;
    its last page holds ctx[b] - (pages - 1) * page_size tokens (1..page_size).
    """
    block_table = np.asarray(block_table)
    indptr, indices, last = [0], [], []
    for b, c in enumerate(np.asarray(ctx).tolist()):
        n = pages_for(int(c), page_size)
        indices.extend(int(x) for x in block_table[b, :n])
        indptr.append(indptr[-1] + n)
        last.append(int(c) - (n - 1) * page_size)
    return (np.array(indptr, np.int32), np.array(indices, np.int32), np.array(last, np.int32))


def csr_to_block_table(indptr, indices, last_page_len, page_size, max_blocks):
    """CSR -> (block table [B, max_blocks] padded with 0, ctx [B]).

    Rejects a sequence with no page or a last_page_len outside 1..page_size:
    the CSR arrays can express them, but a sequence holds at least one token.
    """
    indptr = np.asarray(indptr).tolist()
    indices = np.asarray(indices).tolist()
    last = np.asarray(last_page_len).tolist()
    B = len(indptr) - 1
    table = np.zeros((B, max_blocks), np.int32)
    ctx = np.zeros(B, np.int32)
    for b in range(B):
        n = indptr[b + 1] - indptr[b]
        if n < 1:
            raise ValueError("sequence %d owns no page" % b)
        if not 1 <= last[b] <= page_size:
            raise ValueError("last_page_len[%d] = %d is outside 1..page_size" % (b, last[b]))
        if n > max_blocks:
            raise ValueError("sequence %d needs %d blocks > max_blocks" % (b, n))
        for j in range(n):
            table[b, j] = indices[indptr[b] + j]
        ctx[b] = (n - 1) * page_size + last[b]
    return table, ctx


def csr_from_lengths(ctx, page_ids, page_size):
    """Lay sequences of ctx[b] tokens out on consecutive ids taken from
    page_ids (in order) and return (indptr, indices, last_page_len)."""
    page_ids = list(np.asarray(page_ids).tolist())
    rows, need = [], 0
    for c in np.asarray(ctx).tolist():
        n = pages_for(int(c), page_size)
        rows.append(page_ids[need:need + n])
        need += n
    if need > len(page_ids):
        raise ValueError("not enough page ids")
    width = max((len(r) for r in rows), default=0)
    table = np.zeros((len(rows), max(width, 1)), np.int64)
    for b, r in enumerate(rows):
        table[b, :len(r)] = r
    return block_table_to_csr(table, ctx, page_size)
