"""Plain fp64 CPU oracle of paged Gated Delta-Rule (GDN) prefill and decode.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library ``gated_deltanet_paged_gb300``; the two meet only
through the seeded inputs of ``gated_deltanet_paged_gb300.workloads``.

The arithmetic lives in ``gdn_oracle.c`` (token-by-token fp64 recurrence and
slot derivation by walking token positions); this module marshals numpy arrays
into it.  ``csr.py`` holds the block-table <-> CSR conversions.

Sources ("flashinfer.gdn_paged", docs.flashinfer.ai/api/gdn_paged.html): the
intro, "Page table", the prefill bullets, the decode paragraph and "Slot
arguments of chunk_gated_delta_rule".  Parity of the default ``scale``, the
tensor layouts and the output dtype is unpinned: the pages fix none of them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .csr import block_table_to_csr, csr_to_block_table, csr_from_lengths  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into liboracle.so (plain gcc, OpenMP over chains)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_prefill_slots.argtypes = [i32, P, P, P, P, i32, P, P, P, P]
            lib.oracle_decode_slots.argtypes = [i32, P, P, P, i32, P, P]
            lib.oracle_chunk_gdn_st.argtypes = [i32, P, i32, i32, i32, f64, P, P, P, P, P, P,
                                                P, P, P, P, P, P, P, P, i32, i64, P, P, P, i32]
            lib.oracle_decode_st.argtypes = [i32, i32, i32, i32, f64, P, P, P, P, P, P, P, i64,
                                             P, P, P, P, i32]
            lib.oracle_double_to_bf16.argtypes = [f64]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            for fn in (lib.oracle_prefill_slots, lib.oracle_decode_slots, lib.oracle_chunk_gdn_st,
                       lib.oracle_decode_st):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def _bits(a):
    """bf16 tensors arrive as raw uint16 bit patterns (numpy has no bf16)."""
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs must be passed as uint16 bit patterns")
    return a


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def prefill_slots(cu_seqlens, page_indptr, page_indices, last_page_len, page_size):
    """Pool rows of a paged prefill batch, by walking token positions.

    Returns a dict of four int32 [num_seqs] arrays: state_indices,
    output_state_indices, checkpoint_cu_starts, prefix_lens.
    """
    cu, ip, pi, lpl = map(_i32, (cu_seqlens, page_indptr, page_indices, last_page_len))
    n = len(cu) - 1
    out = {name: np.zeros(n, np.int32) for name in
           ("state_indices", "output_state_indices", "checkpoint_cu_starts", "prefix_lens")}
    rc = _load().oracle_prefill_slots(n, _ptr(cu), _ptr(ip), _ptr(pi), _ptr(lpl), int(page_size),
                                      _ptr(out["state_indices"]), _ptr(out["output_state_indices"]),
                                      _ptr(out["checkpoint_cu_starts"]), _ptr(out["prefix_lens"]))
    if rc != 0:
        raise ValueError("invalid page table")
    return out


def decode_slots(page_indptr, page_indices, last_page_len, page_size):
    """Read and write pool rows of a paged decode batch (two int32 [B] arrays)."""
    ip, pi, lpl = map(_i32, (page_indptr, page_indices, last_page_len))
    b = len(ip) - 1
    out = {"initial_state_indices": np.zeros(b, np.int32), "output_state_indices": np.zeros(b, np.int32)}
    rc = _load().oracle_decode_slots(b, _ptr(ip), _ptr(pi), _ptr(lpl), int(page_size),
                                     _ptr(out["initial_state_indices"]), _ptr(out["output_state_indices"]))
    if rc != 0:
        raise ValueError("invalid page table")
    return out


def _row_stride(pool, H, K, V):
    if pool is None:
        return H * V * K
    if pool.dtype not in (np.float32, np.uint16) or not pool.flags.c_contiguous:
        raise TypeError("pools must be C-contiguous float32, or uint16 holding bf16 bits")
    stride = int(np.prod(pool.shape[1:]))  # a row may be padded past its H*V*K state elements
    if stride < H * V * K:
        raise ValueError("a pool row holds fewer than H*V*K elements")
    return stride


def _state_bf16(pools):
    """1 when the pools hold bf16 bits (uint16), 0 for float32; all alike."""
    kinds = {p.dtype for p in pools if p is not None}
    if len(kinds) > 1:
        raise TypeError("pools must share one element type")
    return int(kinds == {np.dtype(np.uint16)})


def double_to_bf16_bits(x: float) -> int:
    """The bf16 value nearest to x (ties to even) as bits, as the oracle stores
    states in a bf16 pool."""
    return int(_load().oracle_double_to_bf16(float(x)))


def chunk_gated_delta_rule(q, k, v, g, beta, cu_seqlens, scale, *, initial_state=None,
                           state_indices=None, output_state=None, output_state_indices=None,
                           state_checkpoints=None, checkpoint_state_indices=None,
                           checkpoint_cu_starts=None, prefix_lens=None,
                           checkpoint_every_n_tokens=0, chains=None):
    """Prefill with slot arguments, token by token in fp64.

    q, k: uint16 [T, H, K] (bf16 bits); v: uint16 [T, H, V]; g, beta: float32
    [T, H]; pools: float32 [rows, H, V, K] arrays, or uint16 ones holding bf16
    bits (states then rounded to bf16, ties to even), updated in place (they may
    be the same array).  ``chains`` (bool [num_seqs, H]) restricts the work to some
    (sequence, head) chains.  Returns (o float64 [T, H, V], out_written,
    ckpt_written) where the last two flag the rows stored (or None).
    """
    q, k, v = _bits(q), _bits(k), _bits(v)
    g, beta = _f32(g), _f32(beta)
    T, H, K = q.shape
    V = v.shape[2]
    cu = _i32(cu_seqlens)
    num_seqs = len(cu) - 1
    pools = [p for p in (initial_state, output_state, state_checkpoints) if p is not None]
    stride = _row_stride(pools[0] if pools else None, H, K, V)
    for p in pools:
        if _row_stride(p, H, K, V) != stride:
            raise ValueError("pools must share one row stride")
    o = np.zeros((T, H, V), np.float64)
    out_written = np.zeros(output_state.shape[0], np.uint8) if output_state is not None else None
    ckpt_written = np.zeros(state_checkpoints.shape[0], np.uint8) if state_checkpoints is not None else None
    mask = None if chains is None else np.ascontiguousarray(chains, dtype=np.uint8).reshape(-1)
    si, osi, csi, ccs, pl = map(_i32, (state_indices, output_state_indices, checkpoint_state_indices,
                                      checkpoint_cu_starts, prefix_lens))
    rc = _load().oracle_chunk_gdn_st(
        num_seqs, _ptr(cu), H, K, V, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(o), _ptr(initial_state), _ptr(si), _ptr(output_state), _ptr(osi),
        _ptr(state_checkpoints), _ptr(csi), _ptr(ccs), _ptr(pl), int(checkpoint_every_n_tokens),
        stride, _ptr(mask), _ptr(out_written), _ptr(ckpt_written), _state_bf16(pools))
    if rc != 0:
        raise ValueError("oracle_chunk_gdn failed (%d)" % rc)
    return o, out_written, ckpt_written


def chunk_gated_delta_rule_paged(q, k, v, g, beta, cu_seqlens, state_pool, page_indices,
                                 page_indptr, page_size, last_page_len, scale, chains=None):
    """Paged prefill: the slot-argument prefill with one pool for the read,
    final and checkpoint rows, the page list as checkpoint rows and
    N = page_size ("Slot arguments of chunk_gated_delta_rule": the paged call is
    a thin wrapper over these arguments).  Updates state_pool in place and
    returns (o, written) with written flagging the pool rows stored."""
    s = prefill_slots(cu_seqlens, page_indptr, page_indices, last_page_len, page_size)
    o, w_out, w_ckpt = chunk_gated_delta_rule(
        q, k, v, g, beta, cu_seqlens, scale, initial_state=state_pool,
        state_indices=s["state_indices"], output_state=state_pool,
        output_state_indices=s["output_state_indices"], state_checkpoints=state_pool,
        checkpoint_state_indices=_i32(page_indices), checkpoint_cu_starts=s["checkpoint_cu_starts"],
        prefix_lens=s["prefix_lens"], checkpoint_every_n_tokens=page_size, chains=chains)
    return o, (w_out | w_ckpt)


def gated_delta_rule_decode(q, k, v, g, beta, state_pool, initial_state_indices,
                            output_state_indices, scale, chains=None):
    """One token per sequence on explicit read / write rows.  q, k: uint16
    [B, H, K]; v: uint16 [B, H, V]; g, beta: float32 [B, H]; state_pool float32,
    or uint16 holding bf16 bits.  Returns (o float64 [B, H, V], written)."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    g, beta = _f32(g), _f32(beta)
    B, H, K = q.shape
    V = v.shape[2]
    stride = _row_stride(state_pool, H, K, V)
    o = np.zeros((B, H, V), np.float64)
    written = np.zeros(state_pool.shape[0], np.uint8)
    isi, osi = _i32(initial_state_indices), _i32(output_state_indices)
    mask = None if chains is None else np.ascontiguousarray(chains, dtype=np.uint8).reshape(-1)
    rc = _load().oracle_decode_st(B, H, K, V, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                  _ptr(beta), _ptr(o), _ptr(state_pool), stride, _ptr(isi), _ptr(osi),
                                  _ptr(mask), _ptr(written), _state_bf16([state_pool]))
    if rc != 0:
        raise ValueError("oracle_decode failed (%d)" % rc)
    return o, written


def gated_delta_rule_decode_paged(q, k, v, g, beta, state_pool, page_indices, page_indptr,
                                  last_page_len, page_size, scale, chains=None):
    """Paged decode: decode rows from the page table, then one token each."""
    s = decode_slots(page_indptr, page_indices, last_page_len, page_size)
    return gated_delta_rule_decode(q, k, v, g, beta, state_pool, s["initial_state_indices"],
                                   s["output_state_indices"], scale, chains=chains)


def pool_copy_rows(pool, src_rows, dst_rows):
    """Row copies by their definition ("gdn-prefix-cache", §The fix: states
    moved between rows as bit-exact copies): for each pair in order, row dst
    takes the bytes of row src; -1 on either side, or a row outside the pool,
    skips the pair.  pool: any numpy array [rows, ...], updated in place."""
    n = pool.shape[0]
    for s_, d in zip(np.asarray(src_rows).tolist(), np.asarray(dst_rows).tolist()):
        if 0 <= s_ < n and 0 <= d < n:
            pool[d] = pool[s_]
    return pool


def pool_zero_rows(pool, rows):
    """Rows set to zero bits (the zero state); -1 or out-of-range rows skip."""
    n = pool.shape[0]
    for r in np.asarray(rows).tolist():
        if 0 <= r < n:
            pool[r] = 0
    return pool
