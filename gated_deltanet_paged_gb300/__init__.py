"""Paged Gated Delta-Rule (GDN) prefill and decode for GB300 (sm_103a).

Thin ctypes binding over the C ABI in ``include/gdn_paged.h``: each function
checks tensor dtypes / devices, passes ``data_ptr()`` values and the current
CUDA stream, and raises on a non-zero status.  Every step of the computation
runs in the CUDA library ``libgdn_paged.so``; there is no fallback path, and
calling any of these functions without the library (or without an sm_103a GPU)
raises.

Source: "flashinfer.gdn_paged" (docs.flashinfer.ai/api/gdn_paged.html).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "gdn_paged_prefill_slots",
    "gdn_paged_decode_slots",
    "gdn_chunk_gated_delta_rule",
    "gdn_chunk_gated_delta_rule_paged",
    "gdn_gated_delta_rule_decode_paged",
    "gdn_pool_copy_rows",
    "gdn_pool_zero_rows",
    "gdn_prefill_workspace_bytes",
    "gdn_status_string",
    "library",
    "GdnError",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn_paged.so")
_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    """A gdn_* call returned a negative status."""

    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (fn, library().gdn_status_string(status).decode(), status))


class _PrefillSlots(ctypes.Structure):
    _fields_ = [("state_indices", ctypes.c_void_p), ("output_state_indices", ctypes.c_void_p),
                ("checkpoint_cu_starts", ctypes.c_void_p), ("prefix_lens", ctypes.c_void_p)]


class _DecodeSlots(ctypes.Structure):
    _fields_ = [("initial_state_indices", ctypes.c_void_p), ("output_state_indices", ctypes.c_void_p)]


def library():
    """Load libgdn_paged.so (building it first if the sources are newer)."""
    global _lib
    with _lock:
        if _lib is None:
            from . import build as _build
            if not _build.up_to_date():
                try:
                    _build.build()
                except Exception as e:  # no silent fallback: the CUDA library is the product
                    raise RuntimeError("libgdn_paged.so is missing or stale and could not be built: %s" % e)
            lib = ctypes.CDLL(LIB_PATH)
            P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
            sig = {
                "gdn_paged_prefill_slots": [P, P, P, P, i32, i32, P, P, P, P, P],
                "gdn_paged_decode_slots": [P, P, P, i32, P, P, P],
                "gdn_chunk_gated_delta_rule": [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f32,
                                               P, P, P, P, P, P, P, P, i32, i64, P, sz, P, P],
                "gdn_chunk_gated_delta_rule_paged": [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f32,
                                                     P, i32, P, P, i32, P, P, P, sz, P, P],
                "gdn_gated_delta_rule_decode_paged": [P, P, P, P, P, P, i32, i32, i32, i32, f32,
                                                      P, i32, P, P, P, P, P, P],
                "gdn_chunk_gated_delta_rule_ex": [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f32,
                                                  P, P, P, P, P, P, P, P, i32, i64, i32, i32, P, sz, P, P],
                "gdn_chunk_gated_delta_rule_paged_ex": [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f32,
                                                        P, i32, i32, P, P, i32, P, P, P, sz, P, P],
                "gdn_gated_delta_rule_decode_paged_ex": [P, P, P, P, P, P, i32, i32, i32, i32, f32,
                                                         P, i32, i32, P, P, P, P, P, P],
                "gdn_pool_copy_rows": [P, i64, i64, P, P, i32, i32, P, P],
                "gdn_pool_zero_rows": [P, i64, i64, P, i32, i32, P, P],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.gdn_prefill_workspace_bytes.argtypes = [i32, i32, i32]
            lib.gdn_prefill_workspace_bytes.restype = ctypes.c_size_t
            lib.gdn_status_string.argtypes = [ctypes.c_int]
            lib.gdn_status_string.restype = ctypes.c_char_p
            lib.gdn_debug_set_wait_stall.argtypes = [i32]
            lib.gdn_debug_set_wait_stall.restype = None
            _lib = lib
    return _lib


def gdn_debug_set_wait_stall(enable: bool) -> None:
    """Fault injection for tests of the bounded waits: while enabled, the
    state-chain kernel of each later prefill call makes its first wait on a
    barrier that nothing completes; the wait gives up after about 1 ms, before
    any copy or tensor-core operation is issued, and the call records
    GDN_DEVERR_TIMEOUT in err_word and writes nothing."""
    library().gdn_debug_set_wait_stall(1 if enable else 0)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(t):
    return torch.cuda.current_stream(t.device).cuda_stream


def _need(t, dtype, name, ndim=None):
    if t is None:
        raise ValueError("%s is required" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims" % (name, ndim))
    return t


def _opt(t, dtype, name):
    return None if t is None else _need(t, dtype, name)


def _check(fn, status):
    if status != 0:
        raise GdnError(fn, status)


# State pool element types (GDN_STATE_F32 / GDN_STATE_BF16 of the C header).
_STATE_DTYPES = {torch.float32: 0, torch.bfloat16: 1}


def _state_dtype(pools, names):
    """The pools' common element type code; fp32 or bf16 pools, all alike."""
    kinds = {p.dtype for p in pools if p is not None}
    if len(kinds) > 1:
        raise TypeError("%s must share one dtype" % ", ".join(names))
    kind = kinds.pop() if kinds else torch.float32
    if kind not in _STATE_DTYPES:
        raise TypeError("state pools must be float32 or bfloat16, got %s" % kind)
    return _STATE_DTYPES[kind]


# Slot-array element types (GDN_INDEX_I32 / GDN_INDEX_I64 of the C header).
_INDEX_DTYPES = {torch.int32: 0, torch.int64: 1}


def _index_dtype(arrays, names):
    """The slot arrays' common element type code; int32 or int64, all alike."""
    kinds = {t.dtype for t in arrays if t is not None}
    if len(kinds) > 1:
        raise TypeError("%s must share one dtype" % ", ".join(names))
    kind = kinds.pop() if kinds else torch.int32
    if kind not in _INDEX_DTYPES:
        raise TypeError("slot arrays must be int32 or int64, got %s" % kind)
    return _INDEX_DTYPES[kind]


def _pool_arg(t, dtype, name):
    """A state pool [rows, H, V, K] whose rows are dense; the row stride
    (stride(0)) may be padded."""
    if t is None:
        return None
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dim() != 4 or not t[0].is_contiguous() or t.stride(0) < t[0].numel():
        raise ValueError("%s must be [rows, H, V, K] with dense rows" % name)
    return t


def gdn_status_string(status: int) -> str:
    return library().gdn_status_string(status).decode()


def gdn_prefill_workspace_bytes(num_seqs: int, total_tokens: int, H: int) -> int:
    return int(library().gdn_prefill_workspace_bytes(num_seqs, total_tokens, H))


def gdn_paged_prefill_slots(cu_seqlens, page_indptr, page_indices, last_page_len, page_size, out=None):
    """Rows of a paged prefill batch: dict of four int32 [num_seqs] tensors
    (state_indices, output_state_indices, checkpoint_cu_starts, prefix_lens)."""
    i32 = torch.int32
    for t, n in ((cu_seqlens, "cu_seqlens"), (page_indptr, "page_indptr"), (page_indices, "page_indices"),
                 (last_page_len, "last_page_len")):
        _need(t, i32, n)
    n = cu_seqlens.numel() - 1
    names = ("state_indices", "output_state_indices", "checkpoint_cu_starts", "prefix_lens")
    if out is None:
        out = {k: torch.empty(n, dtype=i32, device=cu_seqlens.device) for k in names}
    for k in names:
        _need(out[k], i32, k)
    _check("gdn_paged_prefill_slots", library().gdn_paged_prefill_slots(
        _ptr(cu_seqlens), _ptr(page_indptr), _ptr(page_indices), _ptr(last_page_len), n, int(page_size),
        *[_ptr(out[k]) for k in names], _stream(cu_seqlens)))
    return out


def gdn_paged_decode_slots(page_indptr, page_indices, last_page_len, out=None):
    """Rows of a paged decode batch: dict of two int32 [B] tensors
    (initial_state_indices, output_state_indices)."""
    i32 = torch.int32
    for t, n in ((page_indptr, "page_indptr"), (page_indices, "page_indices"), (last_page_len, "last_page_len")):
        _need(t, i32, n)
    b = page_indptr.numel() - 1
    names = ("initial_state_indices", "output_state_indices")
    if out is None:
        out = {k: torch.empty(b, dtype=i32, device=page_indptr.device) for k in names}
    _check("gdn_paged_decode_slots", library().gdn_paged_decode_slots(
        _ptr(page_indptr), _ptr(page_indices), _ptr(last_page_len), b,
        _ptr(out[names[0]]), _ptr(out[names[1]]), _stream(page_indptr)))
    return out


def _workspace(workspace, num_seqs, T, H, device):
    """The prefill workspace: the caller's uint8 tensor (checked for size) or a
    fresh one from the torch caching allocator."""
    need = gdn_prefill_workspace_bytes(num_seqs, T, H)
    if workspace is None:
        return torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    _need(workspace, torch.uint8, "workspace")
    if workspace.numel() < need:
        raise ValueError("workspace holds %d bytes, the call needs %d" % (workspace.numel(), need))
    return workspace


def _tokens(q, k, v, g, beta):
    _need(q, torch.bfloat16, "q", 3)
    _need(k, torch.bfloat16, "k", 3)
    _need(v, torch.bfloat16, "v", 3)
    _need(g, torch.float32, "g", 2)
    _need(beta, torch.float32, "beta", 2)
    T, H, K = q.shape
    V = v.shape[2]
    if k.shape != q.shape or v.shape[:2] != (T, H) or g.shape != (T, H) or beta.shape != (T, H):
        raise ValueError("q, k: [T, H, K]; v: [T, H, V]; g, beta: [T, H]")
    return T, H, K, V


def gdn_chunk_gated_delta_rule(q, k, v, g, beta, cu_seqlens, *, scale=0.0, initial_state=None,
                               state_indices=None, output_state=None, output_state_indices=None,
                               state_checkpoints=None, checkpoint_state_indices=None,
                               checkpoint_cu_starts=None, prefix_lens=None, checkpoint_every_n_tokens=0,
                               o=None, err_word=None, workspace=None):
    """Chunked prefill with slot arguments (explicit read / final / checkpoint
    rows).  Returns o (bf16 [T, H, V]); pools are updated in place.  The slot
    arrays are int32 or int64 (all alike); the pools fp32 or bf16 (all alike)
    [rows, H, V, K] with dense rows and one row stride, which may be padded.
    ``workspace``: optional uint8 device tensor of at least
    gdn_prefill_workspace_bytes(num_seqs, T, H) bytes."""
    T, H, K, V = _tokens(q, k, v, g, beta)
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    pool_names = ("initial_state", "output_state", "state_checkpoints")
    sd = _state_dtype((initial_state, output_state, state_checkpoints), pool_names)
    pdt = torch.bfloat16 if sd else torch.float32
    pools = [_pool_arg(p, pdt, n) for p, n in zip((initial_state, output_state, state_checkpoints), pool_names)]
    strides = {p.stride(0) for p in pools if p is not None}
    if len(strides) > 1:
        raise ValueError("%s must share one row stride" % ", ".join(pool_names))
    stride = strides.pop() if strides else 0
    idx_names = ("state_indices", "output_state_indices", "checkpoint_state_indices", "checkpoint_cu_starts",
                 "prefix_lens")
    idx = (state_indices, output_state_indices, checkpoint_state_indices, checkpoint_cu_starts, prefix_lens)
    xd = _index_dtype(idx, idx_names)
    idt = torch.int64 if xd else torch.int32
    idx = [_opt(t, idt, n) for t, n in zip(idx, idx_names)]
    if o is None:
        o = torch.empty(T, H, V, dtype=torch.bfloat16, device=q.device)
    _need(o, torch.bfloat16, "o", 3)
    ws = _workspace(workspace, cu_seqlens.numel() - 1, T, H, q.device)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(o), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, H,
            K, V, float(scale), _ptr(pools[0]), _ptr(idx[0]), _ptr(pools[1]), _ptr(idx[1]), _ptr(pools[2]),
            _ptr(idx[2]), _ptr(idx[3]), _ptr(idx[4]), int(checkpoint_every_n_tokens), stride)
    tail = (_ptr(ws), ws.numel(), _ptr(_opt(err_word, torch.int32, "err_word")), _stream(q))
    if sd or xd:
        _check("gdn_chunk_gated_delta_rule_ex", library().gdn_chunk_gated_delta_rule_ex(*args, sd, xd, *tail))
    else:
        _check("gdn_chunk_gated_delta_rule", library().gdn_chunk_gated_delta_rule(*args, *tail))
    return o


def gdn_chunk_gated_delta_rule_paged(q, k, v, g, beta, cu_seqlens, state_pool, page_indices, page_indptr,
                                     page_size, last_page_len, *, scale=0.0, slots=None, o=None, err_word=None,
                                     workspace=None):
    """Paged chunked prefill over state_pool [num_pages, H, V, K].  ``slots``:
    the dict returned by gdn_paged_prefill_slots (optional).  ``workspace``:
    optional uint8 device tensor (see gdn_prefill_workspace_bytes).  Returns o."""
    T, H, K, V = _tokens(q, k, v, g, beta)
    i32 = torch.int32
    _need(cu_seqlens, i32, "cu_seqlens")
    sd = _state_dtype((state_pool,), ("state_pool",))
    _need(state_pool, torch.bfloat16 if sd else torch.float32, "state_pool", 4)
    for t, n in ((page_indices, "page_indices"), (page_indptr, "page_indptr"), (last_page_len, "last_page_len")):
        _need(t, i32, n)
    if o is None:
        o = torch.empty(T, H, V, dtype=torch.bfloat16, device=q.device)
    _need(o, torch.bfloat16, "o", 3)
    ws = _workspace(workspace, cu_seqlens.numel() - 1, T, H, q.device)
    sl = None
    if slots is not None:
        sl = _PrefillSlots(*[_ptr(_need(slots[n], i32, n)) for n in
                             ("state_indices", "output_state_indices", "checkpoint_cu_starts", "prefix_lens")])
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(o), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, H,
            K, V, float(scale), _ptr(state_pool))
    rest = (state_pool.shape[0], _ptr(page_indices), _ptr(page_indptr), int(page_size), _ptr(last_page_len),
            None if sl is None else ctypes.byref(sl), _ptr(ws), ws.numel(), _ptr(_opt(err_word, i32, "err_word")),
            _stream(q))
    if sd:
        _check("gdn_chunk_gated_delta_rule_paged_ex", library().gdn_chunk_gated_delta_rule_paged_ex(*head, sd, *rest))
    else:
        _check("gdn_chunk_gated_delta_rule_paged", library().gdn_chunk_gated_delta_rule_paged(*head, *rest))
    return o


def gdn_gated_delta_rule_decode_paged(q, k, v, g, beta, state_pool, page_indices, page_indptr, last_page_len, *,
                                      scale=0.0, slots=None, o=None, err_word=None):
    """Single-token paged decode.  q, k: bf16 [B, H, K]; v: bf16 [B, H, V];
    g, beta: fp32 [B, H]; ``slots``: dict from gdn_paged_decode_slots
    (optional).  Returns o (bf16 [B, H, V])."""
    B, H, K, V = _tokens(q, k, v, g, beta)
    i32 = torch.int32
    sd = _state_dtype((state_pool,), ("state_pool",))
    _need(state_pool, torch.bfloat16 if sd else torch.float32, "state_pool", 4)
    for t, n in ((page_indices, "page_indices"), (page_indptr, "page_indptr"), (last_page_len, "last_page_len")):
        _need(t, i32, n)
    if o is None:
        o = torch.empty(B, H, V, dtype=torch.bfloat16, device=q.device)
    _need(o, torch.bfloat16, "o", 3)
    sl = None
    if slots is not None:
        sl = _DecodeSlots(*[_ptr(_need(slots[n], i32, n)) for n in ("initial_state_indices", "output_state_indices")])
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(o), B, H, K, V, float(scale), _ptr(state_pool))
    rest = (state_pool.shape[0], _ptr(page_indices), _ptr(page_indptr), _ptr(last_page_len),
            None if sl is None else ctypes.byref(sl), _ptr(_opt(err_word, i32, "err_word")), _stream(q))
    if sd:
        _check("gdn_gated_delta_rule_decode_paged_ex", library().gdn_gated_delta_rule_decode_paged_ex(*head, sd, *rest))
    else:
        _check("gdn_gated_delta_rule_decode_paged", library().gdn_gated_delta_rule_decode_paged(*head, *rest))
    return o


def _pool_rows(pool, name):
    if not pool.is_cuda or pool.dim() < 2:
        raise ValueError("%s must be a CUDA tensor [rows, ...]" % name)
    inner = pool[0]
    if not inner.is_contiguous():
        raise ValueError("%s rows must be contiguous" % name)
    return inner.numel() * pool.element_size(), pool.stride(0) * pool.element_size()


def gdn_pool_copy_rows(pool, src_rows, dst_rows, err_word=None):
    """Bit-exact copies of whole pool rows: row dst_rows[i] <- row src_rows[i]
    (-1 on either side skips).  Any element type; the pool is updated in place."""
    i32 = torch.int32
    _need(src_rows, i32, "src_rows", 1)
    _need(dst_rows, i32, "dst_rows", 1)
    if src_rows.numel() != dst_rows.numel():
        raise ValueError("src_rows and dst_rows must have the same length")
    row_bytes, stride_bytes = _pool_rows(pool, "pool")
    _check("gdn_pool_copy_rows", library().gdn_pool_copy_rows(
        _ptr(pool), row_bytes, stride_bytes, _ptr(src_rows), _ptr(dst_rows), dst_rows.numel(), pool.shape[0],
        _ptr(_opt(err_word, i32, "err_word")), _stream(pool)))
    return pool


def gdn_pool_zero_rows(pool, rows, err_word=None):
    """Whole pool rows set to zero bits (-1 skips); the pool is updated in place."""
    i32 = torch.int32
    _need(rows, i32, "rows", 1)
    row_bytes, stride_bytes = _pool_rows(pool, "pool")
    _check("gdn_pool_zero_rows", library().gdn_pool_zero_rows(
        _ptr(pool), row_bytes, stride_bytes, _ptr(rows), rows.numel(), pool.shape[0],
        _ptr(_opt(err_word, i32, "err_word")), _stream(pool)))
    return pool
