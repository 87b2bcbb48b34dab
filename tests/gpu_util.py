"""Shared helpers of the GPU parity tests: run a call through the CUDA library
and through the oracle on the same inputs, and compare.

Acceptance (written here once, used by every GPU test):
  - slots, page tables, untouched pool rows: bit-exact;
  - outputs o: max-abs difference <= 1e-2 against the fp64 oracle;
  - every written state: relative Frobenius error <= 1e-3 per (row, head);
    in a bf16 pool <= 5e-3: both sides round their state to the nearest bf16
    (the oracle from fp64, the GPU from fp32), which adds at most one bf16
    step, 2^-8 of the value, to the fp32 bound.
"""
import numpy as np
import torch

import gated_deltanet_paged_gb300 as gdn
import oracle
from conftest import bf16_bits, f32, i32

O_TOL = 1e-2
S_TOL = 1e-3
S_TOL_BF16 = 5e-3
SCALE = 128 ** -0.5


class Errors:
    """Largest errors seen, for the test log."""

    def __init__(self):
        self.o = 0.0
        self.state = 0.0

    def __repr__(self):
        return "max|do|=%.3g  max state rel-fro=%.3g" % (self.o, self.state)


def rel_fro_rows(gpu, ref):
    """[rows, H, V, K] -> [rows, H] relative Frobenius errors."""
    g = gpu.astype(np.float64).reshape(gpu.shape[0], gpu.shape[1], -1)
    r = ref.astype(np.float64).reshape(ref.shape[0], ref.shape[1], -1)
    return np.linalg.norm(g - r, axis=2) / np.maximum(np.linalg.norm(r, axis=2), 1e-30)


def check_o(o_gpu, o_ref, errs, rows=None):
    got = o_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got, o_ref = got[rows], o_ref[rows]
    assert np.isfinite(got).all(), "non-finite output"
    d = float(np.abs(got - o_ref).max()) if got.size else 0.0
    errs.o = max(errs.o, d)
    assert d <= O_TOL, "max-abs output error %.4g > %g" % (d, O_TOL)


def bits_equal(a, b):
    it = torch.int16 if a.element_size() == 2 else torch.int32
    return torch.equal(a.view(it), b.view(it))


def bf16_pool_pair(pool_f32):
    """A bf16 pool for the GPU (torch) and the oracle (uint16 bits) from an fp32
    pool: each value cut to its top 16 bits (NaN sentinels stay NaN)."""
    bits = (pool_f32.view(torch.int32) >> 16).to(torch.int16)
    return bits.view(torch.bfloat16), bits.cpu().numpy().view(np.uint16).copy()


def _pool_f64(p):
    """fp32 or bf16 pool (torch or numpy uint16 bits) as float64 numpy."""
    if isinstance(p, torch.Tensor):
        return p.float().cpu().numpy().astype(np.float64)
    if p.dtype == np.uint16:
        return (p.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return p.astype(np.float64)


def check_pool(pool_after, pool_before, ref_pool, written, errs, label="pool"):
    """Written rows within S_TOL of the oracle; all other rows bit-identical
    to their contents before the call."""
    written = np.flatnonzero(np.asarray(written))
    tol = S_TOL_BF16 if pool_after.dtype == torch.bfloat16 else S_TOL
    keep = torch.ones(pool_after.shape[0], dtype=torch.bool, device=pool_after.device)
    if len(written):
        w = torch.as_tensor(written, device=pool_after.device)
        keep[w] = False
        got = _pool_f64(pool_after[w])
        assert np.isfinite(got).all(), "%s: non-finite written state" % label
        e = rel_fro_rows(got, _pool_f64(ref_pool[written]))
        errs.state = max(errs.state, float(e.max()))
        assert e.max() <= tol, "%s: state rel-fro %.4g > %g (row %d)" % (
            label, e.max(), tol, written[np.unravel_index(e.argmax(), e.shape)[0]])
    assert bits_equal(pool_after[keep], pool_before[keep]), "%s: a row outside the write set changed" % label


def prefill_paged_both(call, pool_gpu, pool_ora, errs, use_slots=False, scale=SCALE):
    """One paged prefill call on the GPU and in the oracle; compares
    everything.  pool_gpu (device) and pool_ora (host) are updated in place.
    The call runs twice: with an error word (the kernels built with the device
    checks), compared with the oracle, and without one (the kernels built
    without them, the ones a caller without an error word gets), which must give
    the same bits."""
    dev = lambda t: t.cuda().contiguous()
    cu, ip, pi, lpl = dev(call.cu_seqlens), dev(call.page_indptr), dev(call.page_indices), dev(call.last_page_len)
    slots = gdn.gdn_paged_prefill_slots(cu, ip, pi, lpl, call.page_size)
    ref_slots = oracle.prefill_slots(i32(call.cu_seqlens), i32(call.page_indptr), i32(call.page_indices),
                                     i32(call.last_page_len), call.page_size)
    for k, v in ref_slots.items():
        assert (slots[k].cpu().numpy() == v).all(), "slot %s differs" % k
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = pool_gpu.clone()
    pool_fast = pool_gpu.clone()
    o = gdn.gdn_chunk_gated_delta_rule_paged(dev(call.q), dev(call.k), dev(call.v), dev(call.g), dev(call.beta),
                                             cu, pool_gpu, pi, ip, call.page_size, lpl, scale=scale,
                                             slots=slots if use_slots else None, err_word=err)
    o_fast = gdn.gdn_chunk_gated_delta_rule_paged(dev(call.q), dev(call.k), dev(call.v), dev(call.g), dev(call.beta),
                                                  cu, pool_fast, pi, ip, call.page_size, lpl, scale=scale,
                                                  slots=slots if use_slots else None)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "device error word %#x" % int(err.item())
    assert torch.equal(o.view(torch.int16), o_fast.view(torch.int16)), "outputs differ without the error word"
    assert bits_equal(pool_gpu, pool_fast), "pool differs without the error word"
    del pool_fast
    o_ref, written = oracle.chunk_gated_delta_rule_paged(
        bf16_bits(call.q), bf16_bits(call.k), bf16_bits(call.v), f32(call.g), f32(call.beta), i32(call.cu_seqlens),
        pool_ora, i32(call.page_indices), i32(call.page_indptr), call.page_size, i32(call.last_page_len), scale)
    check_o(o, o_ref, errs)
    check_pool(pool_gpu, before, pool_ora, written, errs)
    return o, written


def decode_paged_both(call, pool_gpu, pool_ora, errs, use_slots=False, scale=SCALE):
    dev = lambda t: t.cuda().contiguous()
    ip, pi, lpl = dev(call.page_indptr), dev(call.page_indices), dev(call.last_page_len)
    slots = gdn.gdn_paged_decode_slots(ip, pi, lpl)
    ref_slots = oracle.decode_slots(i32(call.page_indptr), i32(call.page_indices), i32(call.last_page_len),
                                    call.page_size)
    for k, v in ref_slots.items():
        assert (slots[k].cpu().numpy() == v).all(), "slot %s differs" % k
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = pool_gpu.clone()
    o = gdn.gdn_gated_delta_rule_decode_paged(dev(call.q), dev(call.k), dev(call.v), dev(call.g), dev(call.beta),
                                              pool_gpu, pi, ip, lpl, scale=scale,
                                              slots=slots if use_slots else None, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "device error word %#x" % int(err.item())
    o_ref, written = oracle.gated_delta_rule_decode_paged(
        bf16_bits(call.q), bf16_bits(call.k), bf16_bits(call.v), f32(call.g), f32(call.beta), pool_ora,
        i32(call.page_indices), i32(call.page_indptr), i32(call.last_page_len), call.page_size, scale)
    check_o(o, o_ref, errs)
    check_pool(pool_gpu, before, pool_ora, written, errs)
    return o, written
