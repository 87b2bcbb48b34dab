"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import gated_deltanet_paged_gb300 as gdn
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "gdn_paged.h")


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|void|const char \*)\s*(gdn_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared()
    for n in ("gdn_paged_prefill_slots", "gdn_paged_decode_slots", "gdn_chunk_gated_delta_rule",
              "gdn_chunk_gated_delta_rule_paged", "gdn_gated_delta_rule_decode_paged",
              "gdn_prefill_workspace_bytes", "gdn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(gdn.LIB_PATH if gdn.library() else None)
    for n in declared():
        assert hasattr(lib, n), n


def test_status_strings_and_workspace():
    lib = gdn.library()
    for code in (0, -1, -2, -3):
        assert lib.gdn_status_string(code) and lib.gdn_status_string(code) != b"unknown status"
    assert lib.gdn_status_string(-99) == b"unknown status"
    # 16 bytes per chunk slot (padded to 1 KB) + per (slot, head) a 64 x 64 and a 64 x 128
    # fp16 tile; slots = T / 64 + 2 S + 2
    slots = 100000 // 64 + 2 * 64 + 2
    assert lib.gdn_prefill_workspace_bytes(64, 100000, 32) == (slots * 16 + 16 + 1023) // 1024 * 1024 + slots * 32 * 24576
    assert lib.gdn_prefill_workspace_bytes(-1, 10, 2) == 0


FAKE = 0x10000  # a 16-byte aligned non-null address; never dereferenced by the host checks below


def test_slot_calls_reject_bad_arguments():
    lib = gdn.library()
    p = FAKE
    assert lib.gdn_paged_prefill_slots(p, p, p, p, 4, 100, p, p, p, p, None) == -1  # page_size % 64
    assert lib.gdn_paged_prefill_slots(p, p, p, p, 4, 0, p, p, p, p, None) == -1
    assert lib.gdn_paged_prefill_slots(None, p, p, p, 4, 64, p, p, p, p, None) == -1
    assert lib.gdn_paged_prefill_slots(p, p, p, p, -1, 64, p, p, p, p, None) == -1
    assert lib.gdn_paged_prefill_slots(p, p, p, p, 0, 64, p, p, p, p, None) == 0  # empty batch: no launch
    assert lib.gdn_paged_decode_slots(p, None, p, 3, p, p, None) == -1
    assert lib.gdn_paged_decode_slots(p, p, p, 0, p, p, None) == 0


def _chunk(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, o=FAKE, cu=FAKE, S=2, T=10, H=2, K=128, V=128, scale=0.0,
             init=None, si=None, out=None, osi=None, ck=None, cki=None, ccs=None, pl=None, N=0, stride=0,
             ws=FAKE, wsb=1 << 40, err=None)
    a.update(kw)
    return lib.gdn_chunk_gated_delta_rule(a["q"], a["k"], a["v"], a["g"], a["beta"], a["o"], a["cu"], a["S"],
                                          a["T"], a["H"], a["K"], a["V"], a["scale"], a["init"], a["si"],
                                          a["out"], a["osi"], a["ck"], a["cki"], a["ccs"], a["pl"], a["N"],
                                          a["stride"], a["ws"], a["wsb"], a["err"], None)


def test_prefill_rejects_bad_arguments():
    lib = gdn.library()
    assert _chunk(lib, K=64) == -2
    assert _chunk(lib, V=256) == -2
    assert _chunk(lib, H=0) == -1
    assert _chunk(lib, q=None) == -1
    assert _chunk(lib, q=FAKE + 8) == -1                      # q not 16-byte aligned
    assert _chunk(lib, init=FAKE, stride=2 * 128 * 128) == -1  # pool without read rows
    assert _chunk(lib, ck=FAKE, cki=FAKE, stride=2 * 128 * 128) == -1  # checkpoint arrays partly given
    ck = dict(ck=FAKE, cki=FAKE, ccs=FAKE, stride=2 * 128 * 128)
    assert _chunk(lib, **ck, pl=FAKE, N=0) == -1               # N must be > 0
    assert _chunk(lib, **ck, pl=FAKE, N=96) == -1              # N must be a multiple of 64
    assert _chunk(lib, **ck, N=128) == -1                      # prefix_lens required
    assert _chunk(lib, **dict(ck, stride=100), pl=FAKE, N=128) == -1  # stride < H*V*K
    assert _chunk(lib, S=0) == 0                               # nothing to do
    assert _chunk(lib, T=0) == 0
    need = lib.gdn_prefill_workspace_bytes(2, 10, 2)
    assert _chunk(lib, ws=None) == -1                          # workspace required
    assert _chunk(lib, wsb=need - 1) == -1                     # too small
    assert _chunk(lib, ws=FAKE + 8, wsb=need) == -1            # not 16-byte aligned


def test_general_call_index_and_state_types_are_checked():
    lib = gdn.library()

    def ex(sd=0, xd=0, **kw):
        a = dict(init=FAKE, si=FAKE, out=None, osi=None, stride=2 * 128 * 128)
        a.update(kw)
        return lib.gdn_chunk_gated_delta_rule_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 0, 2, 128, 128, 0.0,
                                                 a["init"], a["si"], a["out"], a["osi"], None, None, None, None, 0,
                                                 a["stride"], sd, xd, FAKE, 1 << 40, None, None)
    assert ex() == 0 and ex(xd=1) == 0 and ex(sd=1) == 0  # T = 0: checks pass, nothing to do
    assert ex(xd=2) == -1 and ex(xd=-1) == -1                # unknown index type
    assert ex(sd=2) == -1                                    # unknown state type
    assert ex(xd=1, si=FAKE + 4) == -1                       # int64 slots must be 8-byte aligned
    assert ex(xd=0, si=FAKE + 4) == 0                        # int32 slots: 4 bytes
    assert ex(xd=0, si=FAKE + 2) == -1
    assert ex(sd=1, stride=2 * 128 * 128 + 4) == -1          # bf16 rows: stride a multiple of 8
    assert ex(sd=0, stride=2 * 128 * 128 + 4) == 0           # fp32 rows: a multiple of 4


def test_paged_calls_reject_bad_arguments():
    lib = gdn.library()
    p = FAKE
    f = lib.gdn_chunk_gated_delta_rule_paged
    big = 1 << 40
    assert f(p, p, p, p, p, p, p, 1, 10, 2, 128, 128, 0.0, p, 8, p, p, 96, p, None, p, big, None, None) == -1
    assert f(p, p, p, p, p, p, p, 1, 10, 2, 128, 128, 0.0, None, 8, p, p, 64, p, None, p, big, None, None) == -1
    assert f(p, p, p, p, p, p, p, 1, 10, 2, 128, 64, 0.0, p, 8, p, p, 64, p, None, p, big, None, None) == -2
    assert f(p, p, p, p, p, p, p, 1, 10, 2, 128, 128, 0.0, p, 0, p, p, 64, p, None, p, big, None, None) == -1
    assert f(p, p, p, p, p, p, p, 1, 10, 2, 128, 128, 0.0, p, 8, p, p, 64, p, None, None, 0, None, None) == -1
    d = lib.gdn_gated_delta_rule_decode_paged
    assert d(p, p, p, p, p, p, 4, 2, 128, 128, 0.0, p, 8, None, p, p, None, None, None) == -1
    assert d(p, p, p, p, p, p, 4, 2, 96, 128, 0.0, p, 8, p, p, p, None, None, None) == -2
    assert d(p, p, p, p, p, p, 0, 2, 128, 128, 0.0, p, 8, p, p, p, None, None, None) == 0


def test_binding_has_no_fallback_without_gpu():
    """The Python entry points go through the CUDA library only; on a
    machine without a GPU they raise instead of computing anything."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    t = torch.zeros(4, dtype=torch.int32)
    with pytest.raises((ValueError, RuntimeError)):
        gdn.gdn_paged_decode_slots(t, t, t)


def test_pool_row_calls_reject_bad_arguments():
    """Host-side checks of the row utilities (no device work is queued)."""
    lib = gdn.library()
    fake = ctypes.c_void_p(16)  # never dereferenced: every case below fails a host check first
    rows = ctypes.c_void_p(32)
    row = 32 * 128 * 128 * 4
    assert lib.gdn_pool_copy_rows(fake, row + 8, row + 16, rows, rows, 1, 4, None, None) == -1  # row bytes % 16
    assert lib.gdn_pool_copy_rows(fake, row, row - 16, rows, rows, 1, 4, None, None) == -1      # stride < row
    assert lib.gdn_pool_copy_rows(fake, row, row, None, rows, 1, 4, None, None) == -1           # no sources
    assert lib.gdn_pool_copy_rows(None, row, row, rows, rows, 1, 4, None, None) == -1           # no pool
    assert lib.gdn_pool_copy_rows(ctypes.c_void_p(24), row, row, rows, rows, 1, 4, None, None) == -1  # misaligned
    assert lib.gdn_pool_zero_rows(fake, row, row, rows, -1, 4, None, None) == -1                 # n < 0
    assert lib.gdn_pool_zero_rows(fake, row, row, rows, 1, 0, None, None) == -1                  # no rows in pool
    assert lib.gdn_pool_zero_rows(fake, row, row, rows, 0, 4, None, None) == 0                   # nothing to do
