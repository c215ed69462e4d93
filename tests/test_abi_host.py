"""The C-ABI library loads and exports what include/gdn.h declares; host-side
argument checks return their codes before any GPU work (CPU only)."""

import ctypes
import os
import re

import pytest

from hybrid_linear_attention_prefill_gb300 import build as B
from hybrid_linear_attention_prefill_gb300 import gdn

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return gdn.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(gdn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_names():
    assert sorted(gdn.EXPORTED) == declared_functions()


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    raw = ctypes.CDLL(B.LIB)
    for name in declared_functions():
        getattr(raw, name)


def test_abi_version_matches_header(lib):
    m = re.search(r"#define GDN_ABI_VERSION (\d+)", open(HEADER).read())
    assert gdn.gdn_abi_version() == int(m.group(1))


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, 7):
        assert isinstance(gdn.gdn_strerror(code), str) and gdn.gdn_strerror(code)


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced


def call(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, cu_seqlens=None, init_state=None,
             out=FAKE, final_state=None, B=1, T=64, Hk=1, Hv=1, dk=128, dv=128, stream=0)
    a.update(kw)
    return gdn.gdn_prefill(**a)


@pytest.mark.parametrize("kw", [dict(B=-1), dict(T=-5), dict(Hk=0), dict(Hv=3, Hk=2), dict(dk=48),
                                dict(dv=256), dict(q=None), dict(out=None), dict(beta=None)])
def test_bad_arguments_rejected(lib, kw):
    assert call(**kw) == gdn.GDN_ERR_ARG


@pytest.mark.parametrize("name", ["q", "k", "v", "g", "beta", "out", "init_state", "final_state",
                                  "cu_seqlens"])
def test_misaligned_pointer_rejected(lib, name):
    assert call(**{name: FAKE + 4}) == gdn.GDN_ERR_ALIGN


def test_nothing_to_do(lib):
    assert call(B=0) == gdn.GDN_OK
    assert call(T=0) == gdn.GDN_OK  # no tokens and no final state requested


def test_host_entry_rejects_bad_arguments(lib):
    assert gdn.gdn_prefill_host(None, None, None, None, None, None, None, None, None,
                                1, 4, 1, 1, 128, 128, 0) == gdn.GDN_ERR_ARG
    assert gdn.gdn_prefill_host(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None,
                                1, 4, 2, 3, 128, 128, 0) == gdn.GDN_ERR_ARG


def test_workspace_bytes(lib):
    per = 2 * 64 * 64 * 2   # Tm + PT per (chunk slot, value head)
    norms = 2 * 64 * 4      # inverse q/k norms per (chunk slot, key head)
    kq128, kq64 = 2 * 16384, 16384  # fp16 [K; Q] image per (chunk slot, key head), by dk
    assert gdn.gdn_workspace_bytes(1, 4096, 16, 32, 128, 128, 0) == 512 + 64 * 32 * per + 64 * 16 * (norms + kq128)
    assert gdn.gdn_workspace_bytes(2, 100, 1, 1, 32, 32, 1) == 512 + (2 + 2) * (per + norms + kq64)
    assert gdn.gdn_workspace_bytes(1, 64, 1, 1, 64, 32, 0) == 512 + per + norms + kq64
    assert gdn.gdn_workspace_bytes(1, 10, 2, 3, 128, 128, 0) == 0


def ws_call(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, cu_seqlens=None, init_state=None,
             out=FAKE, final_state=None, B=1, T=64, Hk=1, Hv=1, dk=128, dv=128,
             workspace=FAKE, workspace_bytes=1 << 30, stream=0)
    a.update(kw)
    return gdn.gdn_prefill_ws(**a)


def test_caller_workspace_checks(lib):
    assert ws_call(workspace=None) == gdn.GDN_ERR_ARG
    assert ws_call(workspace=FAKE + 16) == gdn.GDN_ERR_ALIGN  # needs 256-byte alignment
    need = gdn.gdn_workspace_bytes(1, 64, 1, 1, 128, 128, 0)
    assert ws_call(workspace_bytes=need - 1) == gdn.GDN_ERR_SCRATCH
    assert ws_call(B=0) == gdn.GDN_OK and ws_call(dk=48) == gdn.GDN_ERR_ARG


def test_decode_argument_checks(lib):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state=FAKE, out=FAKE, B=2, Hk=1, Hv=2, dk=128,
             dv=128, stream=0)
    assert gdn.gdn_decode(**{**a, "state": None}) == gdn.GDN_ERR_ARG
    assert gdn.gdn_decode(**{**a, "Hk": 2, "Hv": 3}) == gdn.GDN_ERR_ARG
    assert gdn.gdn_decode(**{**a, "out": FAKE + 2}) == gdn.GDN_ERR_ALIGN
    assert gdn.gdn_decode(**{**a, "B": 0}) == gdn.GDN_OK


def test_prefill_ex_rejects_unknown_flags(lib):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, cu_seqlens=None, init_state=None,
             out=FAKE, final_state=None, B=1, T=64, Hk=1, Hv=1, dk=128, dv=128, stream=0)
    for bad in (8, 1 << 20, 1 << 31, gdn.GDN_FLAG_TWO_LEVEL | gdn.GDN_FLAG_ONE_LEVEL,
                gdn.GDN_FLAG_SLICE32 | gdn.GDN_FLAG_SLICE64, gdn.GDN_FLAG_SLICE16 | gdn.GDN_FLAG_SLICE32,
                gdn.GDN_FLAG_SLICE16 | gdn.GDN_FLAG_SLICE64):
        assert gdn.gdn_prefill_ex(**a, flags=bad) == gdn.GDN_ERR_ARG
    # 64 state rows per CTA need dv to be a multiple of 64
    assert gdn.gdn_prefill_ex(**{**a, "dk": 32, "dv": 32}, flags=gdn.GDN_FLAG_SLICE64) == gdn.GDN_ERR_ARG
    for ok in (gdn.GDN_FLAG_L2NORM_QK, gdn.GDN_FLAG_TWO_LEVEL | gdn.GDN_FLAG_SEGMENTS(5), gdn.GDN_FLAG_ONE_LEVEL,
               gdn.GDN_FLAG_SLICE16, gdn.GDN_FLAG_SLICE32, gdn.GDN_FLAG_SLICE64,
               gdn.GDN_FLAG_SLICE64 | gdn.GDN_FLAG_L2NORM_QK, gdn.GDN_FLAG_WIDE_RANGE,
               gdn.GDN_FLAG_WIDE_RANGE | gdn.GDN_FLAG_SLICE16 | gdn.GDN_FLAG_L2NORM_QK):
        assert gdn.gdn_prefill_ex(**{**a, "B": 0}, flags=ok) == gdn.GDN_OK


def test_segment_flag_encoding():
    """GDN_FLAG_SEGMENTS(n) occupies bits 8..15, as the header defines it."""
    hdr = open(HEADER).read()
    assert "#define GDN_FLAG_SEGMENTS(n) ((((unsigned)(n)) & 0xffu) << 8)" in hdr
    assert gdn.GDN_FLAG_SEGMENTS(3) == 3 << 8 and gdn.GDN_FLAG_SEGMENTS(255) == 0xFF00
    assert (gdn.GDN_FLAG_TWO_LEVEL, gdn.GDN_FLAG_ONE_LEVEL) == (2, 4)
    assert "#define GDN_FLAG_SLICE32 0x10000u" in hdr and "#define GDN_FLAG_SLICE64 0x20000u" in hdr
    assert "#define GDN_FLAG_SLICE16 0x40000u" in hdr
    assert (gdn.GDN_FLAG_SLICE16, gdn.GDN_FLAG_SLICE32, gdn.GDN_FLAG_SLICE64) == (0x40000, 0x10000, 0x20000)
    assert "#define GDN_FLAG_WIDE_RANGE 0x80000u" in hdr and gdn.GDN_FLAG_WIDE_RANGE == 0x80000
    assert "#define GDN_STATUS_NONFINITE_STATE 16" in hdr and gdn.GDN_STATUS_NONFINITE_STATE == 16
    assert "#define GDN_STATUS_SMALL_STATE 32" in hdr and gdn.GDN_STATUS_SMALL_STATE == 32
    assert "#define GDN_STATIC_SCRATCH_BYTES (128u << 20)" in hdr and gdn.GDN_STATIC_SCRATCH_BYTES == 128 << 20


def test_allocation_failure_hook_counts_down(lib):
    """gdn_debug_fail_allocations holds a count of upcoming failures and returns the one it replaces."""
    assert gdn.gdn_debug_fail_allocations(2) == 0
    assert gdn.gdn_debug_fail_allocations(5) == 2
    assert gdn.gdn_debug_fail_allocations(-1) == 5   # negative: off
    assert gdn.gdn_debug_fail_allocations(0) == 0
