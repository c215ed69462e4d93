"""Python binding of the C ABI in ``include/gdn.h`` (ctypes; argument marshalling only).

Every step of the prefill runs in the CUDA library ``libgdn.so``; this module only
turns tensors into pointers.  There is no fallback: if the library cannot be loaded
(not built, or no CUDA runtime) the calls raise.

Functions keep the C names: ``gdn_prefill``, ``gdn_prefill_host``,
``gdn_abi_version``, ``gdn_strerror``, ``gdn_last_cuda_error``,
``gdn_workspace_bytes``, ``gdn_scan_segments``, ``gdn_release_workspace``.  ``prefill`` is a convenience
wrapper that allocates the outputs with PyTorch and checks the status.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

GDN_OK = 0
GDN_ERR_ARG = -1
GDN_ERR_ALIGN = -2
GDN_ERR_ALLOC = -3
GDN_ERR_LAUNCH = -4
GDN_ERR_SCRATCH = -5
GDN_STATIC_SCRATCH_BYTES = 128 << 20
GDN_FLAG_L2NORM_QK = 1
GDN_FLAG_TWO_LEVEL = 2
GDN_FLAG_ONE_LEVEL = 4
GDN_FLAG_SLICE32 = 0x10000
GDN_FLAG_SLICE16 = 0x40000
GDN_FLAG_SLICE64 = 0x20000
GDN_FLAG_WIDE_RANGE = 0x80000
GDN_STATUS_MMA_TIMEOUT = 1
GDN_STATUS_LOAD_TIMEOUT = 2
GDN_STATUS_PREP_LOAD_TIMEOUT = 4
GDN_STATUS_BAD_CU_SEQLENS = 8
GDN_STATUS_NONFINITE_STATE = 16
GDN_STATUS_SMALL_STATE = 32


def GDN_FLAG_SEGMENTS(n: int) -> int:
    """Segment count for GDN_FLAG_TWO_LEVEL, in flag bits 8..15."""
    return (int(n) & 0xFF) << 8


EXPORTED = ("gdn_abi_version", "gdn_strerror", "gdn_last_cuda_error", "gdn_prefill",
            "gdn_prefill_host", "gdn_prefill_static", "gdn_prefill_ws", "gdn_prefill_ex", "gdn_decode",
            "gdn_set_phase_events", "gdn_workspace_bytes", "gdn_scan_segments", "gdn_release_workspace",
            "gdn_device_status", "gdn_selftest_wait_timeout", "gdn_selftest_static_wait_timeout",
            "gdn_debug_fail_allocations")

_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    def __init__(self, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        super().__init__(f"gdn status {status}: {gdn_strerror(status)}"
                         + (f" (cudaError {cuda_error})" if cuda_error else ""))


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libgdn.so (optionally building it first) and declare the signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and _build.needs_build():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "or python -m hybrid_linear_attention_prefill_gb300.build")
        lib = ctypes.CDLL(path)
        vp, fp, ip, i = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
        sig = [vp, vp, vp, fp, fp, ip, fp, vp, fp, i, i, i, i, i, i, vp]
        lib.gdn_prefill.argtypes = sig
        lib.gdn_prefill.restype = i
        lib.gdn_prefill_host.argtypes = sig
        lib.gdn_prefill_host.restype = i
        lib.gdn_prefill_static.argtypes = sig
        lib.gdn_prefill_static.restype = i
        lib.gdn_prefill_ws.argtypes = sig[:-1] + [vp, ctypes.c_size_t, vp]
        lib.gdn_prefill_ws.restype = i
        lib.gdn_prefill_ex.argtypes = sig[:-1] + [ctypes.c_uint, vp]
        lib.gdn_prefill_ex.restype = i
        lib.gdn_decode.argtypes = [vp, vp, vp, fp, fp, fp, vp, i, i, i, i, i, vp]
        lib.gdn_decode.restype = i
        lib.gdn_abi_version.argtypes = []
        lib.gdn_abi_version.restype = i
        lib.gdn_strerror.argtypes = [i]
        lib.gdn_strerror.restype = ctypes.c_char_p
        lib.gdn_last_cuda_error.argtypes = []
        lib.gdn_last_cuda_error.restype = i
        lib.gdn_workspace_bytes.argtypes = [i] * 7
        lib.gdn_workspace_bytes.restype = ctypes.c_size_t
        lib.gdn_scan_segments.argtypes = [i] * 7 + [ctypes.c_uint]
        lib.gdn_scan_segments.restype = i
        lib.gdn_set_phase_events.argtypes = [vp, vp, vp]
        lib.gdn_set_phase_events.restype = None
        lib.gdn_device_status.argtypes = [ctypes.POINTER(ctypes.c_int)]
        lib.gdn_device_status.restype = i
        lib.gdn_selftest_wait_timeout.argtypes = [i, ctypes.POINTER(ctypes.c_int)]
        lib.gdn_selftest_wait_timeout.restype = i
        lib.gdn_selftest_static_wait_timeout.argtypes = [i]
        lib.gdn_selftest_static_wait_timeout.restype = i
        lib.gdn_debug_fail_allocations.argtypes = [i]
        lib.gdn_debug_fail_allocations.restype = i
        lib.gdn_release_workspace.argtypes = []
        lib.gdn_release_workspace.restype = None
        _lib = lib
        return lib


def _ptr(x):
    """Device/host address of a tensor, array or integer (None stays NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):  # torch.Tensor
        return x.data_ptr()
    if hasattr(x, "ctypes"):  # numpy.ndarray
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)!r}")


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def gdn_abi_version() -> int:
    return load().gdn_abi_version()


def gdn_strerror(status: int) -> str:
    return load().gdn_strerror(status).decode()


def gdn_last_cuda_error() -> int:
    return load().gdn_last_cuda_error()


def gdn_workspace_bytes(B, T, Hk, Hv, dk, dv, packed) -> int:
    return load().gdn_workspace_bytes(B, T, Hk, Hv, dk, dv, int(bool(packed)))


def gdn_scan_segments(B, T, Hk, Hv, dk, dv, packed, flags=0) -> int:
    """Segments per sequence gdn_prefill(_ex) would use on the current device (1 = single-level)."""
    return load().gdn_scan_segments(B, T, Hk, Hv, dk, dv, int(bool(packed)), int(flags))


def gdn_set_phase_events(ev_begin, ev_mid, ev_end) -> None:
    """Record three CUDA events around the next gdn_prefill's kernels (handles or torch events)."""
    def h(e):
        if e is None or isinstance(e, int):
            return e
        return e.cuda_event
    load().gdn_set_phase_events(h(ev_begin), h(ev_mid), h(ev_end))


def gdn_device_status():
    """(status code, device status bits of the library workspace and the static array); clears them."""
    st = ctypes.c_int(0)
    rc = load().gdn_device_status(ctypes.byref(st))
    return rc, st.value


def gdn_selftest_wait_timeout(max_polls):
    """(status code, recorded bits) of a bounded wait that is made to run out."""
    st = ctypes.c_int(0)
    rc = load().gdn_selftest_wait_timeout(int(max_polls), ctypes.byref(st))
    return rc, st.value


def gdn_selftest_static_wait_timeout(max_polls) -> int:
    """A bounded wait made to run out, recording into gdn_prefill_static's status word."""
    return load().gdn_selftest_static_wait_timeout(int(max_polls))


def gdn_debug_fail_allocations(count) -> int:
    """Make the library's next `count` device allocations fail; returns the pending count."""
    return load().gdn_debug_fail_allocations(int(count))


def gdn_release_workspace() -> None:
    load().gdn_release_workspace()


def gdn_prefill(q, k, v, g, beta, cu_seqlens, init_state, out, final_state,
                B, T, Hk, Hv, dk, dv, stream=None) -> int:
    """Call the C entry point on device buffers; returns the status code."""
    return load().gdn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                              _ptr(init_state), _ptr(out), _ptr(final_state),
                              int(B), int(T), int(Hk), int(Hv), int(dk), int(dv), _stream(stream))


def gdn_prefill_host(q, k, v, g, beta, cu_seqlens, init_state, out, final_state,
                     B, T, Hk, Hv, dk, dv, stream=None) -> int:
    """Call the C entry point on host buffers (synchronises the stream); returns the status."""
    return load().gdn_prefill_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                   _ptr(init_state), _ptr(out), _ptr(final_state),
                                   int(B), int(T), int(Hk), int(Hv), int(dk), int(dv), _stream(stream))


def gdn_prefill_static(q, k, v, g, beta, cu_seqlens, init_state, out, final_state,
                       B, T, Hk, Hv, dk, dv, stream=None) -> int:
    """Call the allocation-free entry point (fixed device scratch); returns the status."""
    return load().gdn_prefill_static(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                     _ptr(init_state), _ptr(out), _ptr(final_state),
                                     int(B), int(T), int(Hk), int(Hv), int(dk), int(dv), _stream(stream))


def gdn_prefill_ws(q, k, v, g, beta, cu_seqlens, init_state, out, final_state,
                   B, T, Hk, Hv, dk, dv, workspace, workspace_bytes, stream=None) -> int:
    """Call the caller-workspace entry point (no allocation, no host sync); returns the status."""
    return load().gdn_prefill_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                 _ptr(init_state), _ptr(out), _ptr(final_state),
                                 int(B), int(T), int(Hk), int(Hv), int(dk), int(dv),
                                 _ptr(workspace), int(workspace_bytes), _stream(stream))


def gdn_prefill_ex(q, k, v, g, beta, cu_seqlens, init_state, out, final_state,
                   B, T, Hk, Hv, dk, dv, flags, stream=None) -> int:
    """gdn_prefill with option flags (GDN_FLAG_*); returns the status."""
    return load().gdn_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                 _ptr(init_state), _ptr(out), _ptr(final_state),
                                 int(B), int(T), int(Hk), int(Hv), int(dk), int(dv), int(flags),
                                 _stream(stream))


def gdn_decode(q, k, v, g, beta, state, out, B, Hk, Hv, dk, dv, stream=None) -> int:
    """One token per sequence, state updated in place; returns the status."""
    return load().gdn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(out),
                             int(B), int(Hk), int(Hv), int(dk), int(dv), _stream(stream))


def check(status: int) -> None:
    if status != GDN_OK:
        raise GdnError(status, gdn_last_cuda_error())


def prefill(q, k, v, g, beta, cu_seqlens=None, init_state=None, *, B=None, want_final=True, stream=None):
    """Allocate outputs and run ``gdn_prefill`` on CUDA tensors.

    q, k: bf16 [Ttot, Hk, dk]; v: bf16 [Ttot, Hv, dv]; g, beta: fp32 [Ttot, Hv];
    cu_seqlens: int32 [B+1] or None; init_state: fp32 [B, Hv, dv, dk] or None.
    Returns (out bf16 [Ttot, Hv, dv], final_state fp32 [B, Hv, dv, dk] or None).
    """
    import torch

    Ttot, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    if cu_seqlens is not None:
        B = cu_seqlens.numel() - 1
        T = Ttot
    else:
        B = 1 if B is None else B
        T = Ttot // B if B else 0
    out = torch.empty((Ttot, Hv, dv), dtype=torch.bfloat16, device=q.device)
    fin = torch.empty((B, Hv, dv, dk), dtype=torch.float32, device=q.device) if want_final else None
    check(gdn_prefill(q, k, v, g, beta, cu_seqlens, init_state, out, fin, B, T, Hk, Hv, dk, dv, stream))
    return out, fin
