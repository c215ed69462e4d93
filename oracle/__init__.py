"""Float64 CPU oracle for the Gated DeltaNet prefill -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never uses it.

``prefill`` runs the plain token-by-token recurrence written in
``gdn_oracle.c`` (float64, threads over (sequence, value head) pairs).  The
library is compiled with gcc on first use (``build()``), into ``_build/``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc -O2 (no fast-math); returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-fPIC", "-shared", "-std=c11",
           "-Wall", "-Wextra", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            lib.gdn_oracle_prefill.argtypes = [dp, dp, dp, dp, dp, ip, dp, dp, dp] + [ctypes.c_int] * 7
            lib.gdn_oracle_prefill.restype = ctypes.c_int
            lib.gdn_oracle_num_cpus.argtypes = []
            lib.gdn_oracle_num_cpus.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_cpus() -> int:
    return int(_load().gdn_oracle_num_cpus())


def _dptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def prefill(q, k, v, g, beta, cu_seqlens=None, init_state=None, *, B=None, T=None,
            want_final=True, nthreads=0):
    """Run the oracle.

    q, k: float64 [Ttot, Hk, dk]; v: float64 [Ttot, Hv, dv]; g, beta: float64
    [Ttot, Hv]; cu_seqlens: int32 [B+1] or None; init_state: float64
    [B, Hv, dv, dk] or None.  Without cu_seqlens, B defaults to 1 and T to Ttot.
    Returns (out [Ttot, Hv, dv], final_state [B, Hv, dv, dk] or None), float64.
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    g = np.ascontiguousarray(g, dtype=np.float64)
    beta = np.ascontiguousarray(beta, dtype=np.float64)
    Ttot, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    assert k.shape == q.shape and v.shape[0] == Ttot
    assert g.shape == (Ttot, Hv) and beta.shape == (Ttot, Hv)
    cu_p = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        B = len(cu) - 1
        T = Ttot
        assert cu[0] == 0 and cu[-1] == Ttot and np.all(np.diff(cu) >= 0)
        cu_p = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    else:
        if B is None:
            B = 1
        if T is None:
            T = Ttot // B if B else 0
        assert B * T == Ttot
    init = None
    if init_state is not None:
        init = np.ascontiguousarray(init_state, dtype=np.float64)
        assert init.shape == (B, Hv, dv, dk)
    out = np.zeros((Ttot, Hv, dv), dtype=np.float64)
    fin = np.zeros((B, Hv, dv, dk), dtype=np.float64) if want_final else None
    rc = _load().gdn_oracle_prefill(
        _dptr(q), _dptr(k), _dptr(v), _dptr(g), _dptr(beta), cu_p, _dptr(init),
        _dptr(out), _dptr(fin), int(B), int(T), int(Hk), int(Hv), int(dk), int(dv),
        int(nthreads))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_prefill failed with status {rc}")
    if cu_seqlens is not None:
        cu_seqlens_keep = cu  # keep alive through the call
        del cu_seqlens_keep
    return out, fin


def prefill_inputs(inp, *, want_final=True, nthreads=0):
    """Run the oracle on a ``GdnInputs`` problem (the bf16 values, widened exactly)."""
    return prefill(inp.q64(), inp.k64(), inp.v64(), inp.g64(), inp.beta64(),
                   inp.cu_seqlens, inp.init64(), B=inp.B,
                   T=None if inp.cu_seqlens is not None else inp.T,
                   want_final=want_final, nthreads=nthreads)
