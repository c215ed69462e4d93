"""Seeded synthetic inputs for the chunked Gated DeltaNet prefill.

This module is shared by the CUDA path's tests and benchmark and by the
float64 oracle's tests.  It holds no arithmetic of the method itself: it only
draws random numbers, applies the per-token L2 normalisation that the caller
of the prefill performs upstream (the "fused norm ... QK" operation on the
"Open-Jev-27B-v1.1 native text worker" page, section "Validation and
optimization scope"), and rounds to the storage formats the library takes
(bf16 q/k/v, fp32 g/beta/state).

Workloads follow the pages' scoring setting: independent candidate prompts of
up to 4,096 tokens by default and 16,384 at most ("Open-Jev-27B-v1.1 native
text worker", sections "Prepare the checkpoint" and intro), batched as packed
variable-length sequences.

Draw order from ``numpy.random.default_rng(seed)`` (all draws fp32):
sequence lengths (packed workloads only), q, k, v, g, beta, initial state.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns uint16 bits.

    Inputs must be finite.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns exactly to float64."""
    u = (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16)
    return u.view(np.float32).astype(np.float64)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    u = (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16)
    return u.view(np.float32).copy()


def _l2_normalise(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x.astype(np.float32) ** 2, axis=-1, keepdims=True, dtype=np.float32))
    return (x / np.maximum(n, np.float32(1e-6))).astype(np.float32)


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(np.float32(0.0), x).astype(np.float32)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return (np.float32(1.0) / (np.float32(1.0) + np.exp(-x))).astype(np.float32)


@dataclasses.dataclass
class GdnInputs:
    """One prefill problem in the library's layouts.

    q, k: bf16 bits [Ttot, Hk, dk]; v: bf16 bits [Ttot, Hv, dv];
    g, beta: fp32 [Ttot, Hv]; init: fp32 [B, Hv, dv, dk] or None;
    cu_seqlens: int32 [B+1] or None (then B sequences of T tokens each).
    """

    B: int
    T: int  # tokens per sequence (dense) or total tokens (packed)
    Hk: int
    Hv: int
    dk: int
    dv: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    init: Optional[np.ndarray]
    cu_seqlens: Optional[np.ndarray]
    name: str = ""

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[0])

    def seq_bounds(self):
        """List of (start, end) token ranges, one per sequence."""
        if self.cu_seqlens is None:
            return [(b * self.T, (b + 1) * self.T) for b in range(self.B)]
        c = self.cu_seqlens
        return [(int(c[b]), int(c[b + 1])) for b in range(self.B)]

    # float64 views of exactly the values the GPU receives
    def q64(self):
        return bf16_bits_to_f64(self.q)

    def k64(self):
        return bf16_bits_to_f64(self.k)

    def v64(self):
        return bf16_bits_to_f64(self.v)

    def g64(self):
        return self.g.astype(np.float64)

    def beta64(self):
        return self.beta.astype(np.float64)

    def init64(self):
        return None if self.init is None else self.init.astype(np.float64)


def make_gdn_inputs(
    *,
    Hk: int,
    Hv: int,
    dk: int,
    dv: int,
    B: int = 1,
    T: int = 0,
    lengths=None,
    packed: bool = False,
    seed: int = 0,
    g_scale: float = 1.0,
    init_std: Optional[float] = None,
    normalize_qk: bool = True,
    name: str = "",
) -> GdnInputs:
    """Draw one seeded problem (``normalize_qk=False`` leaves q and k un-normalised).

    Dense: ``B`` sequences of ``T`` tokens (cu_seqlens None unless ``packed``).
    Packed: ``lengths`` is a list of sequence lengths, or ``("uniform", n, lo, hi)``
    to draw ``n`` lengths uniformly in [lo, hi] from the same generator first.
    """
    rng = np.random.default_rng(seed)
    if lengths is not None:
        if isinstance(lengths, tuple) and lengths and lengths[0] == "uniform":
            _, n, lo, hi = lengths
            lengths = rng.integers(lo, hi + 1, n)
        lengths = [int(x) for x in lengths]
        B = len(lengths)
        cu = np.zeros(B + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lengths)
        Ttot = int(cu[-1])
        T = Ttot
    else:
        Ttot = B * T
        cu = None
        if packed:
            cu = np.arange(B + 1, dtype=np.int32) * T
            T = Ttot
    f32 = np.float32
    q = rng.standard_normal((Ttot, Hk, dk), dtype=f32)
    k = rng.standard_normal((Ttot, Hk, dk), dtype=f32)
    if normalize_qk:  # the caller's per-token normalisation (else raw projections)
        q, k = _l2_normalise(q), _l2_normalise(k)
    v = rng.standard_normal((Ttot, Hv, dv), dtype=f32)
    g = (-_softplus(rng.standard_normal((Ttot, Hv), dtype=f32)) * f32(g_scale)).astype(f32)
    beta = _sigmoid(rng.standard_normal((Ttot, Hv), dtype=f32))
    init = None
    if init_std is not None:
        init = (rng.standard_normal((B, Hv, dv, dk), dtype=f32) * f32(init_std)).astype(f32)
    return GdnInputs(
        B=B, T=T, Hk=Hk, Hv=Hv, dk=dk, dv=dv,
        q=f32_to_bf16_bits(q), k=f32_to_bf16_bits(k), v=f32_to_bf16_bits(v),
        g=g, beta=beta, init=init, cu_seqlens=cu, name=name,
    )


# The five workloads (plus a smaller packed batch for profiling): shapes and distributions
# of independent candidate prompts (default limit 4,096 tokens, maximum 16,384).
WORKLOADS = {
    "tiny_t64_d32": dict(B=1, T=64, Hk=1, Hv=1, dk=32, dv=32),
    "t1024_h16": dict(B=1, T=1024, Hk=16, Hv=16, dk=128, dv=128),
    "t4096_hk16_hv32": dict(B=1, T=4096, Hk=16, Hv=32, dk=128, dv=128),
    "varlen32_hk16_hv32": dict(lengths=("uniform", 32, 200, 4096), Hk=16, Hv=32, dk=128, dv=128),
    "t16381_hk16_hv32_carry": dict(B=1, T=16381, Hk=16, Hv=32, dk=128, dv=128,
                                   g_scale=0.1, init_std=0.02),
    # the maximum prompt with few heads per GPU (heads split over GPUs), where the
    # chunk-sequential carry alone would leave most SMs idle
    "t16384_hk4_hv4_carry": dict(B=1, T=16384, Hk=4, Hv=4, dk=128, dv=128,
                                 g_scale=0.1, init_std=0.02),
    # the packed batch's length mix at a quarter of its candidates: small enough for a
    # many-pass profiler capture of one launch, larger than L2
    "varlen8_hk16_hv32": dict(lengths=("uniform", 8, 200, 4096), Hk=16, Hv=32, dk=128, dv=128),
}

HEADLINE = "t4096_hk16_hv32"


def workload(name: str, seed: int = 0) -> GdnInputs:
    return make_gdn_inputs(seed=seed, name=name, **WORKLOADS[name])
