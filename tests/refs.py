"""Independent float64 formulations used to pin the oracle (tests only).

Neither shares code with ``oracle/gdn_oracle.c``:

* ``brute_force`` forms the full dk x dk transition matrix each token,
  S <- alpha S (I - beta k k^T) + beta v k^T, exactly as the gated delta rule
  is written, and multiplies matrices with numpy.
* ``chunked`` is the chunk-wise (WY / UT-transform) reformulation of the same
  recurrence.  Within a chunk that starts from state S0, with
  gamma = inclusive cumsum of g, Gamma[r, i] = exp(gamma_r - gamma_i) (i <= r):
      A   = strict_lower(diag(beta) (K K^T) * Gamma)
      Tm  = (I + A)^-1
      U   = Tm (diag(beta) V - diag(beta e^gamma) K S0^T)
      O   = scale (diag(e^gamma) Q S0^T + lower_incl((Q K^T) * Gamma) U)
      S1  = e^{gamma_last} S0 + U^T diag(e^{gamma_last - gamma}) K
  It is exact in real arithmetic for any chunk length, so agreement with the
  token loop pins both the oracle and the algebra the CUDA kernels use.
"""

from __future__ import annotations

import numpy as np


def _bounds(Ttot, B, cu):
    if cu is None:
        T = Ttot // B if B else 0
        return [(b * T, (b + 1) * T) for b in range(B)]
    return [(int(cu[b]), int(cu[b + 1])) for b in range(len(cu) - 1)]


def brute_force(q, k, v, g, beta, cu=None, init=None, B=1):
    Ttot, Hk, dk = q.shape
    Hv, dv = v.shape[1:]
    bounds = _bounds(Ttot, B, cu)
    out = np.zeros((Ttot, Hv, dv))
    fin = np.zeros((len(bounds), Hv, dv, dk))
    eye = np.eye(dk)
    for n, (s, e) in enumerate(bounds):
        for h in range(Hv):
            hk = h // (Hv // Hk)
            S = np.zeros((dv, dk)) if init is None else init[n, h].astype(np.float64).copy()
            for t in range(s, e):
                kt, qt, vt = k[t, hk], q[t, hk], v[t, h]
                M = np.exp(g[t, h]) * (eye - beta[t, h] * np.outer(kt, kt))
                S = S @ M + beta[t, h] * np.outer(vt, kt)
                out[t, h] = S @ qt / np.sqrt(dk)
            fin[n, h] = S
    return out, fin


def chunked(q, k, v, g, beta, cu=None, init=None, B=1, C=64):
    Ttot, Hk, dk = q.shape
    Hv, dv = v.shape[1:]
    bounds = _bounds(Ttot, B, cu)
    scale = 1.0 / np.sqrt(dk)
    out = np.zeros((Ttot, Hv, dv))
    fin = np.zeros((len(bounds), Hv, dv, dk))
    for n, (s, e) in enumerate(bounds):
        for h in range(Hv):
            hk = h // (Hv // Hk)
            S = np.zeros((dv, dk)) if init is None else init[n, h].astype(np.float64).copy()
            for c0 in range(s, e, C):
                c1 = min(c0 + C, e)
                K, Q, V = k[c0:c1, hk], q[c0:c1, hk], v[c0:c1, h]
                bt = beta[c0:c1, h]
                gam = np.cumsum(g[c0:c1, h])
                D = gam[:, None] - gam[None, :]
                low = np.tril(np.ones_like(D, dtype=bool))
                Gam = np.where(low, np.exp(np.where(low, D, 0.0)), 0.0)
                A = np.tril(bt[:, None] * (K @ K.T) * Gam, -1)
                Tm = np.linalg.inv(np.eye(c1 - c0) + A)
                U = Tm @ (bt[:, None] * V - (bt * np.exp(gam))[:, None] * (K @ S.T))
                P = (Q @ K.T) * Gam
                out[c0:c1, h] = scale * (np.exp(gam)[:, None] * (Q @ S.T) + P @ U)
                S = np.exp(gam[-1]) * S + U.T @ (np.exp(gam[-1] - gam)[:, None] * K)
            fin[n, h] = S
    return out, fin
