"""The operand format of the chunk products, checked in float64 (CPU only).

The state carry's tensor-core products take 16-bit operands and accumulate in fp32; the fp32
state and every other quantity stay wide.  This model runs the same chunk-wise recurrence as the
kernels (the WY / UT-transform form pinned in ``refs.chunked``) in float64 and rounds exactly
where the kernels round an operand: Tm and PT = P Tm (P and Tm rounded for that product), the
state S before [X; Y] = [K; Q] S^T, and R before it is multiplied.  The wide-range state carry
then forms [U; Z] = [Tm; PT] R and dS^T = K^T diag(d) U with diag(d) U rounded (three rounds);
the default one forms dS^T = W R with W = K^T diag(d) Tm, rounding diag(d) Tm and W, and
Z = PT R (two rounds).  The errors are measured against the float64 oracle on a stress case (no
decay, beta = 0.999, so nothing is forgotten and rounding accumulates over the whole sequence).

What it pins:
* fp16 single operands everywhere (the default state carry) stay well inside the tolerances
  and below the bf16 hi / lo design (bf16 Tm and PT, state-side operands as bf16 hi + lo pairs,
  the wide-range state carry);
* bf16 single state-side operands would not meet the final-state tolerance, which is why a
  single operand has to be fp16 (or a bf16 hi / lo pair).
"""

import numpy as np
import pytest

from hybrid_linear_attention_prefill_gb300.inputs import bf16_bits_to_f64, make_gdn_inputs

OUT_TOL = 1e-2
STATE_TOL = 2e-3


def _bf16(x):
    x = np.asarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16  # round to nearest even
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def _round(x, fmt):
    if fmt == "f64":
        return np.asarray(x, dtype=np.float64)
    if fmt == "fp16":
        return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float64)
    if fmt == "bf16":
        return _bf16(x)
    if fmt == "hilo":  # bf16 hi part plus the bf16 rounding of the fp32 remainder
        x32 = np.asarray(x, dtype=np.float32).astype(np.float64)
        hi = _bf16(x32)
        return hi + _bf16(x32 - hi)
    raise ValueError(fmt)


def chunked_rounded(inp, fmt_t, fmt_state, two_round=False, C=64):
    """Outputs and final states of the chunk recurrence with the kernels' operand roundings:
    fmt_t for P, Tm, PT and diag(d) Tm, fmt_state for S, R and diag(d) U (three rounds) or W
    (two rounds)."""
    q, k, v = bf16_bits_to_f64(inp.q), bf16_bits_to_f64(inp.k), bf16_bits_to_f64(inp.v)
    g, beta = inp.g.astype(np.float64), inp.beta.astype(np.float64)
    Ttot, Hk, dk = q.shape
    Hv, dv = v.shape[1:]
    scale = 1.0 / np.sqrt(dk)
    out = np.zeros((Ttot, Hv, dv))
    fin = np.zeros((inp.B, Hv, dv, dk))
    for n, (s, e) in enumerate(inp.seq_bounds()):
        for h in range(Hv):
            hk = h // (Hv // Hk)
            S = np.zeros((dv, dk)) if inp.init is None else inp.init[n, h].astype(np.float64).copy()
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
                P = (Q @ K.T) * Gam
                PT = _round(P, fmt_t) @ _round(Tm, fmt_t)
                Tm_r, PT_r = _round(Tm, fmt_t), _round(PT, fmt_t)
                S_op = _round(S, fmt_state)
                X, Y = K @ S_op.T, Q @ S_op.T
                R = bt[:, None] * V - (bt * np.exp(gam))[:, None] * X
                R_op = _round(R, fmt_state)
                Z = PT_r @ R_op
                out[c0:c1, h] = scale * (np.exp(gam)[:, None] * Y + Z)
                d = np.exp(gam[-1] - gam)
                if two_round:
                    W = _round(K.T @ _round(d[:, None] * Tm_r, fmt_t), fmt_state)
                    S = np.exp(gam[-1]) * S + (W @ R_op).T
                else:
                    dU = d[:, None] * (Tm_r @ R_op)
                    S = np.exp(gam[-1]) * S + _round(dU, fmt_state).T @ K
                if fmt_state != "f64":
                    S = S.astype(np.float32).astype(np.float64)  # the state is carried in fp32
            fin[n, h] = S
    return out, fin


@pytest.fixture(scope="module")
def stress():
    import oracle

    inp = make_gdn_inputs(B=1, T=300, Hk=1, Hv=2, dk=128, dv=128, seed=12, init_std=0.1)
    inp.g[:] = 0.0
    inp.beta[:] = 0.999
    return inp, oracle.prefill_inputs(inp)


def _errs(stress, fmt_t, fmt_state, two_round=False):
    inp, (o_ref, s_ref) = stress
    o, s = chunked_rounded(inp, fmt_t, fmt_state, two_round)
    eo = float(np.max(np.abs(o - o_ref)) / np.max(np.abs(o_ref)))
    es = float(np.linalg.norm(s - s_ref) / np.linalg.norm(s_ref))
    return eo, es


def test_fp16_operands_stay_well_inside_the_tolerances_and_below_bf16_hilo(stress):
    eo_hl, es_hl = _errs(stress, "bf16", "hilo")
    for two_round in (True, False):  # the default kernel, and fp16 in the three-round form
        eo16, es16 = _errs(stress, "fp16", "fp16", two_round)
        assert eo16 <= OUT_TOL / 10 and es16 <= STATE_TOL / 2, (two_round, eo16, es16)
        assert es16 < es_hl and eo16 < eo_hl, (two_round, eo16, es16, eo_hl, es_hl)
    assert es_hl <= STATE_TOL and eo_hl <= OUT_TOL  # the wide-range design meets them too


def test_bf16_single_state_operands_would_miss_the_state_tolerance(stress):
    for two_round in (True, False):
        _, es = _errs(stress, "fp16", "bf16", two_round)
        assert es > STATE_TOL, (two_round, es)


def test_model_without_rounding_is_the_oracle(stress):
    """With every rounding switched off the model is the exact chunked form, so the errors above
    come from the roundings alone."""
    for two_round in (True, False):
        eo, es = _errs(stress, "f64", "f64", two_round)
        assert eo <= 1e-10 and es <= 1e-10, (two_round, eo, es)
