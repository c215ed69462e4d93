"""Checks that pin the float64 oracle to facts other than itself (tests only).

Each ``pin_*`` takes a ``prefill`` callable with the signature of
``oracle.prefill`` and raises AssertionError when the callable disagrees with:
an independent formulation (brute-force matrices, the chunked WY form), a
closed form, or an invariant of the gated delta rule
S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
o_t = S_t q_t / sqrt(dk).  The same pins are run against deliberately broken
copies of the oracle to show that each plausible mistake is caught.
"""

from __future__ import annotations

import numpy as np

from refs import brute_force, chunked

TOL = 1e-11


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_problem(rng, *, Hk=1, Hv=1, dk=8, dv=6, lengths=(13,), init=True, g_scale=1.0,
                 packed=None):
    lengths = list(lengths)
    Ttot = sum(lengths)
    q = _unit_rows(rng.standard_normal((Ttot, Hk, dk)))
    k = _unit_rows(rng.standard_normal((Ttot, Hk, dk)))
    v = rng.standard_normal((Ttot, Hv, dv))
    g = -np.logaddexp(0, rng.standard_normal((Ttot, Hv))) * g_scale
    beta = 1 / (1 + np.exp(-rng.standard_normal((Ttot, Hv))))
    B = len(lengths)
    S0 = rng.standard_normal((B, Hv, dv, dk)) * 0.5 if init else None
    if packed is None:
        packed = len(set(lengths)) > 1 or 0 in lengths
    cu = None
    if packed:
        cu = np.zeros(B + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lengths)
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu=cu, init=S0, B=B)


def call(prefill, p, **kw):
    return prefill(p["q"], p["k"], p["v"], p["g"], p["beta"], p["cu"], p["init"],
                   B=p["B"], T=None if p["cu"] is not None else p["q"].shape[0] // p["B"], **kw)


def close(a, b, tol=TOL, what=""):
    err = np.max(np.abs(a - b)) if a.size else 0.0
    ref = max(1.0, np.max(np.abs(b)) if b.size else 0.0)
    assert err <= tol * ref, f"{what}: max abs diff {err:.3e} (scale {ref:.3e})"


# ---- independent formulations -------------------------------------------

def pin_brute_force(prefill, seed=1):
    rng = np.random.default_rng(seed)
    for kw in (dict(), dict(Hk=2, Hv=4, dk=5, dv=3, lengths=(7, 0, 11)),
               dict(Hk=1, Hv=3, dk=4, dv=9, lengths=(9, 9), init=False)):
        p = rand_problem(rng, **kw)
        o, s = call(prefill, p)
        ob, sb = brute_force(p["q"], p["k"], p["v"], p["g"], p["beta"], p["cu"], p["init"], p["B"])
        close(o, ob, what="out vs brute force")
        close(s, sb, what="state vs brute force")


def pin_chunked(prefill, seed=2):
    rng = np.random.default_rng(seed)
    p = rand_problem(rng, Hk=2, Hv=4, dk=16, dv=12, lengths=(70, 5, 130))
    o, s = call(prefill, p)
    for C in (1, 16, 64):
        oc, sc = chunked(p["q"], p["k"], p["v"], p["g"], p["beta"], p["cu"], p["init"], p["B"], C=C)
        close(o, oc, 1e-10, what=f"out vs chunked C={C}")
        close(s, sc, 1e-10, what=f"state vs chunked C={C}")


# ---- closed forms ---------------------------------------------------------

def pin_identity_when_no_write(prefill, seed=3):
    """beta = 0, g = 0: the state never changes and o_t = S0 q_t / sqrt(dk)."""
    rng = np.random.default_rng(seed)
    p = rand_problem(rng, Hk=1, Hv=2, dk=6, dv=5, lengths=(9,))
    p["beta"][:] = 0.0
    p["g"][:] = 0.0
    o, s = call(prefill, p)
    close(s, p["init"], what="state unchanged")
    for h in range(2):
        close(o[:, h], p["q"][:, 0] @ p["init"][0, h].T / np.sqrt(6), what="o = S0 q / sqrt(dk)")


def pin_orthonormal_retrieval(prefill, seed=4):
    """alpha = 1, beta = 1, orthonormal keys: every written value is retrieved."""
    rng = np.random.default_rng(seed)
    dk, dv, T = 8, 5, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:, :T].T  # T orthonormal rows
    p = rand_problem(rng, dk=dk, dv=dv, lengths=(T,))
    p["k"][:, 0] = keys
    p["q"][:, 0] = keys  # query each key right after writing it
    p["g"][:] = 0.0
    p["beta"][:] = 1.0
    o, s = call(prefill, p)
    S = s[0, 0]
    close(S @ keys.T, p["v"][:, 0].T, what="S k_i = v_i")
    close(o[:, 0] * np.sqrt(dk), p["v"][:, 0], what="o_t = v_t / sqrt(dk)")


def pin_reset(prefill, seed=5):
    """g = -inf (alpha = 0): S_t = beta_t v_t k_t^T."""
    rng = np.random.default_rng(seed)
    p = rand_problem(rng, Hk=1, Hv=2, dk=4, dv=3, lengths=(5,))
    p["g"][:] = -np.inf
    o, s = call(prefill, p)
    for h in range(2):
        bt = p["beta"][:, h]
        kq = np.sum(p["k"][:, 0] * p["q"][:, 0], axis=-1)
        close(o[:, h], (bt * kq)[:, None] * p["v"][:, h] / 2.0, what="o after reset")
        close(s[0, h], bt[-1] * np.outer(p["v"][-1, h], p["k"][-1, 0]), what="S after reset")


def pin_single_token(prefill, seed=6):
    """One token: S1 = alpha S0 + beta (v - alpha S0 k) k^T."""
    rng = np.random.default_rng(seed)
    p = rand_problem(rng, Hk=1, Hv=1, dk=7, dv=4, lengths=(1,))
    a = np.exp(p["g"][0, 0])
    b = p["beta"][0, 0]
    S0 = p["init"][0, 0]
    kk, qq, vv = p["k"][0, 0], p["q"][0, 0], p["v"][0, 0]
    S1 = a * S0 + b * np.outer(vv - a * S0 @ kk, kk)
    o, s = call(prefill, p)
    close(s[0, 0], S1, what="state after one token")
    close(o[0, 0], S1 @ qq / np.sqrt(7), what="output after one token")


def pin_hand_worked(prefill, fixture):
    """Values derived by hand with exact fractions (tests/golden)."""
    f = fixture
    q = np.array(f["q"], dtype=np.float64)[:, None, :]
    k = np.array(f["k"], dtype=np.float64)[:, None, :]
    v = np.array(f["v"], dtype=np.float64)[:, None, :]
    g = np.array(f["g"], dtype=np.float64)[:, None]
    beta = np.array(f["beta"], dtype=np.float64)[:, None]
    o, s = prefill(q, k, v, g, beta, None, None, B=1, T=q.shape[0])
    close(o[:, 0], np.array(f["out"]), 1e-12, what="hand-worked outputs")
    close(s[0, 0], np.array(f["final_state"]), 1e-12, what="hand-worked state")


# ---- invariants -----------------------------------------------------------

def pin_split_carry(prefill, seed=7):
    """Running [0, t1) then [t1, T) with the carried state equals one run."""
    rng = np.random.default_rng(seed)
    p = rand_problem(rng, Hk=1, Hv=2, dk=6, dv=4, lengths=(40,), g_scale=0.1)
    o, s = call(prefill, p)
    for t1 in (1, 17, 39):
        a = {kk: (vv[:t1] if isinstance(vv, np.ndarray) and kk not in ("init", "cu") else vv)
             for kk, vv in p.items()}
        o1, s1 = call(prefill, a)
        b = {kk: (vv[t1:] if isinstance(vv, np.ndarray) and kk not in ("init", "cu") else vv)
             for kk, vv in p.items()}
        b["init"] = s1
        o2, s2 = call(prefill, b)
        close(np.concatenate([o1, o2]), o, what=f"split at {t1}: outputs")
        close(s2, s, what=f"split at {t1}: state")


def pin_row_permutation(prefill, seed=8):
    """Permuting the dv coordinate of v and S0 permutes o and S rows alike."""
    rng = np.random.default_rng(seed)
    p = rand_problem(rng, Hk=1, Hv=1, dk=5, dv=7, lengths=(11,))
    o, s = call(prefill, p)
    perm = rng.permutation(7)
    p2 = dict(p)
    p2["v"] = p["v"][:, :, perm]
    p2["init"] = p["init"][:, :, perm, :]
    o2, s2 = call(prefill, p2)
    close(o2, o[:, :, perm], what="permuted outputs")
    close(s2, s[:, :, perm, :], what="permuted state")


def pin_gqa_repeat(prefill, seed=9):
    """Hv = 2 Hk equals a run on explicitly repeat-interleaved q and k."""
    rng = np.random.default_rng(seed)
    p = rand_problem(rng, Hk=2, Hv=4, dk=4, dv=3, lengths=(10,))
    o, s = call(prefill, p)
    p2 = dict(p)
    p2["q"] = np.repeat(p["q"], 2, axis=1)
    p2["k"] = np.repeat(p["k"], 2, axis=1)
    o2, s2 = call(prefill, p2)
    close(o, o2, 0.0, what="GQA outputs")
    close(s, s2, 0.0, what="GQA state")


def pin_varlen_equals_separate(prefill, seed=10):
    rng = np.random.default_rng(seed)
    lens = (5, 0, 12, 1)
    p = rand_problem(rng, Hk=1, Hv=2, dk=4, dv=3, lengths=lens)
    o, s = call(prefill, p)
    cu = p["cu"]
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        sub = dict(q=p["q"][a:b], k=p["k"][a:b], v=p["v"][a:b], g=p["g"][a:b],
                   beta=p["beta"][a:b], cu=None, init=p["init"][n:n + 1], B=1)
        if b == a:
            close(s[n], p["init"][n], 0.0, what="empty sequence keeps its state")
            continue
        o1, s1 = call(prefill, sub)
        close(o[a:b], o1, 0.0, what=f"seq {n} outputs")
        close(s[n], s1[0], 0.0, what=f"seq {n} state")


def pin_padding_tokens(prefill, seed=11):
    """Tokens with beta = 0 and g = 0 leave the final state unchanged."""
    rng = np.random.default_rng(seed)
    p = rand_problem(rng, Hk=1, Hv=1, dk=4, dv=4, lengths=(13,))
    o, s = call(prefill, p)
    pad = 3
    p2 = {kk: (np.concatenate([vv, np.zeros((pad,) + vv.shape[1:])])
               if isinstance(vv, np.ndarray) and kk not in ("init", "cu") else vv)
          for kk, vv in p.items()}
    p2["k"][13:, 0] = _unit_rows(rng.standard_normal((pad, 4)))
    o2, s2 = call(prefill, p2)
    close(o2[:13], o, 0.0, what="outputs before padding")
    close(s2, s, what="state after padding")


def pin_contraction_bound(prefill, seed=12):
    """||S_t||_2 <= alpha_t ||S_{t-1}||_2 + beta_t ||v_t||_2 when ||k_t|| = 1."""
    rng = np.random.default_rng(seed)
    p = rand_problem(rng, Hk=1, Hv=1, dk=5, dv=5, lengths=(12,))
    S = p["init"]
    for t in range(12):
        one = {kk: (vv[t:t + 1] if isinstance(vv, np.ndarray) and kk not in ("init", "cu") else vv)
               for kk, vv in p.items()}
        one["init"] = S
        _, S1 = call(prefill, one)
        lhs = np.linalg.norm(S1[0, 0], 2)
        rhs = np.exp(p["g"][t, 0]) * np.linalg.norm(S[0, 0], 2) + p["beta"][t, 0] * np.linalg.norm(p["v"][t, 0])
        assert lhs <= rhs * (1 + 1e-12), f"contraction bound broken at t={t}: {lhs} > {rhs}"
        S = S1


def pin_scale(prefill, seed=13):
    """The output scale is 1/sqrt(dk): with S0 = 0, one token gives beta (k.q) v / sqrt(dk)."""
    rng = np.random.default_rng(seed)
    for dk in (4, 9, 16):
        p = rand_problem(rng, dk=dk, dv=3, lengths=(1,), init=False)
        o, _ = call(prefill, p)
        want = p["beta"][0, 0] * np.dot(p["k"][0, 0], p["q"][0, 0]) * p["v"][0, 0] / np.sqrt(dk)
        close(o[0, 0], want, what=f"scale at dk={dk}")


ALL_PINS = [pin_brute_force, pin_chunked, pin_identity_when_no_write, pin_orthonormal_retrieval,
            pin_reset, pin_single_token, pin_split_carry, pin_row_permutation, pin_gqa_repeat,
            pin_varlen_equals_separate, pin_padding_tokens, pin_contraction_bound, pin_scale]
