"""The float64 oracle against its pins (CPU only)."""

import ctypes
import json
import os
import subprocess

import numpy as np
import pytest

import oracle_pins as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(oracle_mod, pin):
    pin(oracle_mod.prefill)


def test_hand_worked(oracle_mod):
    with open(os.path.join(GOLDEN, "hand_worked_dk2.json")) as f:
        P.pin_hand_worked(oracle_mod.prefill, json.load(f))


def test_thread_count_does_not_change_bits(oracle_mod):
    rng = np.random.default_rng(20)
    p = P.rand_problem(rng, Hk=2, Hv=4, dk=16, dv=8, lengths=(33, 7, 50))
    o1, s1 = P.call(oracle_mod.prefill, p, nthreads=1)
    o8, s8 = P.call(oracle_mod.prefill, p, nthreads=8)
    assert np.array_equal(o1, o8) and np.array_equal(s1, s8)


def test_tiny_regression_fixture(oracle_mod):
    """The oracle still writes what the committed script recorded for the tiny workload."""
    from hybrid_linear_attention_prefill_gb300.inputs import workload

    d = np.load(os.path.join(GOLDEN, "tiny_t64_d32.npz"))
    o, s = oracle_mod.prefill_inputs(workload("tiny_t64_d32"))
    np.testing.assert_allclose(o, d["out"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(s, d["final_state"], rtol=0, atol=1e-13)


# ---- planted mistakes --------------------------------------------------------
# Each entry patches one line of a private copy of the oracle's source; the
# patched oracle must fail at least one pin.  This shows that the pins would
# catch a dropped term, a wrong sign, a wrong index or a transposed operand.

MUTATIONS = {
    "no_decay": ("Si[j] *= alpha;          /* decay */", "Si[j] *= 1.0;"),
    "decay_after_read": ("sk += Si[j] * kt[j];     /* (alpha S) k */",
                         "sk += Si[j] / alpha * kt[j];"),
    "sign_of_delta": ("const double u = beta * (vt[i] - sk);", "const double u = beta * (vt[i] + sk);"),
    "beta_on_v_only": ("const double u = beta * (vt[i] - sk);", "const double u = beta * vt[i] - sk;"),
    "write_with_q": ("Si[j] += u * kt[j];      /* rank-one write */", "Si[j] += u * qt[j];"),
    "read_before_write": ("sq += Si[j] * qt[j];     /* S_t q_t */", "sq += (Si[j] - u * kt[j]) * qt[j];"),
    "no_scale": ("ot[i] = sq * scale;", "ot[i] = sq;"),
    "gqa_modulo": ("const int hk = h / (Hv / Hk);", "const int hk = h % Hk;"),
    "transposed_state_read": ("sk += Si[j] * kt[j];     /* (alpha S) k */",
                              "sk += S[(long)(j % dv) * dk + (i % dk)] * kt[j];"),
    "init_ignored": ("memcpy(S, J->init + ((long)n * Hv + h) * dv * dk, sizeof(double) * dv * dk);",
                     "memset(S, 0, sizeof(double) * dv * dk);"),
    "key_from_value_head": ("const double *kt = J->k + (t * Hk + hk) * dk;",
                            "const double *kt = J->k + (t * Hk + (h % Hk)) * dk;"),
}


def _build_mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "gdn_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation {name}: target line not found once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-pthread", str(path), "-o", str(so), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    lib.gdn_oracle_prefill.argtypes = [dp, dp, dp, dp, dp, ip, dp, dp, dp] + [ctypes.c_int] * 7
    lib.gdn_oracle_prefill.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(oracle_mod, tmp_path, name):
    lib = _build_mutant(tmp_path, name)
    saved = oracle_mod._lib
    oracle_mod._lib = lib
    try:
        failed = []
        for pin in P.ALL_PINS:
            try:
                pin(oracle_mod.prefill)
            except (AssertionError, FloatingPointError, np.linalg.LinAlgError) as e:
                failed.append((pin.__name__, str(e)[:80]))
        assert failed, f"mutation {name} passed every pin"
    finally:
        oracle_mod._lib = saved
