"""The two-level chunk scan (segments run from zero / identity starts, an fp32
combine of the segment start states, then every segment again) against the
oracle, and against the single-level path, through gdn_prefill_ex (GPU)."""

import numpy as np
import pytest

from gpu_common import OUT_TOL, STATE_TOL, dev_inputs, out_err, state_err
from hybrid_linear_attention_prefill_gb300.inputs import make_gdn_inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hybrid_linear_attention_prefill_gb300 import build
    from hybrid_linear_attention_prefill_gb300 import gdn as g

    build.build()
    g.load()
    return g


def _run(gdn, inp, flags, want_final=True, plain=False):
    d = dev_inputs(inp)
    out = torch.full((inp.total_tokens, inp.Hv, inp.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    fin = torch.full((inp.B, inp.Hv, inp.dv, inp.dk), float("nan"), device="cuda") if want_final else None
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"], out, fin,
            inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv)
    st = gdn.gdn_prefill(*args) if plain else gdn.gdn_prefill_ex(*args, flags)
    gdn.check(st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), None if fin is None else fin.cpu().numpy()


def _check_oracle(o, s, inp):
    import oracle

    o_ref, s_ref = oracle.prefill_inputs(inp, want_final=s is not None)
    eo = out_err(o, o_ref)
    assert eo <= OUT_TOL, eo
    if s is not None:
        es = state_err(s, s_ref)
        assert es <= STATE_TOL, es
    return o_ref, s_ref


def _two(gdn, P=0):
    return gdn.GDN_FLAG_TWO_LEVEL | (gdn.GDN_FLAG_SEGMENTS(P) if P else 0)


@pytest.mark.parametrize("P", [2, 3, 4, 7, 255])
def test_segments_against_oracle_slow_decay_with_carry(gdn, P):
    # 1000 tokens = 15 full chunks + 40: segments of 8/8, 5/5/5+, 4/4/4/3+, 3x5 + 1 + empty, 16 x 1
    inp = make_gdn_inputs(B=1, T=1000, Hk=1, Hv=2, dk=128, dv=128, seed=90 + P, g_scale=0.05, init_std=0.1)
    o, s = _run(gdn, inp, _two(gdn, P))
    _check_oracle(o, s, inp)


def test_batch_ragged_with_heads_groups(gdn):
    inp = make_gdn_inputs(B=2, T=700, Hk=2, Hv=4, dk=128, dv=128, seed=95, g_scale=0.1, init_std=0.1)
    o, s = _run(gdn, inp, _two(gdn, 4))
    _check_oracle(o, s, inp)


@pytest.mark.parametrize("dk,dv", [(32, 128), (128, 32), (64, 64), (64, 128)])
def test_head_dims(gdn, dk, dv):
    inp = make_gdn_inputs(B=1, T=450, Hk=1, Hv=2, dk=dk, dv=dv, seed=96 + dk + dv, g_scale=0.05, init_std=0.1)
    o, s = _run(gdn, inp, _two(gdn, 3))
    _check_oracle(o, s, inp)


def test_no_decay_strong_writes(gdn):
    """g = 0, beta near 1: nothing decays, so every segment's transition carries fully."""
    inp = make_gdn_inputs(B=1, T=300, Hk=1, Hv=2, dk=128, dv=128, seed=97, init_std=0.1)
    inp.g[:] = 0.0
    inp.beta[:] = 0.999
    o, s = _run(gdn, inp, _two(gdn, 4))  # 5 chunks: segments of 2, 2, 1 and an empty one
    _check_oracle(o, s, inp)


@pytest.mark.parametrize("P", [3, 4])
def test_wide_range_state_carry(gdn, P):
    """The two-level scan on the bf16 hi / lo state carry (its transition runs included)."""
    inp = make_gdn_inputs(B=2, T=700, Hk=2, Hv=4, dk=128, dv=128, seed=98 + P, g_scale=0.05, init_std=0.1)
    o, s = _run(gdn, inp, _two(gdn, P) | gdn.GDN_FLAG_WIDE_RANGE)
    _check_oracle(o, s, inp)


def test_zero_init_and_no_final_state(gdn):
    inp = make_gdn_inputs(B=1, T=640, Hk=1, Hv=1, dk=128, dv=128, seed=98, g_scale=0.05)
    o, _ = _run(gdn, inp, _two(gdn, 5), want_final=False)
    _check_oracle(o, None, inp)


def test_final_state_may_alias_init(gdn):
    inp = make_gdn_inputs(B=1, T=500, Hk=1, Hv=2, dk=128, dv=128, seed=99, g_scale=0.05, init_std=0.1)
    d = dev_inputs(inp)
    state = d["init"].clone()
    out = torch.empty((inp.total_tokens, inp.Hv, inp.dv), dtype=torch.bfloat16, device="cuda")
    gdn.check(gdn.gdn_prefill_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], None, state, out, state,
                                 inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, _two(gdn, 4)))
    torch.cuda.synchronize()
    _check_oracle(out.float().cpu().numpy(), state.cpu().numpy(), inp)


def test_agrees_with_single_level(gdn):
    inp = make_gdn_inputs(B=1, T=2000, Hk=2, Hv=2, dk=128, dv=128, seed=100, g_scale=0.02, init_std=0.05)
    o2, s2 = _run(gdn, inp, _two(gdn, 6))
    o1, s1 = _run(gdn, inp, gdn.GDN_FLAG_ONE_LEVEL)
    assert out_err(o2, o1) <= OUT_TOL and state_err(s2, s1) <= STATE_TOL
    _check_oracle(o2, s2, inp)


def test_packed_batches_stay_single_level(gdn):
    """The flag does not apply to packed batches: bitwise the single-level result."""
    inp = make_gdn_inputs(lengths=[300, 500], Hk=1, Hv=2, dk=128, dv=128, seed=101, init_std=0.1)
    o2, s2 = _run(gdn, inp, _two(gdn, 4))
    o1, s1 = _run(gdn, inp, gdn.GDN_FLAG_ONE_LEVEL)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_chosen_automatically_for_a_long_prompt_with_few_heads(gdn):
    """16,384 tokens with 4 value heads: gdn_prefill takes the two-level path on its own
    (bitwise the forced result with the library's segment count) and matches the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # the largest P whose pass A -- 4 heads x ((P - 1) x 4 + (P - 2) x 4) CTAs -- fits one wave
    P = min((sms * 32 // 4 + 128 + 2 * 128) // (128 + 128), 16384 // 64 // 8, 32)
    assert gdn.gdn_scan_segments(1, 16384, 4, 4, 128, 128, 0) == (P if P >= 3 else 1)
    if P < 3:
        pytest.skip("device too small for the automatic choice")
    inp = make_gdn_inputs(B=1, T=16384, Hk=4, Hv=4, dk=128, dv=128, seed=102, g_scale=0.1, init_std=0.02)
    o_auto, s_auto = _run(gdn, inp, 0, plain=True)
    o_two, s_two = _run(gdn, inp, _two(gdn, P))
    assert np.array_equal(o_auto, o_two) and np.array_equal(s_auto, s_two)
    _check_oracle(o_auto, s_auto, inp)


def test_buffer_reuse_across_head_dims(gdn):
    """Calls in the order large-then-small-then-larger head dims reuse the library's scan
    buffer; each must still see an all-zero value tensor for its transition run."""
    for dk, dv, T, Hv in [(128, 128, 700, 4), (32, 128, 450, 2), (128, 32, 450, 2), (64, 64, 300, 2)]:
        inp = make_gdn_inputs(B=1, T=T, Hk=1, Hv=Hv, dk=dk, dv=dv, seed=103 + dk + dv, g_scale=0.05,
                              init_std=0.1)
        o, s = _run(gdn, inp, _two(gdn, 3))
        _check_oracle(o, s, inp)
