"""Failure detection without a GPU fault (GPU).

Every wait in the kernels is bounded; one that runs out records a status bit and
the kernel returns.  Here a wait is made to run out on purpose (an mbarrier that
nothing completes), the host reads the bit, and the context is still usable --
also for the status word of the allocation-free entry point.  A malformed
cu_seqlens is reported the same way, and a workspace allocation that fails (made
to fail on the host) returns GDN_ERR_ALLOC before anything is launched.  Values
beyond the fp16 operands' range make the default state carry's state non-finite,
which its status bit reports; the wide-range state carry takes them.  So does a
state too small for fp16's precision (values of order 1e-6), reported by its own bit.
"""

import numpy as np
import pytest

from gpu_common import OUT_TOL, STATE_TOL, out_err, run_gpu, state_err
from hybrid_linear_attention_prefill_gb300.inputs import f32_to_bf16_bits, make_gdn_inputs

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


def test_clean_runs_leave_no_status_bits(gdn):
    gdn.gdn_device_status()  # clear whatever earlier calls left
    run_gpu(make_gdn_inputs(B=2, T=300, Hk=2, Hv=4, dk=128, dv=128, seed=80))
    run_gpu(make_gdn_inputs(lengths=[0, 120, 7], Hk=2, Hv=4, dk=128, dv=128, seed=80))
    rc, bits = gdn.gdn_device_status()
    assert rc == gdn.GDN_OK and bits == 0


def test_a_wait_that_runs_out_is_reported_and_the_context_survives(gdn):
    import oracle

    rc, bits = gdn.gdn_selftest_wait_timeout(1000)
    assert rc == gdn.GDN_OK and bits == gdn.GDN_STATUS_MMA_TIMEOUT
    inp = make_gdn_inputs(B=1, T=200, Hk=1, Hv=2, dk=128, dv=128, seed=81, init_std=0.1)
    o, s = run_gpu(inp)
    o_ref, s_ref = oracle.prefill_inputs(inp)
    assert out_err(o, o_ref) <= OUT_TOL and state_err(s, s_ref) <= STATE_TOL
    rc, bits = gdn.gdn_device_status()
    assert rc == gdn.GDN_OK and bits == 0


def test_a_timed_out_wait_of_the_static_entry_is_reported(gdn):
    rc, bits = gdn.gdn_device_status()
    assert rc == gdn.GDN_OK
    assert gdn.gdn_selftest_static_wait_timeout(1000) == gdn.GDN_OK
    rc, bits = gdn.gdn_device_status()
    assert rc == gdn.GDN_OK and bits == gdn.GDN_STATUS_MMA_TIMEOUT
    rc, bits = gdn.gdn_device_status()  # read and cleared
    assert rc == gdn.GDN_OK and bits == 0


def _sentinel_run(gdn, inp, fn):
    from gpu_common import dev_inputs

    d = dev_inputs(inp)
    out = torch.full((inp.total_tokens, inp.Hv, inp.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    fin = torch.full((inp.B, inp.Hv, inp.dv, inp.dk), float("nan"), device="cuda")
    rc = fn(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"], out, fin,
            inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv)
    torch.cuda.synchronize()
    return rc, out.float().cpu().numpy(), fin.cpu().numpy()


def test_failed_workspace_allocation_launches_nothing_and_the_next_call_works(gdn):
    import oracle

    inp = make_gdn_inputs(lengths=[150, 0, 90], Hk=2, Hv=4, dk=128, dv=128, seed=82, init_std=0.1)
    gdn.gdn_release_workspace()  # the next call has to allocate
    assert gdn.gdn_debug_fail_allocations(1) == 0
    rc, o, s = _sentinel_run(gdn, inp, gdn.gdn_prefill)
    assert rc == gdn.GDN_ERR_ALLOC
    assert gdn.gdn_last_cuda_error() == 2  # cudaErrorMemoryAllocation
    assert np.all(np.isnan(o)) and np.all(np.isnan(s))  # nothing was launched
    rc, o, s = _sentinel_run(gdn, inp, gdn.gdn_prefill)
    assert rc == gdn.GDN_OK and gdn.gdn_last_cuda_error() == 0
    o_ref, s_ref = oracle.prefill_inputs(inp)
    assert out_err(o, o_ref) <= OUT_TOL and state_err(s, s_ref) <= STATE_TOL
    assert gdn.gdn_debug_fail_allocations(0) == 0  # the failure was used up


def test_malformed_cu_seqlens_sets_its_status_bit(gdn):
    gdn.gdn_device_status()
    good = make_gdn_inputs(lengths=[40, 60], Hk=1, Hv=1, dk=64, dv=64, seed=83)
    run_gpu(good)
    rc, bits = gdn.gdn_device_status()
    assert rc == gdn.GDN_OK and bits == 0
    # not non-decreasing; past T; cu[0] != 0; cu[B] != T -- each over the same 100 tokens
    for bad in ([0, 60, 40, 100], [0, 5000, 100], [3, 40, 100], [0, 40, 90]):
        inp = make_gdn_inputs(lengths=[40, 60], Hk=1, Hv=1, dk=64, dv=64, seed=83)
        inp.cu_seqlens = np.array(bad, dtype=np.int32)
        inp.B = len(bad) - 1
        o, s = run_gpu(inp)
        assert np.all(np.isfinite(s))
        rc, bits = gdn.gdn_device_status()
        assert rc == gdn.GDN_OK and bits == gdn.GDN_STATUS_BAD_CU_SEQLENS, bad


def test_values_beyond_fp16_range_are_reported_and_the_wide_range_carry_takes_them(gdn):
    import oracle

    from gpu_common import dev_inputs

    inp = make_gdn_inputs(lengths=[130, 70], Hk=1, Hv=2, dk=128, dv=128, seed=84, init_std=0.1)
    inp.v = f32_to_bf16_bits((inp.v64() * 1.0e5).astype(np.float32))  # values of order 1e5
    gdn.gdn_device_status()
    run_gpu(inp)
    rc, bits = gdn.gdn_device_status()
    assert rc == gdn.GDN_OK and bits == gdn.GDN_STATUS_NONFINITE_STATE
    d = dev_inputs(inp)
    out = torch.full((inp.total_tokens, inp.Hv, inp.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    fin = torch.full((inp.B, inp.Hv, inp.dv, inp.dk), float("nan"), device="cuda")
    gdn.check(gdn.gdn_prefill_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"], out, fin,
                                 inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, gdn.GDN_FLAG_WIDE_RANGE))
    torch.cuda.synchronize()
    rc, bits = gdn.gdn_device_status()
    assert rc == gdn.GDN_OK and bits == 0
    o_ref, s_ref = oracle.prefill_inputs(inp)
    o, s = out.float().cpu().numpy(), fin.cpu().numpy()
    assert out_err(o, o_ref) <= OUT_TOL and state_err(s, s_ref) <= STATE_TOL


def test_values_below_fp16_precision_are_reported_and_the_wide_range_carry_takes_them(gdn):
    import oracle

    from gpu_common import dev_inputs

    inp = make_gdn_inputs(lengths=[130, 70], Hk=1, Hv=2, dk=128, dv=128, seed=85)
    inp.v = f32_to_bf16_bits((inp.v64() * 1.0e-6).astype(np.float32))  # values of order 1e-6
    gdn.gdn_device_status()
    run_gpu(inp)
    rc, bits = gdn.gdn_device_status()
    assert rc == gdn.GDN_OK and bits == gdn.GDN_STATUS_SMALL_STATE
    d = dev_inputs(inp)
    out = torch.full((inp.total_tokens, inp.Hv, inp.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    fin = torch.full((inp.B, inp.Hv, inp.dv, inp.dk), float("nan"), device="cuda")
    gdn.check(gdn.gdn_prefill_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"], out, fin,
                                 inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, gdn.GDN_FLAG_WIDE_RANGE))
    torch.cuda.synchronize()
    rc, bits = gdn.gdn_device_status()
    assert rc == gdn.GDN_OK and bits == 0
    o_ref, s_ref = oracle.prefill_inputs(inp)
    o, s = out.float().cpu().numpy(), fin.cpu().numpy()
    assert out_err(o, o_ref) <= OUT_TOL and state_err(s, s_ref) <= STATE_TOL
