"""Failure detection without a GPU fault (GPU).

Every wait in the kernels is bounded; one that runs out records a status bit and
the kernel returns.  Here a wait is made to run out on purpose (an mbarrier that
nothing completes), the host reads the bit, and the context is still usable.
"""

import numpy as np
import pytest

from gpu_common import OUT_TOL, STATE_TOL, out_err, run_gpu, state_err
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


def test_clean_runs_leave_no_status_bits(gdn):
    run_gpu(make_gdn_inputs(B=2, T=300, Hk=2, Hv=4, dk=128, dv=128, seed=80))
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
