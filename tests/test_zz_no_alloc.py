"""gdn_prefill_static: the allocation-free entry point (GPU).

Some callers cannot allocate device memory -- a plugin whose host engine owns all
of it, a service with a memory budget fixed at start-up, code that must not take
cudaMalloc's implicit synchronisation.  gdn_prefill_static serves them from a fixed
device array instead of the grow-only workspace.  This file checks, through the C
ABI, that two calls in a row give bit for bit what gdn_prefill gives (the same
kernels on the same inputs), that the result stands against the float64 oracle,
and that a problem larger than the fixed scratch is refused before any launch.
It is named so that pytest collects it last.
"""

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


def _run(gdn, fn, inp):
    d = dev_inputs(inp)
    out = torch.full((inp.total_tokens, inp.Hv, inp.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    fin = torch.full((inp.B, inp.Hv, inp.dv, inp.dk), float("nan"), device="cuda")
    gdn.check(fn(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"], out, fin,
                 inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv))
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), fin.cpu().numpy()


def test_two_calls_match_gdn_prefill(gdn):
    import oracle

    # first a packed batch, then a longer dense problem: the second call reuses the
    # array the first one left behind
    cases = [make_gdn_inputs(lengths=[130, 0, 64, 7], Hk=2, Hv=4, dk=128, dv=128, seed=31, init_std=0.1),
             make_gdn_inputs(B=1, T=4096, Hk=16, Hv=32, dk=128, dv=128, seed=32)]
    for i, inp in enumerate(cases):
        o_ref, s_ref = _run(gdn, gdn.gdn_prefill, inp)
        o, s = _run(gdn, gdn.gdn_prefill_static, inp)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(s))
        assert np.array_equal(o, o_ref) and np.array_equal(s, s_ref)
        if i == 0:
            o64, s64 = oracle.prefill_inputs(inp)
            assert out_err(o, o64) <= OUT_TOL
            assert state_err(s, s64) <= STATE_TOL


def test_too_large_is_refused(gdn):
    # 4,096 chunks of one head need 48.5 KiB each (Tm / PT tiles, the fp16 k / q image and
    # the norms), 194 MiB in all, more than the 128 MiB array.  The buffers are the size the
    # call claims, so even a refusal that went wrong could not read or write past them.
    T_big = 4096 * 64
    need = gdn.gdn_workspace_bytes(1, T_big, 1, 1, 128, 128, 0)
    assert need > gdn.GDN_STATIC_SCRATCH_BYTES
    q = torch.zeros((T_big, 1, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros_like(q)
    v = torch.zeros_like(q)
    g = torch.zeros((T_big, 1), device="cuda")
    beta = torch.zeros_like(g)
    out = torch.full((T_big, 1, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = gdn.gdn_prefill_static(q, k, v, g, beta, None, None, out, None, 1, T_big, 1, 1, 128, 128)
    torch.cuda.synchronize()
    assert st == gdn.GDN_ERR_SCRATCH
    assert "scratch" in gdn.gdn_strerror(st)
    assert bool(torch.isnan(out.float()).all())  # nothing was launched
