"""gdn_decode: one token per sequence on a carried state, against the float64 oracle (GPU)."""

import numpy as np
import pytest

from gpu_common import OUT_TOL, STATE_TOL, dev_inputs, out_err, run_gpu, state_err
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


def _decode_steps(gdn, inp, n_steps):
    """Run tokens 0..n_steps-1 of a single-sequence problem through gdn_decode, one by one."""
    d = dev_inputs(inp)
    Hv, dv, dk = inp.Hv, inp.dv, inp.dk
    state = (d["init"].clone() if d["init"] is not None
             else torch.zeros((1, Hv, dv, dk), device="cuda"))
    outs = []
    for t in range(n_steps):
        o = torch.empty((1, Hv, dv), dtype=torch.bfloat16, device="cuda")
        gdn.check(gdn.gdn_decode(d["q"][t:t + 1].contiguous(), d["k"][t:t + 1].contiguous(),
                                 d["v"][t:t + 1].contiguous(), d["g"][t:t + 1].contiguous(),
                                 d["beta"][t:t + 1].contiguous(), state, o, 1, inp.Hk, Hv, dk, dv))
        outs.append(o)
    torch.cuda.synchronize()
    return torch.cat(outs).float().cpu().numpy(), state.cpu().numpy()


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (32, 128), (128, 32)])
def test_decode_batch_matches_oracle(gdn, dk, dv):
    import oracle

    B, Hk, Hv = 5, 2, 4
    inp = make_gdn_inputs(B=B, T=1, Hk=Hk, Hv=Hv, dk=dk, dv=dv, seed=50 + dk + dv, init_std=0.5)
    d = dev_inputs(inp)
    state = d["init"].clone()
    out = torch.empty((B, Hv, dv), dtype=torch.bfloat16, device="cuda")
    gdn.check(gdn.gdn_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], state, out, B, Hk, Hv, dk, dv))
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.prefill_inputs(inp)
    assert out_err(out.float().cpu().numpy(), o_ref) <= OUT_TOL
    assert state_err(state.cpu().numpy(), s_ref) <= 1e-5  # fp32 arithmetic throughout


def test_decode_steps_match_prefill_oracle(gdn):
    """Thirty decode steps in a row equal the recurrence over those thirty tokens."""
    import oracle

    inp = make_gdn_inputs(B=1, T=30, Hk=2, Hv=4, dk=128, dv=128, seed=60, g_scale=0.1, init_std=0.1)
    o, s = _decode_steps(gdn, inp, 30)
    o_ref, s_ref = oracle.prefill_inputs(inp)
    assert out_err(o, o_ref) <= OUT_TOL
    assert state_err(s, s_ref) <= 1e-5


def test_prefill_then_decode_continues_the_sequence(gdn):
    """prefill(T) then decode(token T+1) agrees with prefill(T+1) on the last output and state."""
    full = make_gdn_inputs(B=1, T=201, Hk=2, Hv=4, dk=128, dv=128, seed=61, init_std=0.1)
    o_full, s_full = run_gpu(full)
    head = make_gdn_inputs(B=1, T=201, Hk=2, Hv=4, dk=128, dv=128, seed=61, init_std=0.1)
    for f in ("q", "k", "v", "g", "beta"):
        setattr(head, f, getattr(full, f)[:200].copy())
    head.T = 200
    _, s_head = run_gpu(head)
    d = dev_inputs(full)
    state = torch.from_numpy(s_head).cuda()
    out = torch.empty((1, 4, 128), dtype=torch.bfloat16, device="cuda")
    gdn.check(gdn.gdn_decode(d["q"][200:].contiguous(), d["k"][200:].contiguous(), d["v"][200:].contiguous(),
                             d["g"][200:].contiguous(), d["beta"][200:].contiguous(), state, out,
                             1, 2, 4, 128, 128))
    torch.cuda.synchronize()
    assert out_err(out.float().cpu().numpy(), o_full[200:]) <= OUT_TOL
    assert state_err(state.cpu().numpy(), s_full) <= STATE_TOL
