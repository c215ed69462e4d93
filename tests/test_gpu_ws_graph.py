"""gdn_prefill_ws: caller-owned workspace, and replay of a captured CUDA graph (GPU).

The pages' workers capture the forward pass per prompt length and replay it with
fresh inputs ("Cua-S1 4B 0.2 native text worker", CUDA Graph paragraph); this is
the library-level form of that calling convention.
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


def _bufs(inp):
    out = torch.empty((inp.total_tokens, inp.Hv, inp.dv), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((inp.B, inp.Hv, inp.dv, inp.dk), device="cuda")
    return out, fin


def _workspace(gdn, inp):
    n = gdn.gdn_workspace_bytes(inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, inp.cu_seqlens is not None)
    return torch.empty(n, dtype=torch.uint8, device="cuda"), n


@pytest.mark.parametrize("packed", [False, True])
def test_caller_workspace_matches_library_workspace(gdn, packed):
    inp = (make_gdn_inputs(lengths=[100, 0, 300], Hk=2, Hv=4, dk=128, dv=128, seed=41, init_std=0.1) if packed
           else make_gdn_inputs(B=2, T=200, Hk=2, Hv=4, dk=128, dv=128, seed=41, init_std=0.1))
    d = dev_inputs(inp)
    o1, f1 = _bufs(inp)
    o2, f2 = _bufs(inp)
    ws, n = _workspace(gdn, inp)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"])
    dims = (inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv)
    gdn.check(gdn.gdn_prefill(*args, o1, f1, *dims))
    gdn.check(gdn.gdn_prefill_ws(*args, o2, f2, *dims, ws, n))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_captured_graph_replays_with_new_inputs(gdn):
    shape = dict(B=1, T=1000, Hk=4, Hv=8, dk=128, dv=128)
    a = make_gdn_inputs(seed=42, init_std=0.05, **shape)
    b = make_gdn_inputs(seed=43, init_std=0.05, **shape)
    da, db = dev_inputs(a), dev_inputs(b)
    out, fin = _bufs(a)
    ws, n = _workspace(gdn, a)
    dims = (a.B, a.T, a.Hk, a.Hv, a.dk, a.dv)
    args = lambda d: (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"])  # noqa: E731
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside the capture
        gdn.check(gdn.gdn_prefill_ws(*args(da), out, fin, *dims, ws, n, s))
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.check(gdn.gdn_prefill_ws(*args(da), out, fin, *dims, ws, n))
    # new values in the captured buffers, then replay
    for key in ("q", "k", "v", "g", "beta", "init"):
        da[key].copy_(db[key])
    graph.replay()
    torch.cuda.synchronize()
    ref_o, ref_f = _bufs(b)
    gdn.check(gdn.gdn_prefill(*args(db), ref_o, ref_f, *dims))
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(fin, ref_f)
    # and the replayed graph's results stand against the float64 oracle on the new inputs
    import oracle

    o_ref, s_ref = oracle.prefill_inputs(b)
    o, f = out.float().cpu().numpy(), fin.cpu().numpy()
    assert out_err(o, o_ref) <= OUT_TOL and state_err(f, s_ref) <= STATE_TOL
    graph.replay()  # a second replay gives the same result
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(fin, ref_f)
