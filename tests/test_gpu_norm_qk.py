"""gdn_prefill_ex with in-kernel q/k L2 normalisation, against the oracle (GPU).

The oracle is given q / max(||q||, 1e-6) and k / max(||k||, 1e-6) computed in
float64 from the same raw bf16 values the GPU receives.
"""

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


def _normalised(x):
    return x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), 1e-6)


def _run_ex(gdn, inp, flags):
    d = dev_inputs(inp)
    out = torch.empty((inp.total_tokens, inp.Hv, inp.dv), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((inp.B, inp.Hv, inp.dv, inp.dk), device="cuda")
    gdn.check(gdn.gdn_prefill_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"], out, fin,
                                 inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, flags))
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), fin.cpu().numpy()


@pytest.mark.parametrize("case", [
    dict(B=1, T=1024, Hk=4, Hv=8, dk=128, dv=128),
    dict(lengths=[70, 0, 200, 5], Hk=2, Hv=4, dk=128, dv=128, init_std=0.1),
    dict(B=2, T=130, Hk=1, Hv=2, dk=64, dv=64),
    dict(B=1, T=100, Hk=1, Hv=1, dk=32, dv=32),
    # more (chunk, key head) items than preparation CTAs: each CTA works on several, writing
    # every item's inverse norms
    dict(B=1, T=4096, Hk=16, Hv=32, dk=128, dv=128),
    dict(lengths=[1500, 0, 900, 77, 640], Hk=8, Hv=16, dk=64, dv=64, init_std=0.1),
])
def test_in_kernel_normalisation_matches_oracle(gdn, case):
    import oracle

    inp = make_gdn_inputs(seed=70, normalize_qk=False, **case)
    o, s = _run_ex(gdn, inp, gdn.GDN_FLAG_L2NORM_QK)
    o_ref, s_ref = oracle.prefill(_normalised(inp.q64()), _normalised(inp.k64()), inp.v64(), inp.g64(),
                                  inp.beta64(), inp.cu_seqlens, inp.init64(), B=inp.B,
                                  T=None if inp.cu_seqlens is not None else inp.T)
    assert np.all(np.isfinite(o))
    assert out_err(o, o_ref) <= OUT_TOL
    assert state_err(s, s_ref) <= STATE_TOL


def test_no_flags_is_gdn_prefill(gdn):
    inp = make_gdn_inputs(B=1, T=300, Hk=2, Hv=4, dk=128, dv=128, seed=71, init_std=0.1)
    o1, s1 = run_gpu(inp)
    o2, s2 = _run_ex(gdn, inp, 0)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)
