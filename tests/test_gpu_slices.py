"""State-carry CTAs of 16, 32 or 64 state rows (GDN_FLAG_SLICE16 / 32 / 64) against the oracle,
and against each other bit for bit (GPU), for both operand formats: the default fp16 state carry
and the wide-range bf16 hi / lo one (GDN_FLAG_WIDE_RANGE).  The library takes 64 rows on its own
for grids of many waves (the packed 32-candidate workload's parity test runs that way) and 16 for
few heads (most small parity cases); these force each width on small inputs: dense and packed
batches, every dk with dv = 32, 64 and 128, an initial state, many chunks, in-kernel q/k
normalisation."""

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


def _run(gdn, inp, flags):
    d = dev_inputs(inp)
    out = torch.full((inp.total_tokens, inp.Hv, inp.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    fin = torch.full((inp.B, inp.Hv, inp.dv, inp.dk), float("nan"), device="cuda")
    gdn.check(gdn.gdn_prefill_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"], out, fin,
                                 inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, flags))
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), fin.cpu().numpy()


def _both_widths_against_oracle(gdn, inp, extra=0, ref=None):
    import oracle

    o_ref, s_ref = ref if ref is not None else oracle.prefill_inputs(inp)
    widths = [("16", gdn.GDN_FLAG_SLICE16), ("32", gdn.GDN_FLAG_SLICE32)]
    if inp.dv % 64 == 0:
        widths.append(("64", gdn.GDN_FLAG_SLICE64))
    for fmt_name, fmt in (("fp16", 0), ("wide", gdn.GDN_FLAG_WIDE_RANGE)):
        res = {}
        for name, flag in widths:
            o, s = _run(gdn, inp, flag | fmt | extra)
            eo, es = out_err(o, o_ref), state_err(s, s_ref)
            print(f"\n[slices] {inp.name or 'case'} {fmt_name} rows {name}: out {eo:.3e} state {es:.3e}")
            assert np.all(np.isfinite(o)) and np.all(np.isfinite(s))
            assert eo <= OUT_TOL and es <= STATE_TOL, (fmt_name, name, eo, es)
            res[name] = (o, s)
        # every width forms each column's products in the same order: bit for bit the same
        for name in res:
            assert np.array_equal(res["32"][0], res[name][0]) and np.array_equal(res["32"][1], res[name][1]), \
                (fmt_name, name)


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (32, 64), (128, 64), (64, 128), (128, 32), (32, 32)])
def test_dense_both_widths(gdn, dk, dv):
    inp = make_gdn_inputs(B=2, T=300, Hk=2, Hv=4, dk=dk, dv=dv, seed=dk + dv, init_std=0.1)
    _both_widths_against_oracle(gdn, inp)


def test_packed_with_empty_sequences_both_widths(gdn):
    inp = make_gdn_inputs(lengths=[0, 70, 0, 1, 64, 130, 0, 300], Hk=2, Hv=4, dk=128, dv=128, seed=101,
                          init_std=0.2)
    _both_widths_against_oracle(gdn, inp)


def test_many_chunks_slow_decay_both_widths(gdn):
    inp = make_gdn_inputs(B=1, T=1100, Hk=1, Hv=2, dk=128, dv=128, seed=102, g_scale=0.01, init_std=0.05)
    _both_widths_against_oracle(gdn, inp)


def test_no_decay_strong_writes_both_widths(gdn):
    inp = make_gdn_inputs(B=1, T=400, Hk=1, Hv=2, dk=128, dv=128, seed=103, init_std=0.1)
    inp.g[:] = 0.0
    inp.beta[:] = 0.999
    _both_widths_against_oracle(gdn, inp)


def _normalised(x):
    return x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), 1e-6)


def test_norm_qk_both_widths(gdn):
    """In-kernel q/k normalisation: the oracle runs on the float64-normalised bf16 inputs."""
    import oracle

    inp = make_gdn_inputs(lengths=[70, 0, 200, 5], Hk=2, Hv=4, dk=128, dv=128, seed=104, normalize_qk=False,
                          init_std=0.1)
    ref = oracle.prefill(_normalised(inp.q64()), _normalised(inp.k64()), inp.v64(), inp.g64(), inp.beta64(),
                         inp.cu_seqlens, inp.init64(), B=inp.B)
    _both_widths_against_oracle(gdn, inp, extra=gdn.GDN_FLAG_L2NORM_QK, ref=ref)
