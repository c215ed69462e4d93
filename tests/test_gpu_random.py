"""Seeded random configurations against the oracle (GPU).

Each case draws, from its own seed: dense or packed (with empty and single-token sequences among
the lengths), the key/value head counts and their ratio, dk and dv, the decay scale, an initial
state or none, and the entry flags (slice width 16 / 32 / 64 / the library's choice, in-kernel q/k
normalisation, the wide-range operand format).  Sizes stay small enough for the oracle to finish in about a second each, and
large enough to span several chunks and a ragged tail."""

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


def _draw(seed, gdn):
    r = np.random.default_rng(1000 + seed)
    dk = int(r.choice([32, 64, 128]))
    dv = int(r.choice([32, 64, 128]))
    Hk = int(r.choice([1, 2, 3, 4]))
    Hv = Hk * int(r.choice([1, 2, 4]))
    g_scale = float(r.choice([1.0, 0.1, 0.01]))
    init_std = None if r.random() < 0.3 else 0.1
    normalize = r.random() < 0.75
    if r.random() < 0.5:
        kw = dict(B=int(r.integers(1, 4)), T=int(r.integers(1, 2000 if r.random() < 0.3 else 600)))
    else:
        n = int(r.integers(2, 12))
        lengths = [int(x) for x in r.integers(0, 400, n)]
        lengths[int(r.integers(0, n))] = 0
        lengths[int(r.integers(0, n))] = 1
        kw = dict(lengths=lengths)
    flags = int(r.choice([0, gdn.GDN_FLAG_SLICE16, gdn.GDN_FLAG_SLICE32] +
                         ([gdn.GDN_FLAG_SLICE64] if dv % 64 == 0 else [])))
    if not normalize:
        flags |= gdn.GDN_FLAG_L2NORM_QK
    if r.random() < 0.25:  # the wide-range (bf16 hi / lo) state carry
        flags |= gdn.GDN_FLAG_WIDE_RANGE
    inp = make_gdn_inputs(Hk=Hk, Hv=Hv, dk=dk, dv=dv, seed=2000 + seed, g_scale=g_scale, init_std=init_std,
                          normalize_qk=normalize, **kw)
    return inp, flags


def _normalised(x):
    return x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), 1e-6)


@pytest.mark.parametrize("seed", range(40))
def test_random_configuration(gdn, seed):
    import oracle

    inp, flags = _draw(seed, gdn)
    d = dev_inputs(inp)
    out = torch.full((inp.total_tokens, inp.Hv, inp.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    fin = torch.full((inp.B, inp.Hv, inp.dv, inp.dk), float("nan"), device="cuda")
    gdn.check(gdn.gdn_prefill_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"], out, fin,
                                 inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, flags))
    torch.cuda.synchronize()
    o, s = out.float().cpu().numpy(), fin.cpu().numpy()
    if flags & gdn.GDN_FLAG_L2NORM_QK:
        o_ref, s_ref = oracle.prefill(_normalised(inp.q64()), _normalised(inp.k64()), inp.v64(), inp.g64(),
                                      inp.beta64(), inp.cu_seqlens, inp.init64(), B=inp.B,
                                      T=None if inp.cu_seqlens is not None else inp.T)
    else:
        o_ref, s_ref = oracle.prefill_inputs(inp)
    desc = (f"B={inp.B} T={inp.T} packed={inp.cu_seqlens is not None} Hk={inp.Hk} Hv={inp.Hv} dk={inp.dk} "
            f"dv={inp.dv} flags={flags:#x}")
    assert np.all(np.isfinite(s)), desc
    if inp.total_tokens > 0:
        assert np.all(np.isfinite(o)), desc
        assert out_err(o, o_ref) <= OUT_TOL, desc
    assert state_err(s, s_ref) <= STATE_TOL, desc
