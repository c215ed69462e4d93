"""CUDA path vs the float64 oracle, element by element (GPU).

Tolerances: max|o - o_ref| <= 1e-2 max|o_ref| (bf16 outputs) and final-state
relative Frobenius error <= 2e-3 (fp32 state), both against the oracle run on
exactly the bf16 / fp32 values the GPU receives.
"""

import numpy as np
import pytest

from gpu_common import (OUT_TOL, STATE_TOL, oracle_pairs, out_err, run_gpu, state_err,
                        sub_problem)
from hybrid_linear_attention_prefill_gb300.inputs import make_gdn_inputs, workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hybrid_linear_attention_prefill_gb300 import build, gdn

    build.build()
    gdn.load()


def check_full(inp, want_final=True):
    import oracle

    o, s = run_gpu(inp, want_final=want_final)
    o_ref, s_ref = oracle.prefill_inputs(inp)
    eo = out_err(o, o_ref)
    print(f"\n[parity] {inp.name or 'case'} B={inp.B} T={inp.T} Hk={inp.Hk} Hv={inp.Hv} dk={inp.dk} "
          f"dv={inp.dv}: out {eo:.3e}" + (f" state {state_err(s, s_ref):.3e}" if want_final else ""))
    assert np.all(np.isfinite(o)), "non-finite outputs"
    assert eo <= OUT_TOL, f"output error {eo:.3e}"
    if want_final:
        es = state_err(s, s_ref)
        assert es <= STATE_TOL, f"state error {es:.3e}"
        for b in range(inp.B):  # every sequence, not just the aggregate
            assert state_err(s[b], s_ref[b]) <= STATE_TOL, f"sequence {b}"
    return o, s


# ---- the five workloads ---------------------------------------------------------

def test_workload_tiny():
    check_full(workload("tiny_t64_d32"))


def test_workload_t1024():
    check_full(workload("t1024_h16"))


def test_workload_t4096_headline():
    check_full(workload("t4096_hk16_hv32"))


def _check_sampled(inp, seqs, heads):
    o, s = run_gpu(inp)
    parts = sub_problem(inp, seqs, heads)
    bounds = inp.seq_bounds()
    for (b, h, st, en, _), (o_ref, s_ref) in zip(parts, oracle_pairs(inp, parts)):
        print(f"\n[parity] {inp.name} seq {b} head {h}: out {out_err(o[st:en, h], o_ref):.3e} "
              f"state {state_err(s[b, h], s_ref):.3e}")
        assert out_err(o[st:en, h], o_ref) <= OUT_TOL, f"seq {b} head {h} outputs"
        assert state_err(s[b, h], s_ref) <= STATE_TOL, f"seq {b} head {h} state"
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(s))
    return o, s


def test_workload_varlen32_sampled():
    inp = workload("varlen32_hk16_hv32")
    L = np.diff(inp.cu_seqlens)
    seqs = sorted({int(np.argmin(L)), int(np.argmax(L)), int(np.where(L % 64 == 0)[0][0]), 0, 31})
    _check_sampled(inp, seqs, [0, 1, 17, 31])


def test_workload_t16381_carry_sampled():
    _check_sampled(workload("t16381_hk16_hv32_carry"), [0], [0, 5, 30, 31])


# ---- edge cases ------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 5, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257, 383])
def test_ragged_lengths(T):
    check_full(make_gdn_inputs(B=2, T=T, Hk=2, Hv=4, dk=128, dv=128, seed=T, init_std=0.1))


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (128, 64), (64, 128), (32, 128), (128, 32)])
def test_head_dims(dk, dv):
    check_full(make_gdn_inputs(B=1, T=150, Hk=1, Hv=2, dk=dk, dv=dv, seed=dk + dv, init_std=0.1))


@pytest.mark.parametrize("Hk,Hv", [(1, 1), (3, 3), (2, 8), (4, 8)])
def test_head_groups(Hk, Hv):
    check_full(make_gdn_inputs(B=1, T=130, Hk=Hk, Hv=Hv, dk=64, dv=64, seed=Hk * 10 + Hv))


def test_packed_with_empty_sequences():
    inp = make_gdn_inputs(lengths=[0, 70, 0, 1, 64, 130, 0, 300], Hk=2, Hv=4, dk=128, dv=128, seed=7,
                          init_std=0.2)
    o, s = check_full(inp)
    for b in (0, 2, 6):  # empty sequences return their initial state exactly
        assert np.array_equal(s[b], inp.init[b])


def test_packed_dispatch_order_many_and_long_sequences():
    """The packed state carries run longest first through a device-built order (a counting sort
    on chunk counts, counts above 1022 sharing one bucket).  More than 1,024 sequences take the
    sort's loops more than once; one sequence of 1,100 chunks lands in the shared bucket; empty
    sequences sort last.  Every sequence is still carried exactly once, from its own state."""
    rng = np.random.default_rng(90)
    lengths = [int(x) for x in rng.integers(0, 140, 1500)]
    lengths[700] = 1100 * 64 - 5
    lengths[3] = 0
    inp = make_gdn_inputs(lengths=lengths, Hk=1, Hv=2, dk=32, dv=32, seed=91, init_std=0.1)
    o, s = check_full(inp)
    for b in [i for i, n in enumerate(lengths) if n == 0][:20]:
        assert np.array_equal(s[b], inp.init[b])


def test_slow_decay_many_chunks_with_carry():
    """g ~ -0.01 softplus keeps the initial state and early chunks alive across 16 chunks."""
    check_full(make_gdn_inputs(B=1, T=1000, Hk=2, Hv=4, dk=128, dv=128, seed=11, g_scale=0.01,
                               init_std=0.05))


def test_no_decay_strong_writes():
    inp = make_gdn_inputs(B=1, T=300, Hk=1, Hv=2, dk=128, dv=128, seed=12, init_std=0.1)
    inp.g[:] = 0.0
    inp.beta[:] = 0.999
    check_full(inp)


def test_strong_decay_resets():
    inp = make_gdn_inputs(B=1, T=300, Hk=1, Hv=2, dk=64, dv=64, seed=13, init_std=1.0)
    inp.g[:] = -30.0
    check_full(inp)


def test_without_final_state():
    check_full(make_gdn_inputs(B=2, T=100, Hk=1, Hv=2, dk=128, dv=128, seed=14), want_final=False)


def test_null_init_equals_zero_init():
    inp = make_gdn_inputs(B=2, T=90, Hk=1, Hv=2, dk=128, dv=128, seed=15)
    o1, s1 = run_gpu(inp)
    z = torch.zeros((2, 2, 128, 128), device="cuda")
    o2, s2 = run_gpu(inp, init_override=z)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_dense_equals_packed():
    inp = make_gdn_inputs(B=3, T=100, Hk=2, Hv=4, dk=128, dv=128, seed=16, init_std=0.1)
    o1, s1 = run_gpu(inp)
    inp.cu_seqlens = np.arange(4, dtype=np.int32) * 100
    inp.T = 300
    o2, s2 = run_gpu(inp)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_split_sequence_carry():
    """Running a prefix and then the rest from the carried state matches one run."""
    inp = make_gdn_inputs(B=1, T=256, Hk=1, Hv=2, dk=128, dv=128, seed=17, g_scale=0.05, init_std=0.1)
    o, s = run_gpu(inp)
    a = make_gdn_inputs(B=1, T=256, Hk=1, Hv=2, dk=128, dv=128, seed=17, g_scale=0.05, init_std=0.1)
    cut = 96
    for f in ("q", "k", "v", "g", "beta"):
        setattr(a, f, getattr(inp, f)[:cut].copy())
    a.T = cut
    o1, s1 = run_gpu(a)
    b = make_gdn_inputs(B=1, T=256, Hk=1, Hv=2, dk=128, dv=128, seed=17, g_scale=0.05, init_std=0.1)
    for f in ("q", "k", "v", "g", "beta"):
        setattr(b, f, getattr(inp, f)[cut:].copy())
    b.T = 256 - cut
    b.init = s1
    o2, s2 = run_gpu(b)
    import oracle

    o_ref, s_ref = oracle.prefill_inputs(inp)
    assert out_err(np.concatenate([o1, o2]), o_ref) <= OUT_TOL
    assert state_err(s2, s_ref) <= STATE_TOL
    # the split moves chunk boundaries, so only rounding may differ from the single run
    assert state_err(s2, s) <= 1e-3


def test_in_place_state_update():
    from gpu_common import dev_inputs
    from hybrid_linear_attention_prefill_gb300 import gdn

    inp = make_gdn_inputs(B=2, T=100, Hk=1, Hv=2, dk=128, dv=128, seed=18, init_std=0.1)
    o_ref, s_ref = run_gpu(inp)
    d = dev_inputs(inp)
    out = torch.empty((200, 2, 128), dtype=torch.bfloat16, device="cuda")
    st = d["init"].clone()
    gdn.check(gdn.gdn_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], None, st, out, st,
                              2, 100, 1, 2, 128, 128))
    torch.cuda.synchronize()
    assert np.array_equal(st.cpu().numpy(), s_ref)


def test_deterministic():
    inp = make_gdn_inputs(B=1, T=333, Hk=2, Hv=4, dk=128, dv=128, seed=19)
    o1, s1 = run_gpu(inp)
    o2, s2 = run_gpu(inp)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_side_stream():
    inp = make_gdn_inputs(B=1, T=200, Hk=1, Hv=2, dk=128, dv=128, seed=20)
    o1, s1 = run_gpu(inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, s2 = run_gpu(inp, stream=s)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_host_entry_matches_device_entry():
    from hybrid_linear_attention_prefill_gb300 import gdn

    inp = make_gdn_inputs(lengths=[100, 37, 200], Hk=2, Hv=4, dk=128, dv=128, seed=21, init_std=0.1)
    o_dev, s_dev = run_gpu(inp)
    out = np.zeros((inp.total_tokens, 4, 128), dtype=np.uint16)
    fin = np.zeros((3, 4, 128, 128), dtype=np.float32)
    gdn.check(gdn.gdn_prefill_host(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens, inp.init,
                                   out, fin, 3, inp.total_tokens, 2, 4, 128, 128, 0))
    from hybrid_linear_attention_prefill_gb300.inputs import bf16_bits_to_f32

    assert np.array_equal(bf16_bits_to_f32(out), o_dev) and np.array_equal(fin, s_dev)


@pytest.mark.parametrize("case", [
    dict(B=1, T=4096, Hk=4, Hv=8, dk=128, dv=128, init_std=0.1),            # dense: 8 token windows
    dict(lengths=[1500, 0, 2600, 77], Hk=3, Hv=6, dk=128, dv=64, init_std=0.1),  # packed: 3 head groups
    dict(B=2, T=3000, Hk=8, Hv=8, dk=64, dv=128),                             # 2 sequences, ragged last chunk
    dict(B=1, T=4096, Hk=8, Hv=16, dk=32, dv=32, init_std=0.1),              # small head dims
    # packed, 4 head groups whose state carries are large enough to run 64 state rows per CTA
    dict(lengths=("uniform", 60, 50, 600), Hk=4, Hv=8, dk=128, dv=128, init_std=0.1),
])
def test_host_entry_pipelined(case):
    """Large enough for gdn_prefill_host to overlap its copies with the kernels: token
    windows whose state carries hand the state on (dense) or head groups on separate
    streams (packed). Bitwise the device entry's results, pinned or pageable."""
    import torch
    from hybrid_linear_attention_prefill_gb300 import gdn
    from hybrid_linear_attention_prefill_gb300.inputs import bf16_bits_to_f32

    inp = make_gdn_inputs(seed=24, **case)
    o_dev, s_dev = run_gpu(inp)
    B, Tt = inp.B, inp.total_tokens
    T = inp.T if inp.cu_seqlens is None else Tt
    for pin in (True, False):
        def host(a):
            t = torch.from_numpy(np.ascontiguousarray(a))
            return t.pin_memory() if pin else t
        out = host(np.zeros((Tt, inp.Hv, inp.dv), dtype=np.int16))
        fin = host(np.zeros((B, inp.Hv, inp.dv, inp.dk), dtype=np.float32))
        init = None if inp.init is None else host(inp.init)
        cu = None if inp.cu_seqlens is None else host(inp.cu_seqlens)
        gdn.check(gdn.gdn_prefill_host(host(inp.q.view(np.int16)), host(inp.k.view(np.int16)),
                                       host(inp.v.view(np.int16)), host(inp.g), host(inp.beta), cu, init,
                                       out, fin, B, T, inp.Hk, inp.Hv, inp.dk, inp.dv, 0))
        o_host = bf16_bits_to_f32(out.numpy().view(np.uint16))
        assert np.array_equal(o_host, o_dev) and np.array_equal(fin.numpy(), s_dev)
    # no final state requested: the windows still hand the state on inside the library
    out = np.zeros((Tt, inp.Hv, inp.dv), dtype=np.int16)
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens
    gdn.check(gdn.gdn_prefill_host(inp.q.view(np.int16), inp.k.view(np.int16), inp.v.view(np.int16), inp.g,
                                   inp.beta, cu, inp.init, out, None, B, T, inp.Hk, inp.Hv, inp.dk, inp.dv, 0))
    assert np.array_equal(bf16_bits_to_f32(out.view(np.uint16)), o_dev)


def test_misaligned_device_pointer_rejected():
    from gpu_common import dev_inputs
    from hybrid_linear_attention_prefill_gb300 import gdn

    inp = make_gdn_inputs(B=1, T=64, Hk=1, Hv=1, dk=128, dv=128, seed=22)
    d = dev_inputs(inp)
    buf = torch.empty(64 * 128 + 1, dtype=torch.bfloat16, device="cuda")
    out = buf[1:]  # 2-byte offset
    assert gdn.gdn_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], None, None, out, None,
                           1, 64, 1, 1, 128, 128) == gdn.GDN_ERR_ALIGN


def test_corrupt_cu_seqlens_stays_in_bounds():
    """Out-of-range boundaries are clamped on the device: no fault, finite results, and
    the malformed array is reported as a status bit."""
    from hybrid_linear_attention_prefill_gb300 import gdn

    gdn.gdn_device_status()  # clear
    inp = make_gdn_inputs(lengths=[50, 50], Hk=1, Hv=1, dk=64, dv=64, seed=23)
    inp.cu_seqlens = np.array([0, 5000, 100], dtype=np.int32)
    o, s = run_gpu(inp)
    assert np.all(np.isfinite(s))
    rc, bits = gdn.gdn_device_status()
    assert rc == gdn.GDN_OK and bits == gdn.GDN_STATUS_BAD_CU_SEQLENS
