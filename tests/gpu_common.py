"""Helpers shared by the GPU parity tests: upload seeded inputs, run the CUDA path
through the C ABI, run the oracle on the same values, and measure the errors."""

import numpy as np

OUT_TOL = 1e-2     # max|o - o_ref| <= OUT_TOL * max|o_ref|
STATE_TOL = 2e-3   # ||S - S_ref||_F / ||S_ref||_F <= STATE_TOL


def dev_inputs(inp, device="cuda"):
    import torch

    def t(a, dt=None):
        x = torch.from_numpy(np.ascontiguousarray(a))
        return (x.view(dt) if dt is not None else x).to(device)

    return dict(
        q=t(inp.q.view(np.int16), torch.bfloat16), k=t(inp.k.view(np.int16), torch.bfloat16),
        v=t(inp.v.view(np.int16), torch.bfloat16), g=t(inp.g), beta=t(inp.beta),
        cu=None if inp.cu_seqlens is None else t(inp.cu_seqlens),
        init=None if inp.init is None else t(inp.init))


def run_gpu(inp, want_final=True, init_override=None, stream=None):
    import torch
    from hybrid_linear_attention_prefill_gb300 import gdn

    d = dev_inputs(inp)
    Ttot = inp.total_tokens
    out = torch.full((Ttot, inp.Hv, inp.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    fin = (torch.full((inp.B, inp.Hv, inp.dv, inp.dk), float("nan"), device="cuda")
           if want_final else None)
    init = d["init"] if init_override is None else init_override
    st = gdn.gdn_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], init, out, fin,
                         inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, stream)
    gdn.check(st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), None if fin is None else fin.cpu().numpy()


def out_err(o, o_ref):
    if o_ref.size == 0:
        return 0.0
    return float(np.max(np.abs(o - o_ref)) / max(np.max(np.abs(o_ref)), 1e-30))


def state_err(s, s_ref):
    n = np.linalg.norm(s_ref)
    if n == 0:
        return float(np.linalg.norm(s))
    return float(np.linalg.norm(s - s_ref) / n)


def sub_problem(inp, seqs, heads):
    """Slice sequences and value heads (with their key heads) out of a problem, so the
    oracle can check a sample of a large workload one (sequence, head) pair at a time."""
    from hybrid_linear_attention_prefill_gb300.inputs import GdnInputs

    bounds = inp.seq_bounds()
    grp = inp.Hv // inp.Hk
    parts = []
    for b in seqs:
        s, e = bounds[b]
        for h in heads:
            hk = h // grp
            parts.append((b, h, s, e, hk))
    return parts


def oracle_pairs(inp, parts):
    """Oracle outputs and final states for (sequence, value head) pairs."""
    import oracle

    from hybrid_linear_attention_prefill_gb300.inputs import bf16_bits_to_f64

    res = []
    for b, h, s, e, hk in parts:
        init = None if inp.init is None else inp.init[b:b + 1, h:h + 1].astype(np.float64)
        o, f = oracle.prefill(bf16_bits_to_f64(inp.q[s:e, hk:hk + 1]),
                              bf16_bits_to_f64(inp.k[s:e, hk:hk + 1]),
                              bf16_bits_to_f64(inp.v[s:e, h:h + 1]),
                              inp.g[s:e, h:h + 1].astype(np.float64),
                              inp.beta[s:e, h:h + 1].astype(np.float64), None, init, B=1, T=e - s)
        res.append((o[:, 0], f[0, 0]))
    return res
