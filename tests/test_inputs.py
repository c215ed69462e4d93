"""Seeded input generator (CPU only)."""

import numpy as np
import pytest
import torch

from hybrid_linear_attention_prefill_gb300 import inputs as I


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10 ** rng.uniform(-20, 20, 100000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 3.3895314e38], dtype=np.float32)])
    ours = I.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = I.bf16_bits_to_f64(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_seeded_and_shapes():
    a = I.workload("t1024_h16")
    b = I.workload("t1024_h16")
    assert np.array_equal(a.q, b.q) and np.array_equal(a.g, b.g)
    assert a.q.shape == (1024, 16, 128) and a.v.shape == (1024, 16, 128) and a.g.shape == (1024, 16)
    assert np.all(a.g <= 0) and np.all((a.beta > 0) & (a.beta < 1))
    n = np.linalg.norm(a.q64(), axis=-1)
    assert np.all(np.abs(n - 1) < 4e-3)


def test_varlen_workload():
    w = I.workload("varlen32_hk16_hv32")
    L = np.diff(w.cu_seqlens)
    assert w.B == 32 and w.cu_seqlens[0] == 0 and w.cu_seqlens[-1] == w.total_tokens == 72102
    assert L.min() >= 200 and L.max() <= 4096
    assert np.sum(L % 64 == 0) == 1


@pytest.mark.parametrize("name", ["tiny_t64_d32", "t16381_hk16_hv32_carry"])
def test_other_workloads(name):
    w = I.workload(name)
    if name.startswith("t16381"):
        assert w.init.shape == (1, 32, 128, 128) and abs(float(w.init.std()) - 0.02) < 1e-3
        assert float(w.g.mean()) > -0.1
    else:
        assert w.init is None and w.total_tokens == 64
