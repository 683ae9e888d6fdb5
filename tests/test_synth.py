"""The seeded input generator: shapes, determinism and distributions."""
import torch

import synth


def test_deterministic_and_shaped():
    a = synth.generate([5, 0, 7], 2, 16, 16, dtype="bf16", s0_std=0.02, seed=3)
    b = synth.generate([5, 0, 7], 2, 16, 16, dtype="bf16", s0_std=0.02, seed=3)
    for x, y in zip((a.q, a.k, a.v, a.log_alpha, a.beta, a.S0),
                    (b.q, b.k, b.v, b.log_alpha, b.beta, b.S0)):
        assert torch.equal(x, y)
    assert a.q.shape == (12, 2, 16) and a.q.dtype == torch.bfloat16
    assert a.log_alpha.dtype == torch.float32 and a.beta.shape == (12, 2)
    assert a.S0.shape == (3, 2, 16, 16)
    assert a.cu_seqlens.tolist() == [0, 5, 5, 12]


def test_distributions():
    a = synth.generate([4096], 4, 128, 128, dtype="fp32", seed=4)
    norms = a.k.norm(dim=-1)
    assert torch.allclose(norms, torch.ones_like(norms), atol=1e-5)
    assert (a.log_alpha <= 0).all() and (a.log_alpha > -5).all()
    assert (a.beta > 0).all() and (a.beta < 1).all()
    assert abs(a.q.std().item() - 128 ** -0.5) < 2e-3
    tiny = synth.workload_inputs(1)
    assert tiny.q.dtype == torch.float32 and tiny.q.shape == (64, 1, 16)
    assert (tiny.log_alpha < 0).all()


def test_varlen_lengths_in_range():
    lens = synth.draw_lengths(synth.WORKLOADS[3])
    assert len(lens) == 16 and all(512 <= x <= 16384 for x in lens)
    assert lens == synth.draw_lengths(synth.WORKLOADS[3])
