"""GPU parity of the fused gate prologue (kda_prefill_fused,
kda_decode_step_fused): the kernels take raw q, k, the gate pre-activation z
and A, and must match the oracle's gate_prologue followed by its recurrence,
on every path (producer / consumer and single-CTA tensor-core kernels, the
CUDA-core kernel, decode)."""
import pytest
import torch

import oracle
import synth
from tests._parity import TOL, assert_close, assert_kernels_agree, compare_out, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_05_gb300 as m
    m.build()
    m.lib()
    return m


def raw_inputs(lengths, H, d, dtype, seed):
    """Raw q and k: the generator's vectors scaled by a random factor per
    row (not unit length); z ~ N(0, 1.5^2), A ~ N(0, 0.5^2)."""
    inp = synth.generate(lengths, H, d, d, dtype=dtype, s0_std=0.05, seed=seed)
    gen = torch.Generator().manual_seed(seed + 1)
    T = inp.q.shape[0]
    cast = torch.bfloat16 if dtype == "bf16" else torch.float32
    sq = torch.rand(T, H, 1, generator=gen) * 4 + 0.25
    sk = torch.rand(T, H, 1, generator=gen) * 4 + 0.25
    inp.q = (inp.q.float() * sq).to(cast)
    inp.k = (inp.k.float() * sk).to(cast)
    z = torch.randn(T, H, d, generator=gen) * 1.5
    A = torch.randn(H, d, generator=gen) * 0.5
    return inp, z, A


def oracle_fused(inp, z, A, q_scale):
    qh, kh, g = oracle.gate_prologue(to64(inp.q), to64(inp.k), to64(z), to64(A), q_scale)
    return oracle.prefill(qh, kh, to64(inp.v), g, to64(inp.beta),
                          S0=None if inp.S0 is None else to64(inp.S0),
                          cu_seqlens=inp.cu_seqlens.cpu().numpy())


CASES = [
    ("bf16", 128, [300, 0, 77, 130], 2, "split"),
    ("bf16", 128, [300, 0, 77, 130], 2, "single"),
    ("bf16", 128, [700], 3, "split"),
    ("fp32", 64, [65, 1, 200], 3, "simt"),
    ("bf16", 32, [129, 64], 2, "simt"),
]


@pytest.mark.parametrize("dtype,d,lengths,H,path", CASES)
def test_prefill_fused_matches_oracle(kda, dtype, d, lengths, H, path):
    inp, z, A = raw_inputs(lengths, H, d, dtype, 900 + d + len(lengths))
    g = inp.to("cuda")
    q_scale = d ** -0.5
    ws = None
    if path == "single":
        N = len(lengths)
        ws = torch.zeros(256 + (N * 4 + 255) // 256 * 256, dtype=torch.uint8, device="cuda")
    o, S = kda.kda_prefill_fused(g.q, g.k, g.v, z.cuda(), A.cuda(), g.beta, S0=g.S0,
                                 cu_seqlens=g.cu_seqlens, q_scale=q_scale, workspace=ws)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle_fused(inp, z, A, q_scale)
    compare_out(o, o_ref, TOL[dtype], "o")
    assert_close(to64(S), S_ref, TOL[dtype], "S_final")


def test_split_and_single_cta_fused_agree(kda):
    inp, z, A = raw_inputs([500, 64, 3], 2, 128, "bf16", 950)
    g = inp.to("cuda")
    zc, Ac = z.cuda(), A.cuda()
    o1, S1 = kda.kda_prefill_fused(g.q, g.k, g.v, zc, Ac, g.beta, S0=g.S0,
                                   cu_seqlens=g.cu_seqlens, q_scale=0.1)
    ws = torch.zeros(512, dtype=torch.uint8, device="cuda")
    o2, S2 = kda.kda_prefill_fused(g.q, g.k, g.v, zc, Ac, g.beta, S0=g.S0,
                                   cu_seqlens=g.cu_seqlens, q_scale=0.1, workspace=ws)
    torch.cuda.synchronize()
    assert_kernels_agree(o1, o2, "o")
    assert_kernels_agree(S1, S2, "S_final")


@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_decode_step_fused_matches_oracle(kda, d, dtype):
    inp, z, A = raw_inputs([1] * 33, 3, d, dtype, 960 + d)
    g = inp.to("cuda")
    S = g.S0.clone()
    q_scale = d ** -0.5
    o = kda.kda_decode_step_fused(g.q, g.k, g.v, z.cuda(), A.cuda(), g.beta, S, q_scale=q_scale)
    torch.cuda.synchronize()
    qh, kh, gg = oracle.gate_prologue(to64(inp.q), to64(inp.k), to64(z), to64(A), q_scale)
    o_ref, S_ref = oracle.decode_step(qh, kh, to64(inp.v), gg, to64(inp.beta), to64(inp.S0))
    compare_out(o, o_ref, TOL[dtype], "o")
    assert_close(to64(S), S_ref, TOL[dtype], "S")


def test_fused_entry_points_need_A(kda):
    inp, z, A = raw_inputs([64], 1, 128, "bf16", 970)
    g = inp.to("cuda")
    lib = kda.lib()
    rc = lib.kda_prefill_fused(None, None, None, None, None, None, None, None, 1, 0, 1, 128, 128,
                               0, 1.0, None, None, None, 0, None)
    assert rc == kda.KDA_ERR_INVALID_ARG
