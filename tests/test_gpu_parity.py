"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs.

Error measure: max |gpu - oracle| / RMS(oracle), per tensor; bound 2e-2 for
bf16 q/k/v (fp32 state), 1e-4 for fp32 q/k/v.  Full-size workloads are checked
on sampled heads and value columns (value columns evolve independently, so the
oracle's restricted run is exact for them).
"""
import numpy as np
import pytest
import torch

import synth
from tests._parity import TOL, assert_close, compare_out, oracle_prefill, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_05_gb300 as m
    m.build()
    m.lib()
    return m


def run_prefill(kda, inp, want_state=True, o_dtype=None):
    d = inp.to("cuda")
    o, S = kda.kda_prefill(d.q, d.k, d.v, d.log_alpha, d.beta, S0=d.S0,
                           cu_seqlens=d.cu_seqlens, want_state=want_state,
                           o_dtype=o_dtype)
    torch.cuda.synchronize()
    return o, S


def check_prefill(kda, inp, dtype, heads=None, cols=None, seg=None, o_dtype=None):
    o, S = run_prefill(kda, inp, o_dtype=o_dtype)
    o_ref, S_ref = oracle_prefill(inp, heads=heads, cols=cols, seg_tokens=seg)
    hi = list(range(inp.q.shape[1])) if heads is None else list(heads)
    ci = list(range(inp.v.shape[2])) if cols is None else list(cols)
    og = o[:, hi][:, :, ci]
    Sg = S[:, hi][:, :, :, ci]
    e1 = compare_out(og, o_ref, TOL[dtype], "o")
    e2 = assert_close(to64(Sg), S_ref, TOL[dtype], "S_final")
    return e1, e2


# --- the five workloads ---------------------------------------------------

def test_recurrent_tiny_fp32(kda):
    inp = synth.workload_inputs(1, device="cpu")
    check_prefill(kda, inp, "fp32")


def test_prefill_h16_t4096(kda):
    inp = synth.workload_inputs(2, device="cpu")
    check_prefill(kda, inp, "bf16")


def test_prefill_h16_t4096_fp32_output(kda):
    # bf16 inputs, fp32 output: the plain bound, with no output rounding.
    inp = synth.workload_inputs(2, device="cpu")
    check_prefill(kda, inp, "bf16", o_dtype=torch.float32)


def test_varlen16_h32_sampled_columns(kda):
    inp = synth.workload_inputs(3, device="cuda")
    check_prefill(kda, inp, "bf16", cols=[0, 17, 38, 63, 64, 90, 111, 127])


def test_varlen16_h32_sampled_columns_fp32_output(kda):
    # bf16 inputs, fp32 output: the plain bound on the varlen workload.
    inp = synth.workload_inputs(3, device="cuda")
    check_prefill(kda, inp, "bf16", cols=[3, 29, 64, 100, 127], o_dtype=torch.float32)


def test_prefill_h32_t1m_sampled(kda):
    inp = synth.workload_inputs(4, device="cuda")
    check_prefill(kda, inp, "bf16", heads=[0, 31], cols=[0, 5, 64, 127],
                  seg=1 << 17)


def test_prefill_h32_t1m_sampled_fp32_output(kda):
    # The plain bound (no output rounding) on the 1M-token workload.
    inp = synth.workload_inputs(4, device="cuda")
    check_prefill(kda, inp, "bf16", heads=[7, 20], cols=[1, 66, 126],
                  seg=1 << 17, o_dtype=torch.float32)


def test_decode_1024x32(kda):
    inp = synth.workload_inputs(5, device="cuda")
    import oracle
    S = inp.S0.clone()
    o = kda.kda_decode_step(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, S)
    torch.cuda.synchronize()
    # Every 8th sequence (all heads, all columns) plus the last one.
    n = torch.tensor(list(range(0, 1024, 8)) + [1023], device="cuda")
    sel = lambda t: to64(t.index_select(0, n))
    o_ref, S_ref = oracle.decode_step(sel(inp.q), sel(inp.k), sel(inp.v),
                                      sel(inp.log_alpha), sel(inp.beta), sel(inp.S0))
    assert_close(sel(o), o_ref, TOL["bf16"], "o", bf16_out=True)
    assert_close(sel(S), S_ref, TOL["bf16"], "S")


# --- head sizes, dtypes, ragged tails ---------------------------------------

RAGGED = [1, 63, 64, 65, 130, 17]


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_head_sizes_ragged(kda, d, dtype):
    inp = synth.generate(RAGGED, 3, d, d, dtype=dtype, s0_std=0.1, seed=100 + d)
    check_prefill(kda, inp, dtype)


def test_empty_sequences(kda):
    inp = synth.generate([0, 5, 0, 70, 0], 2, 64, 64, dtype="fp32", s0_std=0.1, seed=7)
    o, S = run_prefill(kda, inp)
    o_ref, S_ref = oracle_prefill(inp)
    assert_close(to64(o), o_ref, TOL["fp32"], "o")
    assert_close(to64(S), S_ref, TOL["fp32"], "S")
    for n in (0, 2, 4):   # an empty sequence returns its S0 unchanged
        assert torch.equal(S[n].cpu(), inp.S0[n])


def test_zero_tokens(kda):
    S0 = torch.randn(1, 2, 32, 32, device="cuda")
    e = torch.empty(0, 2, 32, device="cuda")
    o, S = kda.kda_prefill(e, e, e, e, torch.empty(0, 2, device="cuda"), S0=S0)
    torch.cuda.synchronize()
    assert o.shape == (0, 2, 32)
    assert torch.equal(S, S0)


def test_lower_bound_stress(kda):
    # log_alpha = -5 everywhere: the lower bound of the decay.
    for dtype in ("fp32", "bf16"):
        inp = synth.generate([300, 77], 2, 128, 128, dtype=dtype, s0_std=0.1,
                             seed=11, gate_shift=-5.0)
        check_prefill(kda, inp, dtype)


def test_beta_two(kda):
    # beta = 2 (a reflection when alpha = 1); the kernels must not assume beta <= 1.
    inp = synth.generate([200], 2, 64, 64, dtype="fp32", s0_std=0.1, seed=12)
    inp.beta.fill_(2.0)
    check_prefill(kda, inp, "fp32")


@pytest.mark.parametrize("gates", ["alpha_one", "realistic"])
def test_beta_two_tensor_cores(kda, gates):
    # beta = 2 on the tensor-core path (bf16, d = 128) with 180 units, more
    # than half the SMs: the single-CTA kernel.
    shift = 0.0 if gates == "alpha_one" else None
    inp = synth.generate([130, 64, 255] * 3, 20, 128, 128, dtype="bf16", s0_std=0.05,
                         seed=16 + len(gates), gate_shift=shift)
    inp.beta.fill_(2.0)
    check_prefill(kda, inp, "bf16")
    check_prefill(kda, inp, "bf16", o_dtype=torch.float32)


# --- chaining, in-place resume, decode == prefill ---------------------------

def test_resume_in_place(kda):
    T1, T2 = 150, 201
    inp = synth.generate([T1 + T2], 4, 128, 128, dtype="bf16", s0_std=0.05, seed=13)
    d = inp.to("cuda")
    o1, S = kda.kda_prefill(d.q[:T1], d.k[:T1], d.v[:T1], d.log_alpha[:T1],
                            d.beta[:T1], S0=d.S0)
    o2, S2 = kda.kda_prefill(d.q[T1:].contiguous(), d.k[T1:].contiguous(),
                             d.v[T1:].contiguous(), d.log_alpha[T1:].contiguous(),
                             d.beta[T1:].contiguous(), S0=S, S_final=S)
    torch.cuda.synchronize()
    assert S2.data_ptr() == S.data_ptr()
    o_ref, S_ref = oracle_prefill(inp)
    compare_out(torch.cat([o1, o2]), o_ref, TOL["bf16"], "o")
    assert_close(to64(S), S_ref, TOL["bf16"], "S")


def test_decode_chain_equals_prefill(kda):
    T, H, d = 70, 2, 64
    inp = synth.generate([T], H, d, d, dtype="fp32", s0_std=0.1, seed=14)
    dv = inp.to("cuda")
    S = dv.S0.clone()
    outs = []
    for t in range(T):
        outs.append(kda.kda_decode_step(dv.q[t:t + 1], dv.k[t:t + 1], dv.v[t:t + 1],
                                        dv.log_alpha[t:t + 1], dv.beta[t:t + 1], S))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle_prefill(inp)
    compare_out(torch.cat(outs), o_ref, TOL["fp32"], "o")
    assert_close(to64(S), S_ref, TOL["fp32"], "S")


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_decode_head_sizes(kda, d, dtype):
    import oracle
    inp = synth.generate([1] * 37, 3, d, d, dtype=dtype, s0_std=0.1, seed=200 + d)
    dv = inp.to("cuda")
    S = dv.S0.clone()
    o = kda.kda_decode_step(dv.q, dv.k, dv.v, dv.log_alpha, dv.beta, S)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.decode_step(to64(inp.q), to64(inp.k), to64(inp.v),
                                      to64(inp.log_alpha), to64(inp.beta), to64(inp.S0))
    compare_out(o, o_ref, TOL[dtype], "o")
    assert_close(to64(S), S_ref, TOL[dtype], "S")


def test_decode_fp32_output(kda):
    import oracle
    inp = synth.generate([1] * 64, 4, 128, 128, dtype="bf16", s0_std=0.02, seed=300)
    dv = inp.to("cuda")
    S = dv.S0.clone()
    o = kda.kda_decode_step(dv.q, dv.k, dv.v, dv.log_alpha, dv.beta, S,
                            o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert o.dtype == torch.float32
    o_ref, S_ref = oracle.decode_step(to64(inp.q), to64(inp.k), to64(inp.v),
                                      to64(inp.log_alpha), to64(inp.beta), to64(inp.S0))
    assert_close(to64(o), o_ref, TOL["bf16"], "o")
    assert_close(to64(S), S_ref, TOL["bf16"], "S")


# --- device-side argument check ---------------------------------------------

def test_invalid_cu_seqlens_sets_error_word(kda):
    inp = synth.generate([10, 10], 1, 32, 32, dtype="fp32", seed=15).to("cuda")
    bad = torch.tensor([0, 15, 12], dtype=torch.int32, device="cuda")   # decreasing
    o = torch.full((20, 1, 32), 7.0, device="cuda")
    ws = torch.zeros(kda.kda_prefill_workspace_bytes(2, 1, 32, 32), dtype=torch.uint8,
                     device="cuda")
    kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, cu_seqlens=bad,
                    o=o, workspace=ws)
    torch.cuda.synchronize()
    assert ws.view(torch.int32)[1].item() != 0
    assert torch.all(o == 7.0)          # nothing written
    kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta,
                    cu_seqlens=inp.cu_seqlens, o=o, workspace=ws)
    torch.cuda.synchronize()
    assert ws.view(torch.int32)[1].item() == 0
