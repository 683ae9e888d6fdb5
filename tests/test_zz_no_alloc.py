"""kda_prefill_noalloc: the prefill entry point for callers that cannot
allocate device memory (for example an engine that plans all device memory at
start-up and forbids allocation afterwards).  It must give the same results as
kda_prefill with a caller-allocated workspace, on repeated calls that reuse its
fixed scratch array.

This file is named so that pytest collects it last.
"""
import ctypes

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
    return m


def _noalloc_abi(lib, d, o, S_final):
    """Call the C ABI entry point directly."""
    T, H, dk = d.q.shape
    code = 0 if o.dtype == torch.bfloat16 else 2
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return lib.kda_prefill_noalloc(
        p(d.q), p(d.k), p(d.v), p(d.log_alpha), p(d.beta), p(d.S0), p(d.cu_seqlens),
        len(d.lengths), T, H, dk, d.v.shape[2], code, p(o), p(S_final),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("lengths,d", [([300, 0, 77, 130], 128), ([65, 1, 200], 64)])
def test_noalloc_matches_workspace_entry_point(kda, lengths, d):
    lib = kda.lib()
    tol = 2e-2
    for call in range(2):     # two calls in a row share the fixed scratch
        inp = synth.generate(lengths, 3, d, d, dtype="bf16", s0_std=0.05,
                             seed=500 + call + d)
        dv = inp.to("cuda")
        o_ref, S_ref = kda.kda_prefill(dv.q, dv.k, dv.v, dv.log_alpha, dv.beta,
                                       S0=dv.S0, cu_seqlens=dv.cu_seqlens)
        o = torch.full_like(o_ref, float("nan"))
        S = torch.full_like(S_ref, float("nan"))
        assert _noalloc_abi(lib, dv, o, S) == kda.KDA_OK
        torch.cuda.synchronize()
        assert_close(to64(o), to64(o_ref), tol, "o (call %d)" % call)
        assert_close(to64(S), to64(S_ref), tol, "S_final (call %d)" % call)
        if call == 1:
            # and against the float64 oracle, not only the other CUDA call
            o64, S64 = oracle_prefill(inp)
            compare_out(o, o64, TOL["bf16"], "o vs oracle")
            assert_close(to64(S), S64, TOL["bf16"], "S_final vs oracle")


def test_noalloc_one_sequence_through_the_wrapper(kda):
    # cu_seqlens = None: one sequence, no work-list kernel; the Python wrapper
    # of the same name.
    inp = synth.generate([333], 4, 128, 128, dtype="bf16", s0_std=0.05, seed=540)
    dv = inp.to("cuda")
    o_ref, S_ref = kda.kda_prefill(dv.q, dv.k, dv.v, dv.log_alpha, dv.beta, S0=dv.S0)
    o, S = kda.kda_prefill_noalloc(dv.q, dv.k, dv.v, dv.log_alpha, dv.beta, S0=dv.S0,
                                   o=torch.empty_like(o_ref), S_final=torch.empty_like(S_ref))
    torch.cuda.synchronize()
    assert_close(to64(o), to64(o_ref), 2e-2, "o")
    assert_close(to64(S), to64(S_ref), 2e-2, "S_final")


def test_noalloc_after_an_invalid_call(kda):
    # A call with an invalid cu_seqlens (cu[N] != total_tokens) writes nothing
    # (and, without a workspace, says so nowhere the caller can read); a later
    # valid call with fewer sequences must not see what it left in the array.
    lib = kda.lib()
    bad = synth.generate([40, 50, 60, 70, 80], 2, 64, 64, dtype="bf16", seed=541).to("cuda")
    bad.cu_seqlens = bad.cu_seqlens.clone()
    bad.cu_seqlens[-1] += 7
    o_bad = torch.full_like(bad.v, 3.0)
    assert _noalloc_abi(lib, bad, o_bad, None) == kda.KDA_OK
    torch.cuda.synchronize()
    assert torch.all(o_bad == 3.0), "an invalid cu_seqlens must leave o untouched"
    inp = synth.generate([90, 0, 31], 2, 64, 64, dtype="bf16", s0_std=0.05, seed=542)
    dv = inp.to("cuda")
    o = torch.full_like(dv.v, float("nan"))
    S = torch.full_like(dv.S0, float("nan"))
    assert _noalloc_abi(lib, dv, o, S) == kda.KDA_OK
    torch.cuda.synchronize()
    o64, S64 = oracle_prefill(inp)
    compare_out(o, o64, TOL["bf16"], "o")
    assert_close(to64(S), S64, TOL["bf16"], "S_final")


def test_noalloc_rejects_too_many_sequences(kda):
    lib = kda.lib()
    inp = synth.generate([1] * 4097, 1, 16, 16, dtype="bf16", seed=9).to("cuda")
    o = torch.empty_like(inp.v)
    assert _noalloc_abi(lib, inp, o, None) == kda.KDA_ERR_WORKSPACE
