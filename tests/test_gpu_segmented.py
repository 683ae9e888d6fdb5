"""GPU parity of the chunk-group parallel prefill of one sequence
(kda_prefill_segmented): the sequence's chunks cut into segments that run at
once, joined by a scan of the segment states and a fix-up of the outputs
(the one-GPU form of KDA context parallelism, "[논문 리뷰] Kimi K3 Technical
Report", section 13; only the state passes between chunks, "Kimi 모델 분석",
section "순환을 GPU에 올리기").

Each case runs against the float64 oracle with the bound of the other parity
tests, and against kda_prefill on the same inputs (a different association of
the same sums: both within the bound of the oracle, so within twice the bound
of each other).  The workspace's timeout and abort
words must stay zero.
"""
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


def run_segmented(kda, inp, segments, o_dtype=None, S0=None):
    d = inp.to("cuda")
    T, H, dk = d.q.shape
    need = kda.kda_prefill_segmented_workspace_bytes(T, H, dk, dk, segments)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    o, S = kda.kda_prefill_segmented(d.q, d.k, d.v, d.log_alpha, d.beta,
                                     S0=d.S0 if S0 is None else S0, segments=segments,
                                     workspace=ws, o_dtype=o_dtype)
    torch.cuda.synchronize()
    words = ws[:28].view(torch.int32).cpu().tolist()
    assert words[2] == 0, "a device-side wait gave up"
    assert words[6] == 0, "the split kernel aborted"
    return o, S, need


def check(kda, inp, segments, o_dtype=None):
    o, S, need = run_segmented(kda, inp, segments, o_dtype)
    base = kda.kda_prefill_workspace_bytes(1, inp.q.shape[1], 128, 128)
    assert need > base, "shape should be cut into segments"
    o_ref, S_ref = oracle_prefill(inp)
    compare_out(o, o_ref, TOL["bf16"], "o (segmented)")
    assert_close(to64(S), S_ref, TOL["bf16"], "S_final (segmented)")
    d = inp.to("cuda")
    o1, S1 = kda.kda_prefill(d.q, d.k, d.v, d.log_alpha, d.beta, S0=d.S0, o_dtype=o_dtype)
    torch.cuda.synchronize()
    # both within the bound of the oracle, so within twice the bound of each other
    compare_out(o, to64(o1), 2 * TOL["bf16"], "o (segmented vs kda_prefill)")
    assert_close(to64(S), to64(S1), 2 * TOL["bf16"], "S_final (segmented vs kda_prefill)")


def test_prefill_h16_t4096_segmented(kda):
    # the short-prompt workload: 16 heads, 64 chunks, in two segments
    inp = synth.workload_inputs(2, device="cpu")
    check(kda, inp, 2)


def test_automatic_choice_cuts_the_short_prompt_in_two(kda):
    # 64 chunks x 16 heads: two segments of 32 chunks, 48 consumer chains
    auto = kda.kda_prefill_segmented_workspace_bytes(4096, 16, 128, 128, 0)
    assert auto == kda.kda_prefill_segmented_workspace_bytes(4096, 16, 128, 128, 2)
    assert auto > kda.kda_prefill_workspace_bytes(1, 16, 128, 128)
    # 24 heads would need 72 chains: not cut
    assert (kda.kda_prefill_segmented_workspace_bytes(4096, 24, 128, 128, 0) ==
            kda.kda_prefill_workspace_bytes(1, 24, 128, 128))


def test_automatic_choice_cuts_a_long_few_head_prompt(kda):
    inp = synth.generate([16384], 4, 128, 128, dtype="bf16", s0_std=0.05, seed=715)
    check(kda, inp, 0)


@pytest.mark.parametrize("segments", [2, 3, 4])
def test_segments_ragged_with_initial_state(kda, segments):
    inp = synth.generate([1000], 4, 128, 128, dtype="bf16", s0_std=0.05, seed=700 + segments)
    check(kda, inp, segments)


def test_segmented_fp32_output(kda):
    inp = synth.generate([777], 3, 128, 128, dtype="bf16", s0_std=0.05, seed=710)
    check(kda, inp, 3, o_dtype=torch.float32)


def test_segmented_wide_chunks(kda):
    # g = -5 everywhere: every chunk in two passes, the largest Gram factors
    inp = synth.generate([900], 4, 128, 128, dtype="bf16", s0_std=0.05, seed=711,
                         gate_shift=-5.0)
    check(kda, inp, 4)


def test_segmented_beta_two(kda):
    inp = synth.generate([640], 4, 128, 128, dtype="bf16", s0_std=0.05, seed=712)
    inp.beta.fill_(2.0)
    check(kda, inp, 3)


def test_segmented_in_place_resume(kda):
    # S_final may be S0 itself: segment 0 reads S0 before the scan writes it
    inp = synth.generate([700], 2, 128, 128, dtype="bf16", s0_std=0.05, seed=713)
    d = inp.to("cuda")
    S = d.S0.clone()
    need = kda.kda_prefill_segmented_workspace_bytes(700, 2, 128, 128, 3)
    assert need > kda.kda_prefill_workspace_bytes(1, 2, 128, 128)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    o, S2 = kda.kda_prefill_segmented(d.q, d.k, d.v, d.log_alpha, d.beta, S0=S, segments=3,
                                      S_final=S, workspace=ws)
    torch.cuda.synchronize()
    assert S2.data_ptr() == S.data_ptr()
    o_ref, S_ref = oracle_prefill(inp)
    compare_out(o, o_ref, TOL["bf16"], "o")
    assert_close(to64(S), S_ref, TOL["bf16"], "S_final")


def test_segmented_falls_back_when_it_cannot_cut(kda):
    # one chunk only, and too many heads for two segments: kda_prefill
    for lengths, H in (([60], 2), ([300], 64)):
        inp = synth.generate(lengths, H, 128, 128, dtype="bf16", s0_std=0.05, seed=714)
        T = sum(lengths)
        assert (kda.kda_prefill_segmented_workspace_bytes(T, H, 128, 128, 0)
                == kda.kda_prefill_workspace_bytes(1, H, 128, 128))
        o, S, _ = run_segmented(kda, inp, 0)
        o_ref, S_ref = oracle_prefill(inp)
        compare_out(o, o_ref, TOL["bf16"], "o")
        assert_close(to64(S), S_ref, TOL["bf16"], "S_final")
