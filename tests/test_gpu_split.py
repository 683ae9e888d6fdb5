"""GPU parity of the producer / consumer prefill (the path for batches with
few (sequence, head) units).

kda_prefill takes it when the units fill at most half of the SMs and the
workspace has room for the operand ring (kda_prefill_workspace_bytes returns
that size).  A workspace of only the base size selects the single-CTA kernel
for the same call, so every case here runs both and checks

  * each against the float64 oracle (the bf16 bound of the other parity
    tests, for both kernels), and
  * the two against each other: they evaluate the same products on the same
    fp16 / bf16 operands in the same order (the split kernel only moves the
    state-independent phases to other CTAs), so o and S_final agree to a
    couple of bf16 ulps at most (tests._parity.assert_kernels_agree);
  * that the split kernel really ran (its job counter in the workspace) and
    no wait gave up (the timeout word).
"""
import pytest
import torch

import synth
from tests._parity import (TOL, assert_close, assert_kernels_agree, compare_out, oracle_prefill,
                           to64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_05_gb300 as m
    m.build()
    m.lib()
    return m


def base_workspace_bytes(num_seqs):
    """The work-list part of the workspace only (no ring)."""
    return 256 + (num_seqs * 4 + 255) // 256 * 256


def run_both(kda, inp, o_dtype=None):
    d = inp.to("cuda")
    N = len(inp.lengths)
    T, H, dk = d.q.shape
    need = kda.kda_prefill_workspace_bytes(N, H, dk, dk)
    assert need > base_workspace_bytes(N), "shape should qualify for the split kernel"
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    o_s, S_s = kda.kda_prefill(d.q, d.k, d.v, d.log_alpha, d.beta, S0=d.S0,
                               cu_seqlens=d.cu_seqlens, workspace=ws, o_dtype=o_dtype)
    torch.cuda.synchronize()
    words = ws[:24].view(torch.int32).cpu()
    jobs = int(ws[16:24].view(torch.int64).item())
    ws1 = torch.zeros(base_workspace_bytes(N), dtype=torch.uint8, device="cuda")
    o_1, S_1 = kda.kda_prefill(d.q, d.k, d.v, d.log_alpha, d.beta, S0=d.S0,
                               cu_seqlens=d.cu_seqlens, workspace=ws1, o_dtype=o_dtype)
    torch.cuda.synchronize()
    assert int(words[2]) == 0, "a device-side wait gave up"
    assert int(ws[24:28].view(torch.int32).item()) == 0, "the split kernel aborted"
    maxlen = max(inp.lengths)
    assert int(words[3]) == maxlen
    # every job was claimed (each producer also makes one failed claim)
    assert jobs >= N * H * ((maxlen + 63) // 64)
    return (o_s, S_s), (o_1, S_1)


def check(kda, inp, o_dtype=None):
    (o_s, S_s), (o_1, S_1) = run_both(kda, inp, o_dtype=o_dtype)
    o_ref, S_ref = oracle_prefill(inp)
    compare_out(o_s, o_ref, TOL["bf16"], "o (split)")
    assert_close(to64(S_s), S_ref, TOL["bf16"], "S_final (split)")
    compare_out(o_1, o_ref, TOL["bf16"], "o (single-CTA)")
    assert_close(to64(S_1), S_ref, TOL["bf16"], "S_final (single-CTA)")
    assert_kernels_agree(o_s, o_1, "o (split vs single-CTA)")
    assert_kernels_agree(S_s, S_1, "S_final (split vs single-CTA)")


CASES = {
    "one_seq_ragged": ([1000], 3),
    "varlen_empty_ragged": ([0, 300, 0, 130, 64, 1, 65], 2),
    "one_unit_long": ([5000], 1),
    "many_chunks_few_units": ([20000], 4),
    # more sequences than a warp's lanes: the producers' table of sequence
    # ranges is filled in two strides; 76 units is the split path's maximum on
    # 152 SMs (half of them)
    "many_seqs": ([(37 * i) % 257 for i in range(40)], 1),
    "max_units": ([(53 * i + 11) % 193 for i in range(76)], 1),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_split_matches_single_cta_and_oracle(kda, name):
    lengths, H = CASES[name]
    inp = synth.generate(lengths, H, 128, 128, dtype="bf16", s0_std=0.05, seed=600 + len(name))
    check(kda, inp)


def test_split_fp32_output(kda):
    inp = synth.generate([700, 129], 3, 128, 128, dtype="bf16", s0_std=0.05, seed=611)
    check(kda, inp, o_dtype=torch.float32)


def test_split_wide_chunks_mixed(kda):
    # Stretches of log_alpha = -5 (the lower bound) make some chunks' decay
    # span too wide for one pass; they are processed as two 32-row steps while
    # their neighbours take one.
    inp = synth.generate([900, 333], 2, 128, 128, dtype="bf16", s0_std=0.05, seed=612)
    g = inp.log_alpha
    for a, b in ((40, 200), (450, 470), (700, 900), (1000, 1100)):
        g[a:b] = -5.0
    check(kda, inp)


def test_split_all_wide(kda):
    inp = synth.generate([640, 77], 2, 128, 128, dtype="bf16", s0_std=0.05, seed=613,
                         gate_shift=-5.0)
    check(kda, inp)


def test_split_all_wide_fp32_output(kda):
    # fp32 output shows the products' rounding without the bf16 output
    # rounding on top; g = -5 makes every chunk two-pass, with the largest
    # Gram factors.
    inp = synth.generate([2000, 333], 4, 128, 128, dtype="bf16", s0_std=0.05, seed=7,
                         gate_shift=-5.0)
    check(kda, inp, o_dtype=torch.float32)


@pytest.mark.parametrize("gates", ["alpha_one", "realistic"])
def test_split_beta_two(kda, gates):
    # beta = 2 on both tensor-core kernels ("Kimi 모델 분석", section "반사가
    # 계층을 바꿈": with alpha = 1 and a unit key the step is the reflection
    # I - 2 k k^T).  T = (I + A)^{-1} Diag(beta) and the fp16 operands grow
    # with beta; nothing in the kernels may assume beta <= 1.
    shift = 0.0 if gates == "alpha_one" else None
    inp = synth.generate([777, 64, 200], 2, 128, 128, dtype="bf16", s0_std=0.05,
                         seed=620 + len(gates), gate_shift=shift)
    inp.beta.fill_(2.0)
    check(kda, inp)
    check(kda, inp, o_dtype=torch.float32)


def test_split_back_to_back_reuses_workspace(kda):
    # Two calls on one workspace: the work-list kernel clears the hand-over
    # flags and counters in between.
    inp = synth.generate([400, 250], 2, 128, 128, dtype="bf16", s0_std=0.05, seed=614)
    d = inp.to("cuda")
    N, H = 2, 2
    ws = torch.zeros(kda.kda_prefill_workspace_bytes(N, H, 128, 128), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for _ in range(2):
        o, S = kda.kda_prefill(d.q, d.k, d.v, d.log_alpha, d.beta, S0=d.S0,
                               cu_seqlens=d.cu_seqlens, workspace=ws)
        torch.cuda.synchronize()
        outs.append((o.clone(), S.clone()))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
    assert int(ws[8:12].view(torch.int32).item()) == 0


def test_split_ignores_workspace_contents(kda):
    # The workspace may hold anything on entry (the binding passes torch.empty);
    # in particular the caller-owned timeout word may already have bit 1 set.
    inp = synth.generate([3000], 4, 128, 128, dtype="bf16", s0_std=0.05, seed=615)
    d = inp.to("cuda")
    need = kda.kda_prefill_workspace_bytes(1, 4, 128, 128)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    o, S = kda.kda_prefill(d.q, d.k, d.v, d.log_alpha, d.beta, S0=d.S0, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[24:28].view(torch.int32).item()) == 0, "the split kernel aborted"
    ws1 = torch.zeros(base_workspace_bytes(1), dtype=torch.uint8, device="cuda")
    o1, S1 = kda.kda_prefill(d.q, d.k, d.v, d.log_alpha, d.beta, S0=d.S0, workspace=ws1)
    torch.cuda.synchronize()
    assert_kernels_agree(o, o1, "o")
    assert_kernels_agree(S, S1, "S_final")


def test_split_abort_path(kda, monkeypatch):
    # The bounded waits' abort path, run on purpose through the library's test
    # hook: the producers exit without publishing anything and every wait
    # gives up after about 2^20 cycles.  The call must return (every CTA
    # exits), with the timeout bit and the abort word set and o untouched; the
    # next normal call on the same workspace must be correct.  Nothing here
    # traps or waits without a bound.
    inp = synth.generate([700, 300], 2, 128, 128, dtype="bf16", s0_std=0.05, seed=630)
    d = inp.to("cuda")
    need = kda.kda_prefill_workspace_bytes(2, 2, 128, 128)
    assert need > base_workspace_bytes(2)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    o = torch.full_like(d.v, 5.0)
    S = torch.full_like(d.S0, 5.0)
    monkeypatch.setenv("KDA_TEST_STARVE_CONSUMERS", "1")
    kda.kda_prefill(d.q, d.k, d.v, d.log_alpha, d.beta, S0=d.S0, cu_seqlens=d.cu_seqlens,
                    o=o, S_final=S, workspace=ws)
    torch.cuda.synchronize()
    monkeypatch.delenv("KDA_TEST_STARVE_CONSUMERS")
    words = ws[:28].view(torch.int32).cpu().tolist()
    assert words[2] & 2, "the timeout bit must be set"
    assert words[6] != 0, "the abort word must be set"
    assert torch.all(o == 5.0) and torch.all(S == 5.0), "an aborted launch writes no result"
    # the next call: the work-list kernel clears the flags and the abort word
    # (the timeout word is the caller's to clear)
    ws[8:12].zero_()
    o2, S2 = kda.kda_prefill(d.q, d.k, d.v, d.log_alpha, d.beta, S0=d.S0,
                             cu_seqlens=d.cu_seqlens, workspace=ws)
    torch.cuda.synchronize()
    words = ws[:28].view(torch.int32).cpu().tolist()
    assert words[2] == 0 and words[6] == 0
    o_ref, S_ref = oracle_prefill(inp)
    compare_out(o2, o_ref, TOL["bf16"], "o after the aborted call")
    assert_close(to64(S2), S_ref, TOL["bf16"], "S_final after the aborted call")
