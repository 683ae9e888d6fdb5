"""GPU parity of kda_prefill_snapshots (prefix-state snapshots for a prefix
cache) against the oracle's prefill_snapshots, on the tensor-core paths
(producer / consumer and single-CTA) and the CUDA-core path.  The outputs o
and S_final must be those of kda_prefill bit for bit, and a snapshot must
resume the sequence: running the rest of it from the snapshot gives the same
outputs as the unbroken run."""
import pytest
import torch

import oracle
import synth
from tests._parity import TOL, assert_close, compare_out, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_05_gb300 as m
    m.build()
    m.lib()
    return m


def base_ws(n):
    return 256 + (n * 4 + 255) // 256 * 256


def oracle_snaps(inp, interval):
    cu = inp.cu_seqlens.cpu().numpy()
    return oracle.prefill_snapshots(to64(inp.q), to64(inp.k), to64(inp.v), to64(inp.log_alpha),
                                    to64(inp.beta), S0=None if inp.S0 is None else to64(inp.S0),
                                    cu_seqlens=cu, interval=interval)


CASES = [
    ("bf16", 128, [0, 64, 200, 256, 700, 1280], 2, 64, "split"),
    ("bf16", 128, [0, 64, 200, 256, 700, 1280], 2, 128, "single"),
    ("bf16", 128, [1000, 3, 512], 3, 256, "split"),
    ("fp32", 64, [0, 64, 130, 512], 2, 64, "simt"),
    ("bf16", 32, [300, 64], 2, 128, "simt"),
]


@pytest.mark.parametrize("dtype,d,lengths,H,interval,path", CASES)
def test_snapshots_match_oracle(kda, dtype, d, lengths, H, interval, path):
    inp = synth.generate(lengths, H, d, d, dtype=dtype, s0_std=0.05, seed=700 + interval + d)
    g = inp.to("cuda")
    N = len(lengths)
    ws = None
    if path == "single":
        ws = torch.zeros(base_ws(N), dtype=torch.uint8, device="cuda")
    o, S, snaps, off = kda.kda_prefill_snapshots(g.q, g.k, g.v, g.log_alpha, g.beta, S0=g.S0,
                                                 cu_seqlens=g.cu_seqlens, interval=interval,
                                                 workspace=ws)
    o1, S1 = kda.kda_prefill(g.q, g.k, g.v, g.log_alpha, g.beta, S0=g.S0,
                             cu_seqlens=g.cu_seqlens, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o, o1) and torch.equal(S, S1)
    o_ref, S_ref, snap_ref, off_ref = oracle_snaps(inp, interval)
    assert off.cpu().tolist() == off_ref.tolist()
    tol = TOL[dtype]
    compare_out(o, o_ref, tol, "o")
    assert_close(to64(S), S_ref, tol, "S_final")
    if snap_ref.shape[0]:
        assert_close(to64(snaps), snap_ref, tol, "snapshots")
    for n, L in enumerate(lengths):      # the last snapshot of a divisible length is S_final
        if L and L % interval == 0:
            assert torch.equal(snaps[int(off[n + 1]) - 1], S[n])


def test_single_sequence_snapshots_and_resume(kda):
    T, H, interval = 1000, 4, 128
    inp = synth.generate([T], H, 128, 128, dtype="bf16", s0_std=0.05, seed=731)
    g = inp.to("cuda")
    o, S, snaps, _ = kda.kda_prefill_snapshots(g.q, g.k, g.v, g.log_alpha, g.beta, S0=g.S0,
                                               interval=interval)
    torch.cuda.synchronize()
    assert snaps.shape[0] == T // interval
    o_ref, S_ref, snap_ref, _ = oracle_snaps(inp, interval)
    assert_close(to64(snaps), snap_ref, TOL["bf16"], "snapshots")
    # resume from snapshot j: the rest of the sequence reproduces the unbroken run
    j = 3
    t = (j + 1) * interval
    o2, S2 = kda.kda_prefill(g.q[t:].contiguous(), g.k[t:].contiguous(), g.v[t:].contiguous(),
                             g.log_alpha[t:].contiguous(), g.beta[t:].contiguous(),
                             S0=snaps[j:j + 1].contiguous())
    torch.cuda.synchronize()
    compare_out(o2, o_ref[t:], TOL["bf16"], "o after resuming")
    assert_close(to64(S2), S_ref, TOL["bf16"], "S_final after resuming")


def test_snapshot_arguments_are_checked(kda):
    inp = synth.generate([200, 300], 2, 128, 128, dtype="bf16", seed=732).to("cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_snapshots(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta,
                                  cu_seqlens=inp.cu_seqlens, interval=100)
    assert e.value.code == kda.KDA_ERR_INVALID_ARG
    # offsets that do not match floor(len / interval): error word set, nothing written
    off = torch.tensor([0, 2, 4], dtype=torch.int32, device="cuda")     # true counts: 3, 4
    snaps = torch.full((4, 2, 128, 128), 7.0, device="cuda")
    o = torch.full_like(inp.v, 5.0)
    ws = torch.zeros(kda.kda_prefill_workspace_bytes(2, 2, 128, 128), dtype=torch.uint8,
                     device="cuda")
    kda.kda_prefill_snapshots(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta,
                              cu_seqlens=inp.cu_seqlens, interval=64, snap_offsets=off,
                              snapshots=snaps, o=o, workspace=ws)
    torch.cuda.synchronize()
    assert ws[4:8].view(torch.int32).item() != 0
    assert torch.all(snaps == 7.0) and torch.all(o == 5.0)
