"""kda_prefill_host: one sequence whose inputs and output live in host
memory, pipelined over segments.  It must equal kda_prefill on device
buffers bit for bit (the state passes between segments at a chunk boundary,
in fp32), for segment counts of one and several and a ragged last segment,
on the tensor-core and CUDA-core paths."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_05_gb300 as m
    m.build()
    m.lib()
    return m


@pytest.mark.parametrize("T,H,d,dtype,seg", [
    (1000, 4, 128, "bf16", 256),       # several segments, ragged last one
    (4096, 2, 128, "bf16", 1024),
    (300, 3, 128, "bf16", 4096),       # one segment
    (500, 2, 64, "fp32", 128),         # the CUDA-core path
])
def test_host_prefill_equals_device_prefill(kda, T, H, d, dtype, seg):
    inp = synth.generate([T], H, d, d, dtype=dtype, s0_std=0.05, seed=1000 + T)
    g = inp.to("cuda")
    o_ref, S_ref = kda.kda_prefill(g.q, g.k, g.v, g.log_alpha, g.beta, S0=g.S0)
    pin = lambda t: t.contiguous().pin_memory()
    qh, kh, vh, gh, bh = (pin(x) for x in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta))
    oh = torch.empty(o_ref.shape, dtype=o_ref.dtype).pin_memory()
    S = torch.empty_like(S_ref)
    hp = kda.HostPrefill(H, d, g.q.dtype, segment_tokens=seg)
    hp(qh, kh, vh, gh, bh, oh, S0=g.S0, S_final=S)
    hp.compute.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(oh, o_ref.cpu())
    assert torch.equal(S, S_ref)


def test_host_prefill_checks_its_arguments(kda):
    lib = kda.lib()
    assert lib.kda_prefill_host_staging_bytes(4, 128, 128, 0, 100) == 0     # not a multiple of 64
    assert lib.kda_prefill_host_staging_bytes(4, 128, 128, 0, 128) > 0
    rc = lib.kda_prefill_host(None, None, None, None, None, None, 10, 1, 128, 128, 0, None, None,
                              None, 0, 64, None, None, None)
    assert rc == kda.KDA_ERR_INVALID_ARG


def test_host_prefill_back_to_back_calls(kda):
    # Two calls on one staging area, enqueued without a host sync in between:
    # the second call's first copy in must wait for the first call's compute
    # on the same slots.
    H, d, seg = 4, 128, 512
    ins = [synth.generate([3000], H, d, d, dtype="bf16", s0_std=0.05, seed=1100 + i)
           for i in range(2)]
    refs = []
    for inp in ins:
        g = inp.to("cuda")
        refs.append(kda.kda_prefill(g.q, g.k, g.v, g.log_alpha, g.beta, S0=g.S0))
    pin = lambda t: t.contiguous().pin_memory()
    hp = kda.HostPrefill(H, d, torch.bfloat16, segment_tokens=seg)
    outs = []
    for inp, (o_ref, S_ref) in zip(ins, refs):
        oh = torch.empty(o_ref.shape, dtype=o_ref.dtype).pin_memory()
        S = torch.empty_like(S_ref)
        S0 = inp.S0.cuda()
        # the host inputs stay referenced until the copies have run
        hin = [pin(x) for x in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)]
        hp(*hin, oh, S0=S0, S_final=S)
        outs.append((oh, S, hin))
    hp.compute.synchronize()
    torch.cuda.synchronize()
    for (oh, S, _), (o_ref, S_ref) in zip(outs, refs):
        assert torch.equal(oh, o_ref.cpu())
        assert torch.equal(S, S_ref)
