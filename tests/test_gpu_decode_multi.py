"""GPU parity of kda_decode_multi (several decode tokens per sequence, every
intermediate state kept, as the verification step of speculative decoding
needs) and kda_state_gather (the state after each sequence's accepted
prefix), against the oracle's decode_multi; and consistency with the
one-token decode and with prefill."""
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


def multi_inputs(N, Ts, H, d, dtype, seed):
    """N sequences of Ts tokens each, laid out [N, Ts, H, .] (synth draws the
    packed [N * Ts, H, .] batch; sequences are contiguous in it)."""
    inp = synth.generate([Ts] * N, H, d, d, dtype=dtype, s0_std=0.1, seed=seed)
    shp = lambda x: x.reshape(N, Ts, *x.shape[1:])
    return inp, shp(inp.q), shp(inp.k), shp(inp.v), shp(inp.log_alpha), shp(inp.beta), inp.S0


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_decode_multi_matches_oracle(kda, d, dtype):
    N, Ts, H = 37, 5, 3
    _, q, k, v, g, b, S0 = multi_inputs(N, Ts, H, d, dtype, 800 + d)
    o, st = kda.kda_decode_multi(*(x.cuda() for x in (q, k, v, g, b, S0)))
    torch.cuda.synchronize()
    o_ref, st_ref = oracle.decode_multi(to64(q), to64(k), to64(v), to64(g), to64(b), to64(S0))
    compare_out(o, o_ref, TOL[dtype], "o")
    assert_close(to64(st), st_ref, TOL[dtype], "states")


def test_decode_multi_equals_repeated_decode_steps(kda):
    N, Ts, H, d = 16, 4, 2, 128
    _, q, k, v, g, b, S0 = multi_inputs(N, Ts, H, d, "bf16", 810)
    q, k, v, g, b, S0 = (x.cuda() for x in (q, k, v, g, b, S0))
    o, st = kda.kda_decode_multi(q, k, v, g, b, S0)
    S = S0.clone()
    for t in range(Ts):
        ot = kda.kda_decode_step(q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous(),
                                 g[:, t].contiguous(), b[:, t].contiguous(), S)
        torch.cuda.synchronize()
        assert torch.equal(ot, o[:, t]), "token %d output" % t
        assert torch.equal(S, st[:, t]), "token %d state" % t


def test_state_gather(kda):
    N, Ts, H, d = 6, 5, 2, 64
    _, q, k, v, g, b, S0 = multi_inputs(N, Ts, H, d, "fp32", 820)
    q, k, v, g, b, S0 = (x.cuda() for x in (q, k, v, g, b, S0))
    o, st = kda.kda_decode_multi(q, k, v, g, b, S0)
    accept = torch.tensor([0, 1, Ts, 3, 9, -2], dtype=torch.int32, device="cuda")   # last two clamp
    out = kda.kda_state_gather(st, S0, accept)
    torch.cuda.synchronize()
    for n, a in enumerate([0, 1, Ts, 3, Ts, 0]):
        assert torch.equal(out[n], S0[n] if a == 0 else st[n, a - 1]), n
    # in place: the cache itself advances to the accepted states
    S = S0.clone()
    kda.kda_state_gather(st, S, accept, S_out=S)
    torch.cuda.synchronize()
    assert torch.equal(S, out)


def test_decode_multi_arguments_are_checked(kda):
    N, Ts, H, d = 2, 3, 1, 32
    _, q, k, v, g, b, S0 = multi_inputs(N, Ts, H, d, "fp32", 830)
    q, k, v, g, b, S0 = (x.cuda() for x in (q, k, v, g, b, S0))
    st = torch.empty((N, Ts, H, d, d), device="cuda")
    with pytest.raises(kda.KdaError) as e:       # states overlapping S_in
        kda.kda_decode_multi(q, k, v, g, b, st.view(-1)[: N * H * d * d].view(N, H, d, d),
                             states=st)
    assert e.value.code == kda.KDA_ERR_INVALID_ARG
    with pytest.raises(kda.KdaError) as e:       # o overlapping states
        kda.kda_decode_multi(q, k, v, g, b, S0, states=st,
                             o=st.view(-1)[: N * Ts * H * d].view(N, Ts, H, d))
    assert e.value.code == kda.KDA_ERR_INVALID_ARG


def test_prefill_then_multi_token_equals_prefill(kda):
    # a prompt by prefill, then Ts draft tokens by decode_multi == prefill of prompt + draft
    N, P, Ts, H, d = 3, 200, 6, 2, 128
    inp = synth.generate([P + Ts] * N, H, d, d, dtype="bf16", s0_std=0.05, seed=840)
    g = inp.to("cuda")
    T = N * (P + Ts)
    idx = torch.arange(T, device="cuda").view(N, P + Ts)
    pre = idx[:, :P].reshape(-1)
    dra = idx[:, P:]
    cu = torch.arange(0, N * P + 1, P, dtype=torch.int32, device="cuda")
    take = lambda x, i: x[i].contiguous()
    o_p, S_p = kda.kda_prefill(take(g.q, pre), take(g.k, pre), take(g.v, pre),
                               take(g.log_alpha, pre), take(g.beta, pre), S0=g.S0, cu_seqlens=cu)
    o_d, st = kda.kda_decode_multi(take(g.q, dra), take(g.k, dra), take(g.v, dra),
                                   take(g.log_alpha, dra), take(g.beta, dra), S_p)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.prefill(to64(inp.q), to64(inp.k), to64(inp.v), to64(inp.log_alpha),
                                  to64(inp.beta), S0=to64(inp.S0),
                                  cu_seqlens=inp.cu_seqlens.cpu().numpy())
    o_ref = o_ref.reshape(N, P + Ts, H, d)
    compare_out(o_d, o_ref[:, P:], TOL["bf16"], "draft outputs")
    assert_close(to64(st[:, -1]), S_ref, TOL["bf16"], "state after the draft")
