"""kda_prefill_host's host side (no GPU): the staging size and the argument
checks, which return before anything is enqueued."""
import pytest

import gated_delta_rule_05_gb300 as kda


@pytest.fixture(scope="module")
def lib():
    kda.build()
    return kda.lib()


def align256(x):
    return (x + 255) // 256 * 256


def staging_formula(lib, H, d, dtype, seg):
    """Two input slots (q | k | v | log_alpha | beta, each 256-aligned), two
    output slots, two states and the prefill workspace."""
    isz = 4 if dtype == kda.KDA_FP32 else 2
    osz = 2 if dtype == kda.KDA_BF16 else 4
    sizes = [seg * H * d * isz] * 3 + [seg * H * d * 4, seg * H * 4]
    in_slot = 5 * 256 + sum(sizes)
    out_slot = align256(seg * H * d * osz)
    state = align256(H * d * d * 4)
    ws = align256(lib.kda_prefill_workspace_bytes(1, H, d, d))
    return 2 * align256(in_slot) + 2 * out_slot + 2 * state + ws


@pytest.mark.parametrize("H,d,dtype,seg", [(2, 128, kda.KDA_BF16, 128), (3, 64, kda.KDA_FP32, 64),
                                           (32, 128, kda.KDA_BF16_F32OUT, 16384)])
def test_staging_bytes(lib, H, d, dtype, seg):
    assert lib.kda_prefill_host_staging_bytes(H, d, d, dtype, seg) == staging_formula(lib, H, d, dtype, seg)


@pytest.mark.parametrize("args", [(2, 128, 128, kda.KDA_BF16, 100),    # not a multiple of 64
                                  (2, 128, 128, kda.KDA_BF16, 0),
                                  (2, 128, 64, kda.KDA_BF16, 128),     # d_k != d_v
                                  (0, 128, 128, kda.KDA_BF16, 128)])
def test_staging_bytes_rejects(lib, args):
    assert lib.kda_prefill_host_staging_bytes(*args) == 0


A = 0x10000          # fake addresses: never dereferenced, every call fails validation first


def host(lib, **kw):
    args = dict(q=A, k=A, v=A, g=A, b=A, S0=None, T=1000, H=2, dk=128, dv=128, dt=kda.KDA_BF16,
                o=A, Sf=None, staging=A * 16, staging_bytes=1 << 40, seg=256,
                compute=None, h2d=None, d2h=None)
    args.update(kw)
    return lib.kda_prefill_host(*args.values())


@pytest.mark.parametrize("kw,code", [
    (dict(dt=7), kda.KDA_ERR_UNSUPPORTED),
    (dict(dk=96, dv=96), kda.KDA_ERR_UNSUPPORTED),
    (dict(dk=128, dv=64), kda.KDA_ERR_UNSUPPORTED),
    (dict(H=0), kda.KDA_ERR_INVALID_ARG),
    (dict(T=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(T=1 << 31), kda.KDA_ERR_INVALID_ARG),
    (dict(seg=100), kda.KDA_ERR_INVALID_ARG),
    (dict(seg=0), kda.KDA_ERR_INVALID_ARG),
    (dict(q=None), kda.KDA_ERR_INVALID_ARG),
    (dict(o=None), kda.KDA_ERR_INVALID_ARG),
    (dict(staging=None), kda.KDA_ERR_WORKSPACE),
    (dict(staging=A * 16 + 16), kda.KDA_ERR_WORKSPACE),    # not 256-byte aligned
    (dict(staging_bytes=4096), kda.KDA_ERR_WORKSPACE),
])
def test_host_prefill_rejects(lib, kw, code):
    assert host(lib, **kw) == code
