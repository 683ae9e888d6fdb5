"""Parity helpers: run the float64 oracle on exactly the values the GPU saw and
compare with the error measure the tests use.

Error measure: max |x_gpu - x_ref| over the compared elements, divided by the
RMS of x_ref over the same elements.  Tolerances: 2e-2 for bf16 inputs with an
fp32 state, 1e-4 for fp32 inputs.

A result stored in bfloat16 carries its own rounding, up to half an ulp
(2^-8 |x| relative) per element; even the exactly rounded oracle value exceeds
2e-2 x RMS by that alone once max|o| is about 8 x RMS.  For bf16 outputs the
bound is therefore applied to what the kernel adds beyond that rounding:
max(|x_gpu - x_ref| - 2^-8 |x_ref|) <= tol x RMS(x_ref).  fp32 results (S_final,
and o with an fp32 output) are held to the plain bound.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {"bf16": 2e-2, "fp32": 1e-4, torch.bfloat16: 2e-2, torch.float32: 1e-4}


def to64(t):
    """Exact widening of a (CPU or CUDA) tensor to a float64 numpy array."""
    return t.detach().to("cpu").double().numpy()


BF16_HALF_ULP = 2.0 ** -8


def rel_err(x, ref, bf16_out=False):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    assert np.all(np.isfinite(x)), "non-finite values in the GPU result"
    rms = float(np.sqrt(np.mean(ref * ref)))
    d = np.abs(x - ref)
    if bf16_out:
        d = d - BF16_HALF_ULP * np.abs(ref)
    err = float(np.max(d))
    return err / rms if rms > 0 else err


def assert_close(x, ref, tol, what="", bf16_out=False):
    e = rel_err(x, ref, bf16_out)
    assert e <= tol, "%s: max|err|/rms = %.3e > %.1e" % (what, e, tol)
    return e


def compare_out(o_gpu, ref, tol, what="o"):
    """Compare an output tensor (bf16 or fp32) with the rule for its dtype."""
    return assert_close(to64(o_gpu), ref, tol, what,
                        bf16_out=(o_gpu.dtype == torch.bfloat16))


def oracle_prefill(inp, heads=None, cols=None, seg_tokens=None, nthreads=None):
    """float64 oracle on the batch ``inp`` (a synth.Inputs), restricted to
    ``heads`` and value columns ``cols`` (value columns evolve independently,
    so the restriction is exact).  A single long sequence may be processed in
    time segments of ``seg_tokens`` tokens, chaining the state between them.
    Returns (o_ref [T, len(heads), len(cols)], S_ref [N, len(heads), d_k, len(cols)]).
    """
    H = inp.q.shape[1]
    dv = inp.v.shape[2]
    heads = list(range(H)) if heads is None else list(heads)
    cols = list(range(dv)) if cols is None else list(cols)
    hi = torch.tensor(heads, dtype=torch.long)
    ci = torch.tensor(cols, dtype=torch.long)

    def take(t, s, e, last_cols=False):
        x = t[s:e].index_select(1, hi.to(t.device))
        if last_cols:
            x = x.index_select(2, ci.to(t.device))
        return to64(x)

    cu = inp.cu_seqlens.to("cpu").long().numpy()
    T = inp.total_tokens
    S0 = None
    if inp.S0 is not None:
        S0 = to64(inp.S0.index_select(1, hi.to(inp.S0.device))
                  .index_select(3, ci.to(inp.S0.device)))
    if seg_tokens is None or len(cu) != 2:
        o, S = oracle.prefill(take(inp.q, 0, T), take(inp.k, 0, T),
                              take(inp.v, 0, T, True), take(inp.log_alpha, 0, T),
                              to64(inp.beta[:, hi.to(inp.beta.device)]),
                              S0=S0, cu_seqlens=cu, nthreads=nthreads)
        return o, S
    outs = []
    S = S0
    for s in range(0, T, seg_tokens):
        e = min(T, s + seg_tokens)
        o, S = oracle.prefill(take(inp.q, s, e), take(inp.k, s, e),
                              take(inp.v, s, e, True), take(inp.log_alpha, s, e),
                              to64(inp.beta[s:e][:, hi.to(inp.beta.device)]),
                              S0=S, nthreads=nthreads)
        outs.append(o)
    return np.concatenate(outs, axis=0), S


def assert_kernels_agree(a, b, what=""):
    """Two prefill kernels on the same call: they evaluate the same products on
    the same 16-bit operands.  Any rounding difference between them (a UT
    solve product accurate to about 2^-22 that moves an fp16 rounding of T)
    moves o and S by about 2^-11 of a term, and with no decay (alpha = 1) such
    moves add up over the whole sequence.  So the check allows two bf16 ulps
    of each element (for bf16 outputs) plus 1e-2 of the RMS, half of either's
    bound against the oracle; a structural fault (a chunk, head or token out
    of place) moves o by its own size."""
    x, y = a.double(), b.double()
    rms = y.pow(2).mean().sqrt().item() if y.numel() else 0.0
    bound = torch.full_like(y, 1e-2 * rms)
    if a.dtype == torch.bfloat16:
        mag = y.abs().clamp_min(1e-30)
        bound = bound + 2 * torch.exp2(torch.floor(torch.log2(mag)) - 7)
    bad = (x - y).abs() > bound
    assert not bool(bad.any()), "%s: kernels differ by %.3g (RMS %.3g) at %d elements" % (
        what, (x - y).abs().max().item(), rms, int(bad.sum()))
