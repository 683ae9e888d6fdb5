"""float64 CPU oracle for the Kimi Delta Attention (KDA) recurrence.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline / reference legs of ``bench.py`` may
import this package.  It shares no code with the CUDA library
(``gated_delta_rule_05_gb300``) and never imports it.

The arithmetic lives in ``kda_oracle.c`` (plain C, float64, libm ``exp``); this
module only compiles it with gcc and marshals numpy arrays through ctypes.

Source of the method: "[논문 리뷰] Kimi K3 Technical Report" (jw9603.github.io),
sections 3.2 (update and readout), 3.3 (delta form), 3.5 (alpha = exp(g)).

Every function here is pinned by ``tests/test_oracle_pins.py`` (see the list in
the C file's header); no function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")

_lock = threading.Lock()
_lib = None

_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def compile_library(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle into a shared library (IEEE float64, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (force or not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        compile_library()
    return _LIB_PATH


def _declare(lib):
    lib.kda_oracle_prefill.restype = ctypes.c_int
    lib.kda_oracle_prefill.argtypes = [
        _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _i64p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        _f64p, _f64p, ctypes.c_int]
    lib.kda_oracle_decode_step.restype = ctypes.c_int
    lib.kda_oracle_decode_step.argtypes = [
        _f64p, _f64p, _f64p, _f64p, _f64p, _f64p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        _f64p, ctypes.c_int]
    return lib


def load_library(path: str):
    """Load an oracle library from an explicit path (used by the mutant test)."""
    return _declare(ctypes.CDLL(path))


def _get():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


def _c64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_f64p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def prefill(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None,
            nthreads: int | None = None, lib=None):
    """Run the recurrence over packed sequences.

    q, k, log_alpha: [T_tot, H, dk]; v: [T_tot, H, dv]; beta: [T_tot, H];
    S0: [N, H, dk, dv] or None (zeros); cu_seqlens: [N+1] or None (one
    sequence of all T_tot tokens).  Inputs are widened to float64 exactly.
    Returns (o [T_tot, H, dv], S_final [N, H, dk, dv]) as float64 arrays.
    """
    lib = lib or _get()
    q, k, v, g, b = (_c64(x) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    N = cu.shape[0] - 1
    if int(cu[-1]) != T:
        raise ValueError("cu_seqlens[-1] must equal the number of tokens")
    s0 = None if S0 is None else _c64(S0)
    if s0 is not None and s0.shape != (N, H, dk, dv):
        raise ValueError("S0 must have shape [N, H, dk, dv]")
    o = np.empty((T, H, dv), dtype=np.float64)
    S_final = np.empty((N, H, dk, dv), dtype=np.float64)
    rc = lib.kda_oracle_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(s0),
        cu.ctypes.data_as(_i64p), N, H, dk, dv, _ptr(o), _ptr(S_final),
        nthreads or default_threads())
    if rc != 0:
        raise ValueError("kda_oracle_prefill rejected its arguments (rc=%d)" % rc)
    return o, S_final


def decode_step(q, k, v, log_alpha, beta, S, nthreads: int | None = None,
                lib=None):
    """One token per sequence.  q, k, log_alpha: [N, H, dk]; v: [N, H, dv];
    beta: [N, H]; S: [N, H, dk, dv].  Returns (o [N, H, dv], S_new)."""
    lib = lib or _get()
    q, k, v, g, b = (_c64(x) for x in (q, k, v, log_alpha, beta))
    N, H, dk = q.shape
    dv = v.shape[2]
    S_new = np.array(S, dtype=np.float64, copy=True, order="C")
    o = np.empty((N, H, dv), dtype=np.float64)
    rc = lib.kda_oracle_decode_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(S_new),
        N, H, dk, dv, _ptr(o), nthreads or default_threads())
    if rc != 0:
        raise ValueError("kda_oracle_decode_step rejected its arguments (rc=%d)" % rc)
    return o, S_new


def snapshot_counts(lengths, interval: int):
    """Snapshots per sequence for a given interval: floor(len / interval)."""
    return [int(n) // int(interval) for n in lengths]


def prefill_snapshots(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, interval: int = 64,
                      nthreads: int | None = None, lib=None):
    """The recurrence over packed sequences, also returning the state of every
    sequence after every `interval` tokens: the prefix states a serving stack
    caches and restores ("[논문 리뷰] Kimi K3 Technical Report", section 13, the
    KDA-aware prefix cache; "Kimi 모델 분석", section "요약본 저장 위치").
    Snapshot j of sequence n is the state after its first (j + 1) * interval
    tokens; they are stacked over sequences in order.

    Each sequence is run as consecutive segments of `interval` tokens, each
    starting from the state the previous one ended in (the recurrence only
    carries S from token to token, section 3.2).
    Returns (o, S_final, snapshots [n_snap, H, dk, dv], offsets [N+1]).
    """
    q, k, v, g, b = (_c64(x) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = np.array([0, T], dtype=np.int64) if cu_seqlens is None else \
        np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    N = cu.shape[0] - 1
    interval = int(interval)
    if interval < 1:
        raise ValueError("interval must be positive")
    s0 = None if S0 is None else _c64(S0)
    o = np.empty((T, H, dv), dtype=np.float64)
    S_final = np.empty((N, H, dk, dv), dtype=np.float64)
    counts = snapshot_counts(np.diff(cu), interval)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    snaps = np.empty((int(offsets[-1]), H, dk, dv), dtype=np.float64)
    for n in range(N):
        S = np.zeros((1, H, dk, dv)) if s0 is None else s0[n:n + 1].copy()
        bos, eos = int(cu[n]), int(cu[n + 1])
        j = 0
        for s in range(bos, eos, interval):
            e = min(eos, s + interval)
            o[s:e], S = prefill(q[s:e], k[s:e], v[s:e], g[s:e], b[s:e], S0=S,
                                nthreads=nthreads, lib=lib)
            if e - s == interval:
                snaps[offsets[n] + j] = S[0]
                j += 1
        S_final[n] = S[0]
    return o, S_final, snaps, offsets


def decode_multi(q, k, v, log_alpha, beta, S, nthreads: int | None = None, lib=None):
    """Several tokens per sequence, keeping the state after every token: the
    verification step of speculative decoding must be able to return to the
    state after any accepted prefix, since the state is overwritten in place
    and cannot be truncated ("[논문 리뷰] Kimi K3 Technical Report", section
    13, speculative decoding replay; "Kimi 모델 분석", section "Dspark 투기적
    디코딩").  q, k, log_alpha: [N, Ts, H, dk]; v: [N, Ts, H, dv];
    beta: [N, Ts, H]; S: [N, H, dk, dv].  Token t of every sequence is one
    decode step from the state after token t - 1.
    Returns (o [N, Ts, H, dv], states [N, Ts, H, dk, dv])."""
    q, k, v, g, b = (_c64(x) for x in (q, k, v, log_alpha, beta))
    N, Ts, H, dk = q.shape
    dv = v.shape[3]
    o = np.empty((N, Ts, H, dv), dtype=np.float64)
    states = np.empty((N, Ts, H, dk, dv), dtype=np.float64)
    cur = _c64(S)
    for t in range(Ts):
        o[:, t], cur = decode_step(q[:, t], k[:, t], v[:, t], g[:, t], b[:, t], cur,
                                   nthreads=nthreads, lib=lib)
        states[:, t] = cur
    return o, states


G_MIN = -5.0


def gate_prologue(q, k, z, A, q_scale: float):
    """The steps in front of the recurrence, in float64: the lower-bounded
    log-decay g = g_min * sigmoid(e^A z) with g_min = -5 ("[논문 리뷰] Kimi K3
    Technical Report", section 3.5, so that g lies in (-5, 0) and
    alpha = exp(g) in (e^-5, 1)), and the L2 normalisation of q and k over
    the key channels, q also multiplied by q_scale.

    q, k, z: [..., H, d_k]; A: [H, d_k] (one value per head and key channel;
    a per-head A is the same value repeated over the channels).
    Returns (q_hat, k_hat, g)."""
    q, k, z, A = (_c64(x) for x in (q, k, z, A))
    s = np.exp(A) * z
    g = G_MIN * 0.5 * (1.0 + np.tanh(0.5 * s))     # sigmoid(s), without overflow
    qn = np.sqrt(np.sum(q * q, axis=-1, keepdims=True))
    kn = np.sqrt(np.sum(k * k, axis=-1, keepdims=True))
    return q * (float(q_scale) / qn), k / kn, g
