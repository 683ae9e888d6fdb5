"""Python binding of libkda.so, the KDA recurrence library for GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI of ``include/kda.h``.  PyTorch is used for device
memory and streams.  There is no CPU or PyTorch fallback: if the library is
not built, every call raises.

Functions (same names as the C ABI):
  kda_prefill(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, ...)
  kda_prefill_snapshots(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *, interval, ...)
  kda_decode_step(q, k, v, log_alpha, beta, S_inout, ...)
  kda_decode_multi(q, k, v, log_alpha, beta, S_in, ...)
  kda_prefill_fused(q, k, v, z, A, beta, ..., q_scale)
  kda_prefill_host(q, k, v, log_alpha, beta (host), ..., segment_tokens)
  kda_decode_step_fused(q, k, v, z, A, beta, S_inout, ..., q_scale)
  kda_state_gather(states, S_in, accept, ...)
  kda_prefill_workspace_bytes(num_seqs, H, d_k, d_v)
  kda_status_string(code)
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB_PATH, build  # noqa: F401  (re-exported)

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE, KDA_ERR_CUDA = range(5)
KDA_BF16, KDA_FP32, KDA_BF16_F32OUT = 0, 1, 2

# Every symbol include/kda.h declares.
EXPORTS = ("kda_prefill_workspace_bytes", "kda_prefill", "kda_decode_step",
           "kda_status_string", "kda_prefill_noalloc", "kda_prefill_snapshots",
           "kda_decode_multi", "kda_state_gather", "kda_prefill_fused",
           "kda_decode_step_fused", "kda_prefill_host_staging_bytes", "kda_prefill_host",
           "kda_prefill_segmented_workspace_bytes", "kda_prefill_segmented")


class KdaError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s: %s" % (where, kda_status_string(code)))


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


def _declare(lib):
    lib.kda_prefill_workspace_bytes.restype = _sz
    lib.kda_prefill_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32]
    lib.kda_prefill.restype = ctypes.c_int
    lib.kda_prefill.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                _i32, _i64, _i32, _i32, _i32, ctypes.c_int,
                                _vp, _vp, _vp, _sz, _vp]
    lib.kda_decode_step.restype = ctypes.c_int
    lib.kda_decode_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp,
                                    _i32, _i32, _i32, _i32, ctypes.c_int, _vp, _vp]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_prefill_host_staging_bytes.restype = _sz
    lib.kda_prefill_host_staging_bytes.argtypes = [_i32, _i32, _i32, ctypes.c_int, _i64]
    lib.kda_prefill_host.restype = ctypes.c_int
    lib.kda_prefill_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32,
                                     ctypes.c_int, _vp, _vp, _vp, _sz, _i64, _vp, _vp, _vp]
    lib.kda_prefill_fused.restype = ctypes.c_int
    lib.kda_prefill_fused.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                      _i32, _i64, _i32, _i32, _i32, ctypes.c_int, ctypes.c_float,
                                      _vp, _vp, _vp, _sz, _vp]
    lib.kda_decode_step_fused.restype = ctypes.c_int
    lib.kda_decode_step_fused.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                          _i32, ctypes.c_int, ctypes.c_float, _vp, _vp]
    lib.kda_decode_multi.restype = ctypes.c_int
    lib.kda_decode_multi.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                     ctypes.c_int, _vp, _vp, _vp]
    lib.kda_state_gather.restype = ctypes.c_int
    lib.kda_state_gather.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp]
    lib.kda_prefill_segmented_workspace_bytes.restype = _sz
    lib.kda_prefill_segmented_workspace_bytes.argtypes = [_i64, _i32, _i32, _i32, _i32]
    lib.kda_prefill_segmented.restype = ctypes.c_int
    lib.kda_prefill_segmented.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32,
                                          ctypes.c_int, _vp, _vp, _i32, _vp, _sz, _vp]
    lib.kda_prefill_snapshots.restype = ctypes.c_int
    lib.kda_prefill_snapshots.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                          _i32, _i64, _i32, _i32, _i32, ctypes.c_int,
                                          _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp]
    return lib


def _declare_noalloc(lib):
    lib.kda_prefill_noalloc.restype = ctypes.c_int
    lib.kda_prefill_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _i32, _i64, _i32, _i32, _i32, ctypes.c_int,
                                        _vp, _vp, _vp]
    return lib


def lib():
    """The loaded libkda.so (ctypes handle).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "libkda.so is not built (%s); run "
                    "`python -m gated_delta_rule_05_gb300._build`" % LIB_PATH)
            _lib = _declare_noalloc(_declare(ctypes.CDLL(LIB_PATH)))
        return _lib


def kda_status_string(code: int) -> str:
    return lib().kda_status_string(int(code)).decode()


def kda_prefill_workspace_bytes(num_seqs: int, H: int, d_k: int, d_v: int) -> int:
    return int(lib().kda_prefill_workspace_bytes(num_seqs, H, d_k, d_v))


def _torch():
    import torch
    return torch


def _dtype_code(t, out_dtype):
    """The C ABI's dtype code for inputs of t.dtype and an output of out_dtype."""
    torch = _torch()
    if t.dtype == torch.bfloat16 and out_dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.bfloat16 and out_dtype == torch.float32:
        return KDA_BF16_F32OUT
    if t.dtype == torch.float32 and out_dtype == torch.float32:
        return KDA_FP32
    raise TypeError("unsupported input/output dtypes %s -> %s" % (t.dtype, out_dtype))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_cuda(name, t, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))


def _stream_handle(stream, device):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def kda_prefill(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *,
                o=None, S_final=None, want_state=True, workspace=None,
                stream=None, o_dtype=None):
    """Chunked KDA prefill over packed sequences (C ABI: kda_prefill).

    q, k, log_alpha: [T, H, d_k]; v: [T, H, d_v]; beta: [T, H];
    S0: [N, H, d_k, d_v] fp32 or None; cu_seqlens: int32 [N+1] or None.
    Returns (o, S_final); S_final is None when ``want_state`` is False and no
    buffer was given.  ``S_final`` may be ``S0`` itself (in-place resume).
    ``o_dtype`` (default: o's dtype if given, else q's) may be float32 for
    bfloat16 inputs.
    """
    torch = _torch()
    T, H, dk = q.shape
    dv = v.shape[2]
    if o_dtype is None:
        o_dtype = o.dtype if o is not None else q.dtype
    dt = _dtype_code(q, o_dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("beta", beta, torch.float32)
    _check_cuda("S0", S0, torch.float32)
    _check_cuda("cu_seqlens", cu_seqlens, torch.int32)
    N = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    dev = q.device
    if o is None:
        o = torch.empty((T, H, dv), dtype=o_dtype, device=dev)
    _check_cuda("o", o, o_dtype)
    if S_final is None and want_state:
        S_final = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _check_cuda("S_final", S_final, torch.float32)
    need = kda_prefill_workspace_bytes(N, H, dk, dv)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check_cuda("workspace", workspace)
    with torch.cuda.device(dev):
        rc = lib().kda_prefill(
            _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
            _ptr(cu_seqlens), N, T, H, dk, dv, dt, _ptr(o), _ptr(S_final),
            _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream_handle(stream, dev))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill")
    return o, S_final


def kda_prefill_segmented_workspace_bytes(T: int, H: int, d_k: int, d_v: int,
                                          segments: int = 0) -> int:
    return int(lib().kda_prefill_segmented_workspace_bytes(T, H, d_k, d_v, segments))


def kda_prefill_segmented(q, k, v, log_alpha, beta, S0=None, *, segments=0, o=None,
                          S_final=None, want_state=True, workspace=None, stream=None,
                          o_dtype=None):
    """Chunk-group parallel prefill of ONE sequence (C ABI:
    kda_prefill_segmented): the sequence's chunks in ``segments`` groups that
    run at once (<= 0: chosen by the library), joined by a scan of the
    segment states and a fix-up of the outputs.  Same arguments and results as
    kda_prefill with N = 1.  Returns (o, S_final)."""
    torch = _torch()
    T, H, dk = q.shape
    dv = v.shape[2]
    if o_dtype is None:
        o_dtype = o.dtype if o is not None else q.dtype
    dt = _dtype_code(q, o_dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("beta", beta, torch.float32)
    _check_cuda("S0", S0, torch.float32)
    dev = q.device
    if o is None:
        o = torch.empty((T, H, dv), dtype=o_dtype, device=dev)
    _check_cuda("o", o, o_dtype)
    if S_final is None and want_state:
        S_final = torch.empty((1, H, dk, dv), dtype=torch.float32, device=dev)
    _check_cuda("S_final", S_final, torch.float32)
    with torch.cuda.device(dev):
        need = kda_prefill_segmented_workspace_bytes(T, H, dk, dv, segments)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check_cuda("workspace", workspace)
    with torch.cuda.device(dev):
        rc = lib().kda_prefill_segmented(
            _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0), T, H, dk, dv, dt,
            _ptr(o), _ptr(S_final), int(segments), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill_segmented")
    return o, S_final


def kda_decode_step(q, k, v, log_alpha, beta, S_inout, *, o=None, stream=None,
                    o_dtype=None):
    """One decode step, state updated in place (C ABI: kda_decode_step).

    q, k, log_alpha: [N, H, d_k]; v: [N, H, d_v]; beta: [N, H];
    S_inout: [N, H, d_k, d_v] fp32.  Returns o [N, H, d_v].
    """
    torch = _torch()
    N, H, dk = q.shape
    dv = v.shape[2]
    if o_dtype is None:
        o_dtype = o.dtype if o is not None else q.dtype
    dt = _dtype_code(q, o_dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("beta", beta, torch.float32)
    _check_cuda("S_inout", S_inout, torch.float32)
    if o is None:
        o = torch.empty((N, H, dv), dtype=o_dtype, device=q.device)
    _check_cuda("o", o, o_dtype)
    with torch.cuda.device(q.device):
        rc = lib().kda_decode_step(
            _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S_inout),
            N, H, dk, dv, dt, _ptr(o), _stream_handle(stream, q.device))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step")
    return o


def kda_prefill_noalloc(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *,
                        o, S_final=None, stream=None):
    """kda_prefill without a workspace (C ABI: kda_prefill_noalloc), for
    callers that cannot allocate device memory: the library uses a fixed
    scratch array of its own (at most 4096 sequences).  ``o`` (and
    ``S_final``, if wanted) must be given; this wrapper allocates nothing.
    Returns (o, S_final)."""
    torch = _torch()
    T, H, dk = q.shape
    dv = v.shape[2]
    dt = _dtype_code(q, o.dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("beta", beta, torch.float32)
    _check_cuda("S0", S0, torch.float32)
    _check_cuda("cu_seqlens", cu_seqlens, torch.int32)
    _check_cuda("o", o, o.dtype)
    _check_cuda("S_final", S_final, torch.float32)
    N = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    with torch.cuda.device(q.device):
        rc = lib().kda_prefill_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
            _ptr(cu_seqlens), N, T, H, dk, dv, dt, _ptr(o), _ptr(S_final),
            _stream_handle(stream, q.device))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill_noalloc")
    return o, S_final


def snapshot_offsets(cu_seqlens, interval):
    """snap_offsets for kda_prefill_snapshots from cu_seqlens (int32 [N+1],
    on the device): exclusive prefix sums of floor(len_n / interval).  Index
    bookkeeping for the caller's buffers; returns (offsets, total)."""
    torch = _torch()
    counts = torch.div(cu_seqlens[1:] - cu_seqlens[:-1], interval, rounding_mode="floor")
    off = torch.zeros(cu_seqlens.shape[0], dtype=torch.int32, device=cu_seqlens.device)
    off[1:] = torch.cumsum(counts, 0)
    return off, int(off[-1].item())


def kda_prefill_snapshots(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *, interval,
                          snap_offsets=None, snapshots=None, o=None, S_final=None,
                          want_state=True, workspace=None, stream=None, o_dtype=None):
    """kda_prefill that also returns the state of every sequence after every
    ``interval`` tokens (a positive multiple of 64), for a prefix cache
    (C ABI: kda_prefill_snapshots).  ``snapshots`` is [snap_offsets[N], H,
    d_k, d_v] fp32, snapshot j of sequence n at snap_offsets[n] + j.  When
    they are not given, offsets are derived from cu_seqlens and the buffer is
    allocated (which reads the total back to the host).
    Returns (o, S_final, snapshots, snap_offsets)."""
    torch = _torch()
    T, H, dk = q.shape
    dv = v.shape[2]
    if o_dtype is None:
        o_dtype = o.dtype if o is not None else q.dtype
    dt = _dtype_code(q, o_dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("beta", beta, torch.float32)
    _check_cuda("S0", S0, torch.float32)
    _check_cuda("cu_seqlens", cu_seqlens, torch.int32)
    N = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    dev = q.device
    if snap_offsets is None and cu_seqlens is not None:
        snap_offsets, total = snapshot_offsets(cu_seqlens, interval)
    elif cu_seqlens is None:
        total = T // interval if interval > 0 else 0
    else:
        total = int(snap_offsets[-1].item())
    _check_cuda("snap_offsets", snap_offsets, torch.int32)
    if snapshots is None:
        snapshots = torch.empty((max(total, 0), H, dk, dv), dtype=torch.float32, device=dev)
    _check_cuda("snapshots", snapshots, torch.float32)
    if o is None:
        o = torch.empty((T, H, dv), dtype=o_dtype, device=dev)
    _check_cuda("o", o, o_dtype)
    if S_final is None and want_state:
        S_final = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _check_cuda("S_final", S_final, torch.float32)
    need = kda_prefill_workspace_bytes(N, H, dk, dv)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check_cuda("workspace", workspace)
    # No snapshot is due (every sequence shorter than the interval): the C ABI
    # still wants a buffer, which is never written.
    snap_buf = snapshots if snapshots.numel() > 0 else \
        torch.empty(4, dtype=torch.float32, device=dev)
    snap_ptr = _ptr(snap_buf)
    with torch.cuda.device(dev):
        rc = lib().kda_prefill_snapshots(
            _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
            _ptr(cu_seqlens), N, T, H, dk, dv, dt, _ptr(o), _ptr(S_final),
            int(interval), _ptr(snap_offsets), snap_ptr,
            _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream_handle(stream, dev))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill_snapshots")
    return o, S_final, snapshots, snap_offsets


def kda_decode_multi(q, k, v, log_alpha, beta, S_in, *, o=None, states=None, stream=None,
                     o_dtype=None):
    """Ts decode tokens per sequence keeping every intermediate state
    (C ABI: kda_decode_multi).  q, k, log_alpha: [N, Ts, H, d_k]; v:
    [N, Ts, H, d_v]; beta: [N, Ts, H]; S_in: [N, H, d_k, d_v] (not modified).
    Returns (o [N, Ts, H, d_v], states [N, Ts, H, d_k, d_v])."""
    torch = _torch()
    N, Ts, H, dk = q.shape
    dv = v.shape[3]
    if o_dtype is None:
        o_dtype = o.dtype if o is not None else q.dtype
    dt = _dtype_code(q, o_dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("beta", beta, torch.float32)
    _check_cuda("S_in", S_in, torch.float32)
    if o is None:
        o = torch.empty((N, Ts, H, dv), dtype=o_dtype, device=q.device)
    if states is None:
        states = torch.empty((N, Ts, H, dk, dv), dtype=torch.float32, device=q.device)
    _check_cuda("o", o, o_dtype)
    _check_cuda("states", states, torch.float32)
    with torch.cuda.device(q.device):
        rc = lib().kda_decode_multi(
            _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S_in),
            N, Ts, H, dk, dv, dt, _ptr(o), _ptr(states), _stream_handle(stream, q.device))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_multi")
    return o, states


def kda_state_gather(states, S_in, accept, *, S_out=None, stream=None):
    """The state after each sequence's accepted prefix (C ABI:
    kda_state_gather): S_out[n] = states[n, accept[n] - 1], or S_in[n] when
    accept[n] is 0.  S_out may be S_in (in place).  Returns S_out."""
    torch = _torch()
    N, Ts, H, dk, dv = states.shape
    _check_cuda("states", states, torch.float32)
    _check_cuda("S_in", S_in, torch.float32)
    _check_cuda("accept", accept, torch.int32)
    if S_out is None:
        S_out = torch.empty_like(S_in)
    _check_cuda("S_out", S_out, torch.float32)
    with torch.cuda.device(states.device):
        rc = lib().kda_state_gather(_ptr(states), _ptr(S_in), _ptr(accept), N, Ts, H, dk, dv,
                                    _ptr(S_out), _stream_handle(stream, states.device))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_state_gather")
    return S_out


def kda_prefill_fused(q, k, v, z, A, beta, S0=None, cu_seqlens=None, *, q_scale, o=None,
                      S_final=None, want_state=True, workspace=None, stream=None, o_dtype=None):
    """kda_prefill with the gate prologue in the kernels (C ABI:
    kda_prefill_fused): raw q, k (L2-normalised inside, q times q_scale), the
    gate pre-activation z [T, H, d_k] and A [H, d_k] (g = -5 sigmoid(e^A z)).
    Returns (o, S_final)."""
    torch = _torch()
    T, H, dk = q.shape
    dv = v.shape[2]
    if o_dtype is None:
        o_dtype = o.dtype if o is not None else q.dtype
    dt = _dtype_code(q, o_dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("z", z, torch.float32)
    _check_cuda("A", A, torch.float32)
    _check_cuda("beta", beta, torch.float32)
    _check_cuda("S0", S0, torch.float32)
    _check_cuda("cu_seqlens", cu_seqlens, torch.int32)
    N = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    dev = q.device
    if o is None:
        o = torch.empty((T, H, dv), dtype=o_dtype, device=dev)
    _check_cuda("o", o, o_dtype)
    if S_final is None and want_state:
        S_final = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _check_cuda("S_final", S_final, torch.float32)
    need = kda_prefill_workspace_bytes(N, H, dk, dv)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check_cuda("workspace", workspace)
    with torch.cuda.device(dev):
        rc = lib().kda_prefill_fused(
            _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta), _ptr(S0),
            _ptr(cu_seqlens), N, T, H, dk, dv, dt, float(q_scale), _ptr(o), _ptr(S_final),
            _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream_handle(stream, dev))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill_fused")
    return o, S_final


def kda_decode_step_fused(q, k, v, z, A, beta, S_inout, *, q_scale, o=None, stream=None,
                          o_dtype=None):
    """kda_decode_step with the gate prologue in the kernel (C ABI:
    kda_decode_step_fused).  Returns o; S_inout is updated in place."""
    torch = _torch()
    N, H, dk = q.shape
    dv = v.shape[2]
    if o_dtype is None:
        o_dtype = o.dtype if o is not None else q.dtype
    dt = _dtype_code(q, o_dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("z", z, torch.float32)
    _check_cuda("A", A, torch.float32)
    _check_cuda("beta", beta, torch.float32)
    _check_cuda("S_inout", S_inout, torch.float32)
    if o is None:
        o = torch.empty((N, H, dv), dtype=o_dtype, device=q.device)
    _check_cuda("o", o, o_dtype)
    with torch.cuda.device(q.device):
        rc = lib().kda_decode_step_fused(
            _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta), _ptr(S_inout),
            N, H, dk, dv, dt, float(q_scale), _ptr(o), _stream_handle(stream, q.device))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step_fused")
    return o


class HostPrefill:
    """kda_prefill_host for repeated calls: holds the device staging area and
    the three streams the pipeline runs on (C ABI: kda_prefill_host).

        hp = HostPrefill(H, d, dtype=torch.bfloat16, segment_tokens=16384)
        hp(q_h, k_h, v_h, log_alpha_h, beta_h, o_h, S0=None, S_final=None)

    q_h, k_h, v_h, log_alpha_h, beta_h, o_h are CPU tensors (pinned for full
    speed) of one sequence; S0 / S_final are CUDA tensors [1, H, d, d] or
    None.  The call returns once the work is enqueued; hp.compute (a torch
    stream) completes when everything has, o_h included."""

    def __init__(self, H, d, dtype, segment_tokens=16384, o_dtype=None, device=None):
        torch = _torch()
        self.H, self.d, self.seg = H, d, int(segment_tokens)
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        probe = torch.empty(0, dtype=dtype)
        self.dt = _dtype_code(probe, o_dtype or dtype)
        nbytes = int(lib().kda_prefill_host_staging_bytes(H, d, d, self.dt, self.seg))
        if nbytes == 0:
            raise KdaError(KDA_ERR_INVALID_ARG, "kda_prefill_host_staging_bytes")
        self.staging = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self.compute = torch.cuda.Stream(self.device)
        self.h2d = torch.cuda.Stream(self.device)
        self.d2h = torch.cuda.Stream(self.device)

    def __call__(self, q, k, v, log_alpha, beta, o, S0=None, S_final=None):
        T = q.shape[0]
        hp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
        with _torch().cuda.device(self.device):
            rc = lib().kda_prefill_host(
                hp(q), hp(k), hp(v), hp(log_alpha), hp(beta), _ptr(S0), T, self.H, self.d,
                self.d, self.dt, hp(o), _ptr(S_final), _ptr(self.staging),
                self.staging.numel(), self.seg, ctypes.c_void_p(self.compute.cuda_stream),
                ctypes.c_void_p(self.h2d.cuda_stream), ctypes.c_void_p(self.d2h.cuda_stream))
        if rc != KDA_OK:
            raise KdaError(rc, "kda_prefill_host")
        return o, S_final
