"""Pins of the oracle's prefix snapshots (prefill_snapshots) and multi-token
decode (decode_multi) against closed forms of the recurrence
("[논문 리뷰] Kimi K3 Technical Report", section 3.2):

  * no writes (beta = 0): the state after t tokens is Diag(alpha^t) S0, with
    alpha = exp(g) constant per channel;
  * alpha = 1, beta = 1 and orthonormal keys: writing v at key e_i sets row i
    of S to v, so the state after t tokens holds, in row i, the value last
    written at e_i (exact recall);
  * the last snapshot of a sequence whose length is a multiple of the
    interval is its final state, and the snapshot count is floor(len / interval).
"""
import numpy as np

import oracle


def _decay_only(lengths, H, d, g_val, seed):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, H, d))
    v = rng.standard_normal((T, H, d))
    g = np.broadcast_to(g_val, (T, H, d)).copy()
    beta = np.zeros((T, H))
    S0 = rng.standard_normal((len(lengths), H, d, d))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    return q, k, v, g, beta, S0, cu


def test_snapshots_of_pure_decay_are_powers_of_alpha():
    lengths, H, d, interval = [0, 7, 20, 12], 2, 4, 4
    g_val = np.array([-0.1, -0.5, -0.02, -1.3])
    q, k, v, g, beta, S0, cu = _decay_only(lengths, H, d, g_val, 1)
    o, S_final, snaps, off = oracle.prefill_snapshots(q, k, v, g, beta, S0=S0, cu_seqlens=cu,
                                                      interval=interval)
    assert list(np.diff(off)) == [n // interval for n in lengths]
    for n, L in enumerate(lengths):
        for j in range(L // interval):
            t = (j + 1) * interval
            expect = np.exp(g_val * t)[None, :, None] * S0[n]
            np.testing.assert_allclose(snaps[off[n] + j], expect, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(S_final[n], np.exp(g_val * L)[None, :, None] * S0[n],
                                   rtol=1e-13, atol=1e-15)


def test_snapshots_with_orthonormal_keys_recall_the_last_write():
    H, d, T, interval = 1, 4, 13, 3
    rng = np.random.default_rng(2)
    keys = rng.integers(0, d, size=T)
    k = np.zeros((T, H, d))
    k[np.arange(T), 0, keys] = 1.0
    v = rng.standard_normal((T, H, d))
    q = rng.standard_normal((T, H, d))
    g = np.zeros((T, H, d))
    beta = np.ones((T, H))
    o, S_final, snaps, off = oracle.prefill_snapshots(q, k, v, g, beta, interval=interval)
    assert snaps.shape[0] == T // interval
    for j in range(T // interval):
        t = (j + 1) * interval
        expect = np.zeros((d, d))
        for s in range(t):
            expect[keys[s]] = v[s, 0]
        np.testing.assert_allclose(snaps[j, 0], expect, rtol=0, atol=1e-14)


def test_last_snapshot_is_the_final_state_when_the_length_divides():
    rng = np.random.default_rng(3)
    lengths, H, d, interval = [8, 16, 5], 2, 3, 4
    T = sum(lengths)
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    g = -np.abs(rng.standard_normal((T, H, d)))
    beta = rng.uniform(0, 1, (T, H))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    o, S_final, snaps, off = oracle.prefill_snapshots(q, k, v, g, beta, cu_seqlens=cu,
                                                      interval=interval)
    o2, S2 = oracle.prefill(q, k, v, g, beta, cu_seqlens=cu)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S_final, S2, rtol=1e-12, atol=1e-12)
    for n, L in enumerate(lengths):
        if L % interval == 0:
            np.testing.assert_array_equal(snaps[off[n + 1] - 1], S_final[n])


def test_decode_multi_of_pure_decay_and_exact_recall():
    # pure decay: the state after token t is Diag(alpha^(t+1)) S
    rng = np.random.default_rng(4)
    N, Ts, H, d = 3, 5, 2, 4
    g_val = np.array([-0.2, -0.7, -0.05, -1.1])
    q, k, v = (rng.standard_normal((N, Ts, H, d)) for _ in range(3))
    g = np.broadcast_to(g_val, (N, Ts, H, d)).copy()
    beta = np.zeros((N, Ts, H))
    S = rng.standard_normal((N, H, d, d))
    o, states = oracle.decode_multi(q, k, v, g, beta, S)
    for t in range(Ts):
        np.testing.assert_allclose(states[:, t], np.exp(g_val * (t + 1))[None, None, :, None] * S,
                                   rtol=1e-13, atol=1e-15)
    # exact recall: o_t = S_t^T q with q = e_i returns the value last written at e_i
    keys = rng.integers(0, d, size=(N, Ts))
    k = np.zeros((N, Ts, H, d))
    for n in range(N):
        for t in range(Ts):
            k[n, t, :, keys[n, t]] = 1.0
    q = k.copy()
    g = np.zeros((N, Ts, H, d))
    beta = np.ones((N, Ts, H))
    S = np.zeros((N, H, d, d))
    o, states = oracle.decode_multi(q, k, v, g, beta, S)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-14)
