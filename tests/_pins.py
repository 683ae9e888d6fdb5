"""Pins for the float64 oracle: checks against what the pages and plain
mathematics fix, none of which re-types the oracle's own loop.

Source pages (cited by title and section):
  [K3R]  "[논문 리뷰] Kimi K3 Technical Report" (jw9603.github.io)
  [KMA]  "Kimi 모델 분석" (rlaope.github.io)

Each ``pin_*`` takes an oracle handle ``O`` (an object with ``prefill`` and
``decode_step`` like the ``oracle`` package) and raises AssertionError when the
oracle disagrees.  The same functions run against the real oracle
(test_oracle_pins.py) and against deliberately broken copies of it
(test_oracle_mutants.py), which must each fail at least one pin.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


def _unit(rng, d):
    x = rng.standard_normal(d)
    return x / np.linalg.norm(x)


def _rand_problem(rng, T, H, dk, dv, unit_k=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -rng.uniform(0.0, 2.0, (T, H, dk))
    b = rng.uniform(0.0, 1.0, (T, H))
    return q, k, v, g, b


# ---------------------------------------------------------------------------
# [K3R] section 3.4: the worked example and the two beta extremes.
# ---------------------------------------------------------------------------
def pin_worked_example(O):
    gold = read_golden("worked_example.txt")
    pred, val, beta = gold["prediction"][0], gold["value"][0], gold["beta"][0]
    for bkey, bval in (("readout", beta), ("readout_beta0", 0.0),
                       ("readout_beta1", 1.0)):
        # One key channel, one value channel: k = [1], Sbar = [[pred]] with
        # alpha = 1, and the readout query equals the key.
        q = np.ones((1, 1, 1))
        k = np.ones((1, 1, 1))
        v = np.full((1, 1, 1), val)
        g = np.zeros((1, 1, 1))
        b = np.full((1, 1), bval)
        S0 = np.full((1, 1, 1, 1), pred)
        o, _ = O.prefill(q, k, v, g, b, S0=S0)
        assert abs(o[0, 0, 0] - gold[bkey][0]) < 1e-15, (bkey, o[0, 0, 0])

    # The same example embedded in d = 6: a random unit key and a random state
    # whose decayed prediction at that key is 0.2 in every value column.
    rng = np.random.default_rng(1)
    dk, dv = 6, 4
    kk = _unit(rng, dk)
    alpha = rng.uniform(0.3, 1.0, dk)
    S0 = rng.standard_normal((dk, dv))
    Sbar = alpha[:, None] * S0
    S0 = S0 + np.outer(kk / alpha, pred - Sbar.T @ kk)   # now Sbar^T k = pred
    q = kk.reshape(1, 1, dk)
    o, _ = O.prefill(q, kk.reshape(1, 1, dk), np.full((1, 1, dv), val),
                     np.log(alpha).reshape(1, 1, dk), np.full((1, 1), beta),
                     S0=S0.reshape(1, 1, dk, dv))
    np.testing.assert_allclose(o[0, 0], gold["readout"][0], rtol=0, atol=1e-13)


def pin_beta_zero_alpha_one_is_identity(O):
    # [K3R] 3.4 (beta = 0 keeps the old value) with alpha = 1 (g = 0): the
    # state is unchanged and the readout is S0^T q.
    rng = np.random.default_rng(2)
    T, H, dk, dv = 5, 2, 4, 3
    q, k, v, _, _ = _rand_problem(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv))
    o, S = O.prefill(q, k, v, np.zeros((T, H, dk)), np.zeros((T, H)), S0=S0)
    np.testing.assert_array_equal(S, S0)
    for t in range(T):
        for h in range(H):
            np.testing.assert_allclose(o[t, h], S0[0, h].T @ q[t, h],
                                       rtol=0, atol=1e-14)


def pin_beta_one_unit_key_stores_value(O):
    # [K3R] 3.4 (beta = 1 replaces the value): with a unit key, S_t^T k_t = v_t
    # whatever the previous state and the decay.
    rng = np.random.default_rng(3)
    T, H, dk, dv = 6, 2, 5, 4
    _, k, v, g, _ = _rand_problem(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv))
    o, S = O.prefill(k, k, v, g, np.ones((T, H)), S0=S0)   # q = k reads S_t^T k_t
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-13)


def pin_diag_example(O):
    # [K3R] 3.2, "Diag는 무엇인가?": alpha = (0.9, 0.5, 0.2) keeps 90/50/20 %
    # of key channels (rows) 1..3.  beta = 0 isolates the decay.
    gold = read_golden("diag_example.txt")
    alpha = np.array(gold["alpha"])
    kept = np.array(gold["retained"])
    rng = np.random.default_rng(4)
    dk, dv = 3, 5
    S0 = rng.standard_normal((1, 1, dk, dv))
    o, S = O.prefill(np.zeros((1, 1, dk)), np.ones((1, 1, dk)) / np.sqrt(3),
                     rng.standard_normal((1, 1, dv)),
                     np.log(alpha).reshape(1, 1, dk), np.zeros((1, 1)), S0=S0)
    np.testing.assert_allclose(S[0, 0], kept[:, None] * S0[0, 0],
                               rtol=1e-15, atol=0)


# ---------------------------------------------------------------------------
# [K3R] 3.2 product form, evaluated with explicit dense matrices.
# ---------------------------------------------------------------------------
def _transition(alpha, k, beta):
    """(I - beta k k^T) Diag(alpha): the matrix that multiplies S_{t-1}."""
    dk = k.shape[0]
    return (np.eye(dk) - beta * np.outer(k, k)) @ np.diag(alpha)


def pin_product_form(O):
    rng = np.random.default_rng(5)
    T, H, dk, dv = 9, 3, 5, 7
    q, k, v, g, b = _rand_problem(rng, T, H, dk, dv, unit_k=False)
    b = rng.uniform(0.0, 2.0, (T, H))            # the form holds for any beta
    S0 = rng.standard_normal((1, H, dk, dv))
    o, S = O.prefill(q, k, v, g, b, S0=S0)
    for h in range(H):
        St = S0[0, h].copy()
        for t in range(T):
            St = (_transition(np.exp(g[t, h]), k[t, h], b[t, h]) @ St
                  + b[t, h] * np.outer(k[t, h], v[t, h]))
            np.testing.assert_allclose(o[t, h], St.T @ q[t, h], rtol=1e-12,
                                       atol=1e-12)
        np.testing.assert_allclose(S[0, h], St, rtol=1e-12, atol=1e-12)


def pin_gradient_step(O):
    # [KMA] "덮어쓰기가 되게 만들기": the delta rule is one gradient step with
    # step size beta on L(S) = 1/2 ||S^T k - v||^2, taken at the decayed state.
    # The gradient is taken numerically (central differences are exact for a
    # quadratic up to rounding), not from a formula.
    rng = np.random.default_rng(6)
    dk, dv = 4, 3
    k = rng.standard_normal(dk)
    v = rng.standard_normal(dv)
    alpha = rng.uniform(0.2, 1.0, dk)
    beta = 0.7
    S0 = rng.standard_normal((dk, dv))
    Sbar = alpha[:, None] * S0

    def loss(S):
        r = S.T @ k - v
        return 0.5 * float(r @ r)

    grad = np.zeros_like(Sbar)
    h = 1e-3
    for i in range(dk):
        for j in range(dv):
            E = np.zeros_like(Sbar)
            E[i, j] = h
            grad[i, j] = (loss(Sbar + E) - loss(Sbar - E)) / (2 * h)
    expect = Sbar - beta * grad
    _, S = O.prefill(np.zeros((1, 1, dk)), k.reshape(1, 1, dk),
                     v.reshape(1, 1, dv), np.log(alpha).reshape(1, 1, dk),
                     np.full((1, 1), beta), S0=S0.reshape(1, 1, dk, dv))
    np.testing.assert_allclose(S[0, 0], expect, rtol=0, atol=1e-9)


def pin_householder_reflection(O):
    # [KMA] "반사가 계층을 바꿈": with alpha = 1, beta = 2 and a unit key the
    # transition is the Householder reflection I - 2 k k^T; with v = 0 a step
    # preserves the Frobenius norm, and the same step twice is the identity.
    rng = np.random.default_rng(7)
    dk, dv = 6, 5
    k = _unit(rng, dk)
    S0 = rng.standard_normal((1, 1, dk, dv))
    kk = np.stack([k, k]).reshape(2, 1, dk)
    o, S = O.prefill(np.zeros((2, 1, dk)), kk, np.zeros((2, 1, dv)),
                     np.zeros((2, 1, dk)), np.full((2, 1), 2.0), S0=S0)
    np.testing.assert_allclose(S, S0, rtol=0, atol=1e-14)
    _, S1 = O.prefill(np.zeros((1, 1, dk)), kk[:1], np.zeros((1, 1, dv)),
                      np.zeros((1, 1, dk)), np.full((1, 1), 2.0), S0=S0)
    assert abs(np.linalg.norm(S1) - np.linalg.norm(S0)) < 1e-13
    np.testing.assert_allclose(S1[0, 0], S0[0, 0] - 2 * np.outer(k, k @ S0[0, 0]),
                               rtol=0, atol=1e-14)


def pin_repeated_key_closed_form(O):
    # Closed form: a fixed unit key, a scalar decay a on every channel and a
    # constant value v.  By [K3R] 3.4, x_t = S_t^T k obeys
    # x_t = (1 - beta) a x_{t-1} + beta v, so
    # x_T = r^T x_0 + beta v (1 - r^T) / (1 - r) with r = (1 - beta) a.
    rng = np.random.default_rng(8)
    T, dk, dv = 40, 5, 3
    k = _unit(rng, dk)
    a, beta = 0.93, 0.35
    v = rng.standard_normal(dv)
    S0 = rng.standard_normal((1, 1, dk, dv))
    x0 = S0[0, 0].T @ k
    kk = np.tile(k, (T, 1)).reshape(T, 1, dk)
    o, S = O.prefill(kk, kk, np.tile(v, (T, 1)).reshape(T, 1, dv),
                     np.full((T, 1, dk), np.log(a)), np.full((T, 1), beta), S0=S0)
    r = (1 - beta) * a
    for t in range(1, T + 1):
        xt = r ** t * x0 + beta * v * (1 - r ** t) / (1 - r)
        np.testing.assert_allclose(o[t - 1, 0], xt, rtol=0, atol=1e-13)


def pin_orthonormal_keys_exact_recall(O):
    # alpha = 1, beta = 1, S0 = 0, orthonormal keys: every write lands in its
    # own direction, so S_T = sum_i k_i v_i^T and querying with k_j recalls v_j.
    rng = np.random.default_rng(9)
    dk, dv = 8, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm.T                                   # rows are orthonormal
    T = dk
    v = rng.standard_normal((T, 1, dv))
    j = 3
    q = np.zeros((T, 1, dk))
    q[-1, 0] = keys[j]
    o, S = O.prefill(q, keys.reshape(T, 1, dk), v, np.zeros((T, 1, dk)),
                     np.ones((T, 1)))
    np.testing.assert_allclose(S[0, 0], keys.T @ v[:, 0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(o[-1, 0], v[j, 0], rtol=0, atol=1e-13)


def pin_brute_force_unrolled(O):
    # Brute force on tiny inputs, in extended precision: the closed unrolling
    # S_t = Phi(t,1) S_0 + sum_{i<=t} Phi(t,i+1) beta_i k_i v_i^T with
    # Phi(t,s) = A_t ... A_s and A_t = (I - beta_t k_t k_t^T) Diag(alpha_t),
    # o_t = S_t^T q_t.  No step-by-step state is carried.
    rng = np.random.default_rng(10)
    ld = np.longdouble
    for (T, dk, dv) in ((1, 1, 1), (3, 2, 3), (8, 4, 4), (7, 3, 2)):
        q, k, v, g, b = _rand_problem(rng, T, 1, dk, dv, unit_k=False)
        S0 = rng.standard_normal((1, 1, dk, dv))
        o, S = O.prefill(q, k, v, g, b, S0=S0)
        A = [(np.eye(dk, dtype=ld) - ld(b[t, 0]) * np.outer(k[t, 0].astype(ld),
                                                            k[t, 0].astype(ld)))
             @ np.diag(np.exp(g[t, 0].astype(ld))) for t in range(T)]

        def phi(t, s):
            M = np.eye(dk, dtype=ld)
            for r in range(s, t + 1):
                M = A[r] @ M
            return M

        for t in range(T):
            St = phi(t, 0) @ S0[0, 0].astype(ld)
            for i in range(t + 1):
                St = St + phi(t, i + 1) @ (ld(b[i, 0]) * np.outer(
                    k[i, 0].astype(ld), v[i, 0].astype(ld)))
            np.testing.assert_allclose(o[t, 0], (St.T @ q[t, 0].astype(ld)).astype(float),
                                       rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(S[0, 0], St.astype(float), rtol=1e-12, atol=1e-12)


def pin_varlen_equals_separate(O):
    # Packed sequences are independent: each one equals its own run, starting
    # from its own S0; an empty sequence returns its S0 unchanged.
    rng = np.random.default_rng(11)
    lens = [3, 0, 5, 1]
    H, dk, dv = 2, 3, 4
    T = sum(lens)
    q, k, v, g, b = _rand_problem(rng, T, H, dk, dv)
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, S = O.prefill(q, k, v, g, b, S0=S0, cu_seqlens=cu)
    for n, L in enumerate(lens):
        s, e = cu[n], cu[n + 1]
        if L == 0:
            np.testing.assert_array_equal(S[n], S0[n])
            continue
        # Each head of each sequence, checked against the product form.
        for h in range(H):
            St = S0[n, h].copy()
            for t in range(s, e):
                St = (_transition(np.exp(g[t, h]), k[t, h], b[t, h]) @ St
                      + b[t, h] * np.outer(k[t, h], v[t, h]))
                np.testing.assert_allclose(o[t, h], St.T @ q[t, h], rtol=1e-12,
                                           atol=1e-12)
            np.testing.assert_allclose(S[n, h], St, rtol=1e-12, atol=1e-12)


def pin_decode_step(O):
    # A decode step is one token of the same recurrence per (sequence, head);
    # checked against the product form of [K3R] 3.2.
    rng = np.random.default_rng(12)
    N, H, dk, dv = 3, 2, 4, 5
    q, k, v, g, b = _rand_problem(rng, N, H, dk, dv)
    S = rng.standard_normal((N, H, dk, dv))
    o, S1 = O.decode_step(q, k, v, g, b, S)
    for n in range(N):
        for h in range(H):
            St = (_transition(np.exp(g[n, h]), k[n, h], b[n, h]) @ S[n, h]
                  + b[n, h] * np.outer(k[n, h], v[n, h]))
            np.testing.assert_allclose(S1[n, h], St, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(o[n, h], St.T @ q[n, h], rtol=1e-13,
                                       atol=1e-13)


def pin_column_independence(O):
    # The update acts on each value column j with v_j alone, so a run on a
    # subset of value columns returns exactly those columns of o and S.  The
    # parity tests use this to check sampled columns of very long sequences.
    rng = np.random.default_rng(13)
    T, H, dk, dv = 12, 2, 4, 6
    q, k, v, g, b = _rand_problem(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv))
    o, S = O.prefill(q, k, v, g, b, S0=S0)
    cols = [1, 4]
    o2, S2 = O.prefill(q, k, v[:, :, cols], g, b, S0=S0[..., cols])
    np.testing.assert_array_equal(o2, o[:, :, cols])
    np.testing.assert_array_equal(S2, S[..., cols])


def pin_resume(O):
    # Running T1 tokens, then T2 more starting from the returned state, equals
    # one run of T1 + T2 tokens (the state is the whole memory).
    rng = np.random.default_rng(14)
    T1, T2, H, dk, dv = 4, 6, 2, 3, 3
    q, k, v, g, b = _rand_problem(rng, T1 + T2, H, dk, dv)
    o, S = O.prefill(q, k, v, g, b)
    oa, Sa = O.prefill(q[:T1], k[:T1], v[:T1], g[:T1], b[:T1])
    ob, Sb = O.prefill(q[T1:], k[T1:], v[T1:], g[T1:], b[T1:], S0=Sa)
    np.testing.assert_array_equal(np.concatenate([oa, ob]), o)
    np.testing.assert_array_equal(Sb, S)


def pin_lower_bound_stress(O):
    # [K3R] 3.5: g is bounded below by -5.  A long run at the bound stays
    # finite and matches the product form.
    rng = np.random.default_rng(15)
    T, dk, dv = 30, 4, 3
    q, k, v, _, b = _rand_problem(rng, T, 1, dk, dv)
    g = np.full((T, 1, dk), -5.0)
    o, S = O.prefill(q, k, v, g, b)
    St = np.zeros((dk, dv))
    for t in range(T):
        St = (_transition(np.exp(g[t, 0]), k[t, 0], b[t, 0]) @ St
              + b[t, 0] * np.outer(k[t, 0], v[t, 0]))
        np.testing.assert_allclose(o[t, 0], St.T @ q[t, 0], rtol=1e-12, atol=1e-14)
    assert np.all(np.isfinite(S))


PINS = [
    pin_worked_example,
    pin_beta_zero_alpha_one_is_identity,
    pin_beta_one_unit_key_stores_value,
    pin_diag_example,
    pin_product_form,
    pin_gradient_step,
    pin_householder_reflection,
    pin_repeated_key_closed_form,
    pin_orthonormal_keys_exact_recall,
    pin_brute_force_unrolled,
    pin_varlen_equals_separate,
    pin_decode_step,
    pin_column_independence,
    pin_resume,
    pin_lower_bound_stress,
]
