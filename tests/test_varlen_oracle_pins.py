"""Pins of the packed variable-length oracle (several sequences in one row, each with its
own state) against closed forms, the padded-batch oracle and finite differences.

A packed sequence must start from its own h0[i] and its own gate product: a state or a
cumulative gate carried across a boundary, a sequence run from the wrong h0, or an
off-by-one at a boundary fails the closed forms below.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(4321)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


CU = [0, 5, 5, 17, 18, 30]  # lengths 5, 0, 12, 1, 12


def _bounds(cu):
    return list(zip(cu[:-1], cu[1:]))


def test_seq_bounds_validation():
    assert oracle.seq_bounds([0, 3, 3, 7], 7) == [(0, 3), (3, 3), (3, 7)]
    assert oracle.seq_bounds([0], 0) == []
    for bad, T in (([1, 7], 7), ([0, 5], 7), ([0, 4, 3, 7], 7), ([], 0)):
        with pytest.raises(ValueError):
            oracle.seq_bounds(bad, T)


def test_varlen_beta_zero_decays_each_h0_from_its_own_start():
    """beta = 0: inside sequence i, S_t = exp(sum_{s = start_i}^{t} g_s) h0[i] and
    o_t = S_t^T q_t; h_T[i] is the decayed h0[i] (h0[i] itself for an empty sequence)."""
    T, Hqk, H, dk, dv = CU[-1], 2, 4, 5, 3
    N = len(CU) - 1
    qh, kh = rand(1, T, Hqk, dk), rand(1, T, Hqk, dk)
    v = rand(1, T, H, dv)
    g = -np.abs(rand(1, T, H)) * 0.3
    beta = np.zeros((1, T, H))
    h0 = rand(N, H, dk, dv)
    o, hT = oracle.core_fwd_varlen(qh, kh, v, g, beta, CU, h0)
    r = H // Hqk
    for i, (s, e) in enumerate(_bounds(CU)):
        decay = np.exp(np.cumsum(g[0, s:e], axis=0))      # [L, H]
        for h in range(H):
            for t in range(s, e):
                exp_o = decay[t - s, h] * (h0[i, h].T @ qh[0, t, h // r])
                np.testing.assert_allclose(o[0, t, h], exp_o, rtol=1e-12, atol=1e-13)
            last = decay[-1, h] if e > s else 1.0
            np.testing.assert_allclose(hT[i, h], last * h0[i, h], rtol=1e-12, atol=0)


def test_varlen_orthonormal_keys_restart_from_each_h0():
    """alpha = 1, beta = 1, keys orthonormal along the whole row: inside sequence i,
    S_t = (I - sum_{s in [start_i, t]} k_s k_s^T) h0[i] + sum_{s in [start_i, t]} k_s v_s^T,
    so only the sequence's own keys and values and its own h0 appear."""
    T, H, dk, dv = CU[-1], 2, 32, 4
    N = len(CU) - 1
    Q, _ = np.linalg.qr(rand(dk, dk))
    kh = Q[:T].reshape(1, T, 1, dk)
    qh = rand(1, T, 1, dk)
    v = rand(1, T, H, dv)
    g = np.zeros((1, T, H))
    beta = np.ones((1, T, H))
    h0 = rand(N, H, dk, dv)
    o, hT = oracle.core_fwd_varlen(qh, kh, v, g, beta, CU, h0)
    for i, (s, e) in enumerate(_bounds(CU)):
        for h in range(H):
            S = h0[i, h].copy()
            for t in range(s, e):
                K = kh[0, s:t + 1, 0]                       # keys of the sequence so far
                S = (np.eye(dk) - K.T @ K) @ h0[i, h] + K.T @ v[0, s:t + 1, h]
                np.testing.assert_allclose(o[0, t, h], S.T @ qh[0, t, 0], rtol=1e-10,
                                           atol=1e-11)
            np.testing.assert_allclose(hT[i, h], S, rtol=1e-10, atol=1e-11)


def _gates(T, H):
    a = rand(1, T, H)
    b = rand(1, T, H)
    A_log = np.log(RNG.uniform(1, 16, H))
    dt_bias = rand(H)
    return a, b, A_log, dt_bias


def _padded(x, cu, Lmax):
    """[N, Lmax, ...] rows of the packed sequences, zero past each length."""
    out = np.zeros((len(cu) - 1, Lmax) + x.shape[2:])
    for i, (s, e) in enumerate(_bounds(cu)):
        out[i, :e - s] = x[0, s:e]
    return out


def test_varlen_equals_the_padded_batch():
    """Packed rows give what the trailing-padding batch (one sequence per row, valid_len =
    its length) gives on the valid tokens, forward and backward."""
    T, Hqk, H, dk, dv = CU[-1], 1, 2, 6, 5
    N = len(CU) - 1
    q, k, v = rand(1, T, Hqk, dk), rand(1, T, Hqk, dk), rand(1, T, H, dv)
    a, b, A_log, dt_bias = _gates(T, H)
    h0, dHT = rand(N, H, dk, dv), rand(N, H, dk, dv)
    dO = rand(1, T, H, dv)
    lens = [e - s for s, e in _bounds(CU)]
    Lmax = max(lens)
    P = lambda x: _padded(x, CU, Lmax)  # noqa: E731
    o, hT = oracle.fwd_varlen(q, k, v, a, b, A_log, dt_bias, CU, h0)
    po, phT = oracle.fwd(P(q), P(k), P(v), P(a), P(b), A_log, dt_bias, h0=h0, valid_len=lens)
    np.testing.assert_allclose(P(o), po, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hT, phT, rtol=1e-12, atol=1e-13)
    g = oracle.bwd_varlen(q, k, v, a, b, A_log, dt_bias, CU, dO, dHT, h0)
    pg = oracle.bwd(P(q), P(k), P(v), P(a), P(b), A_log, dt_bias, P(dO), dHT, h0=h0,
                    valid_len=lens)
    for x, px in zip(g[:5], pg[:5]):
        np.testing.assert_allclose(P(x), px, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g[5], pg[5], rtol=1e-12, atol=1e-13)


def _fd(fun, x, eps=1e-6):
    grad = np.zeros_like(x)
    flat, gflat = x.reshape(-1), grad.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        flat[i] = old + eps
        fp = fun()
        flat[i] = old - eps
        fm = fun()
        flat[i] = old
        gflat[i] = (fp - fm) / (2 * eps)
    return grad


def test_varlen_gradients_match_finite_differences():
    """Every gradient of sum <dO, o> + sum_i <dHT[i], h_T[i]> over packed rows (one empty
    sequence, one of a single token), against central differences of the forward."""
    cu = [0, 3, 3, 4, 8]
    T, Hqk, H, dk, dv = cu[-1], 1, 2, 4, 3
    N = len(cu) - 1
    q, k, v = rand(1, T, Hqk, dk), rand(1, T, Hqk, dk), rand(1, T, H, dv)
    a, b, A_log, dt_bias = _gates(T, H)
    h0, dHT = rand(N, H, dk, dv), rand(N, H, dk, dv)
    dO = rand(1, T, H, dv)
    dq, dk_, dv_, dg, dbe, dH0 = oracle.bwd_varlen(q, k, v, a, b, A_log, dt_bias, cu, dO, dHT,
                                                   h0)

    def f():
        o, hT = oracle.fwd_varlen(q, k, v, a, b, A_log, dt_bias, cu, h0)
        return float(np.sum(o * dO) + np.sum(hT * dHT))

    for x, gx in ((q, dq), (k, dk_), (v, dv_), (h0, dH0)):
        np.testing.assert_allclose(gx, _fd(f, x), rtol=1e-6, atol=1e-8)
    # dg, dbeta are w.r.t. the gates the prologue forms: differentiate the core run
    qh, kh, gg, be = oracle.prologue(q, k, a, b, A_log, dt_bias)

    def fc():
        o, hT = oracle.core_fwd_varlen(qh, kh, v, gg, be, cu, h0)
        return float(np.sum(o * dO) + np.sum(hT * dHT))

    np.testing.assert_allclose(dg, _fd(fc, gg), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dbe, _fd(fc, be), rtol=1e-6, atol=1e-8)
