"""Pins of the fp64 oracle against facts fixed by the definition, not by itself.

Each test picks a case where the gated delta rule has a closed form, an
invariant, a library routine or an independent formulation to compare with, so
that a dropped term, a wrong sign or index or a transposed operand anywhere in
``oracle/gdn_oracle.c`` fails at least one of them.  The pages print no worked
example values, so there are no golden vectors from them.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.chunked_numpy import chunked_fwd

RNG = np.random.default_rng(1234)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def orthonormal_keys(B, T, Hqk, dk):
    """k[b, :, hq] are T <= dk mutually orthonormal rows."""
    out = np.zeros((B, T, Hqk, dk))
    for b in range(B):
        for hq in range(Hqk):
            Q, _ = np.linalg.qr(rand(dk, dk))
            out[b, :, hq] = Q[:T]
    return out


# ------------------------------------------------------------------ closed forms

def test_beta_zero_is_pure_gated_decay_of_h0():
    """beta = 0: S_t = (prod_{s<=t} alpha_s) h0 and o_t = S_t^T q_t."""
    B, T, Hqk, H, dk, dv = 2, 37, 2, 4, 5, 3
    qh, kh = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk)
    v = rand(B, T, H, dv)
    g = -np.abs(rand(B, T, H)) * 0.3
    beta = np.zeros((B, T, H))
    h0 = rand(B, H, dk, dv)
    o, hT = oracle.core_fwd(qh, kh, v, g, beta, h0)
    decay = np.exp(np.cumsum(g, axis=1))                    # [B,T,H]
    r = H // Hqk
    for b in range(B):
        for h in range(H):
            for t in range(T):
                exp_o = decay[b, t, h] * (h0[b, h].T @ qh[b, t, h // r])
                np.testing.assert_allclose(o[b, t, h], exp_o, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(hT[b, h], decay[b, -1, h] * h0[b, h], rtol=1e-12)


def test_alpha_one_beta_zero_keeps_h0():
    """alpha = 1 and beta = 0 (taken literally): S is h0 at every step, o_t = h0^T q_t."""
    B, T, Hqk, H, dk, dv = 1, 20, 1, 2, 6, 4
    qh, kh = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk)
    v = rand(B, T, H, dv)
    g = np.zeros((B, T, H))
    beta = np.zeros((B, T, H))
    h0 = rand(B, H, dk, dv)
    o, hT = oracle.core_fwd(qh, kh, v, g, beta, h0)
    exp_o = np.einsum("bhij,bthi->bthj", h0, np.repeat(qh, H // Hqk, axis=2))
    np.testing.assert_allclose(o, exp_o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hT, h0, rtol=0, atol=0)


def test_alpha_one_orthogonal_keys_is_causal_linear_attention():
    """alpha = 1, h0 = 0, orthonormal keys: k_t^T S_{t-1} = 0, so
    o_t = sum_{j<=t} beta_j (q_t . k_j) v_j -- causal linear attention."""
    B, T, Hqk, H, dk, dv = 2, 12, 2, 4, 16, 5
    kh = orthonormal_keys(B, T, Hqk, dk)
    qh = rand(B, T, Hqk, dk)
    v = rand(B, T, H, dv)
    g = np.zeros((B, T, H))
    beta = 1.0 / (1.0 + np.exp(-rand(B, T, H)))
    o, _ = oracle.core_fwd(qh, kh, v, g, beta, None)
    r = H // Hqk
    for b in range(B):
        for h in range(H):
            Q, K = qh[b, :, h // r], kh[b, :, h // r]
            attn = np.tril(Q @ K.T) * beta[b, :, h][None, :]
            np.testing.assert_allclose(o[b, :, h], attn @ v[b, :, h], rtol=1e-11, atol=1e-12)


def test_beta_one_orthonormal_keys_overwrites_the_key_slot():
    """beta = 1 with a unit key: k_t^T S_t = v_t^T exactly, for any alpha and h0.
    With q_t = k_t the output is therefore v_t."""
    B, T, Hqk, H, dk, dv = 1, 10, 1, 3, 10, 4
    kh = orthonormal_keys(B, T, Hqk, dk)
    qh = kh.copy()
    v = rand(B, T, H, dv)
    g = -np.abs(rand(B, T, H))
    beta = np.ones((B, T, H))
    h0 = rand(B, H, dk, dv)
    o, _ = oracle.core_fwd(qh, kh, v, g, beta, h0)
    np.testing.assert_allclose(o, v, rtol=1e-11, atol=1e-12)


# ------------------------------------------------------- independent formulation

@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_chunked_form_equals_recurrence(T):
    """The chunked form (cumulative gates, triangular solve, inter-chunk pass)
    equals the token recurrence up to fp64 rounding."""
    B, Hqk, H, dk, dv = 2, 2, 4, 8, 6
    qh = unit_rows(rand(B, T, Hqk, dk)) / np.sqrt(dk)
    kh = unit_rows(rand(B, T, Hqk, dk))
    v = rand(B, T, H, dv)
    g = -0.05 * np.abs(rand(B, T, H))                # slow decay: state survives chunks
    beta = 1.0 / (1.0 + np.exp(-rand(B, T, H)))
    h0 = rand(B, H, dk, dv)
    o, hT = oracle.core_fwd(qh, kh, v, g, beta, h0)
    o2, hT2 = chunked_fwd(qh, kh, v, g, beta, h0)
    np.testing.assert_allclose(o, o2, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(hT, hT2, rtol=1e-10, atol=1e-11)


# ---------------------------------------------------------------------- prologue

def test_prologue_matches_torch_library_routines():
    """q_hat = scale*normalize(q), k_hat = normalize(k) (eps = 0),
    g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)."""
    B, T, Hqk, H, dk = 2, 9, 2, 4, 8
    q, k = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk)
    a, b = rand(B, T, H) * 8, rand(B, T, H) * 8       # reaches the softplus threshold
    A_log = np.log(RNG.uniform(1, 16, H))
    dt_bias = rand(H) * 8
    scale = 0.37
    qh, kh, g, be = oracle.prologue(q, k, a, b, A_log, dt_bias, eps=0.0, scale=scale)
    tq, tk = torch.from_numpy(q), torch.from_numpy(k)
    np.testing.assert_allclose(qh, scale * torch.nn.functional.normalize(tq, dim=-1, eps=0).numpy(),
                               rtol=1e-13)
    np.testing.assert_allclose(kh, torch.nn.functional.normalize(tk, dim=-1, eps=0).numpy(),
                               rtol=1e-13)
    exp_g = -torch.exp(torch.from_numpy(A_log)) * torch.nn.functional.softplus(
        torch.from_numpy(a) + torch.from_numpy(dt_bias))
    np.testing.assert_allclose(g, exp_g.numpy(), rtol=1e-12)
    np.testing.assert_allclose(be, torch.sigmoid(torch.from_numpy(b)).numpy(), rtol=1e-13)


def test_prologue_default_scale_and_padding():
    B, T, Hqk, H, dk = 2, 6, 1, 2, 16
    q, k = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk)
    a, b = rand(B, T, H), rand(B, T, H)
    qh, kh, g, be = oracle.prologue(q, k, a, b, np.zeros(H), np.zeros(H), valid_len=[4, 6])
    np.testing.assert_allclose(np.linalg.norm(qh, axis=-1), 0.25, rtol=1e-6)   # 1/sqrt(16)
    np.testing.assert_allclose(np.linalg.norm(kh, axis=-1), 1.0, rtol=1e-6)
    assert np.all(g[0, 4:] == 0) and np.all(be[0, 4:] == 0)
    assert np.all(g[0, :4] < 0) and np.all(be[1] > 0)


# --------------------------------------------------------------------- summaries

def _gates(B, T, H, slow=True):
    a, b = rand(B, T, H), rand(B, T, H)
    A_log = np.log(RNG.uniform(1, 16, H))
    dt_bias = (-6.0 + 0.1 * rand(H)) if slow else rand(H)
    return a, b, A_log, dt_bias


def test_summary_is_the_affine_map_of_the_segment():
    """run from X = M X + S for random X (linearity of the recurrence in the state)."""
    B, T, Hqk, H, dk, dv = 2, 50, 1, 2, 6, 5
    q, k, v = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk), rand(B, T, H, dv)
    a, b, A_log, dt_bias = _gates(B, T, H)
    M, S = oracle.summary(k, v, a, b, A_log, dt_bias)
    for _ in range(3):
        X = rand(B, H, dk, dv)
        _, hT = oracle.fwd(q, k, v, a, b, A_log, dt_bias, h0=X)
        np.testing.assert_allclose(hT, np.einsum("bhij,bhjk->bhik", M, X) + S, rtol=1e-11,
                                   atol=1e-12)


def test_summary_M_is_the_explicit_product_of_token_maps():
    """M = A_T ... A_1 with A_t = alpha_t (I - beta_t k_t k_t^T), formed explicitly."""
    B, T, Hqk, H, dk, dv = 1, 9, 1, 2, 4, 3
    q, k, v = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk), rand(B, T, H, dv)
    a, b, A_log, dt_bias = _gates(B, T, H)
    M, S = oracle.summary(k, v, a, b, A_log, dt_bias)
    _, kh, g, be = oracle.prologue(q, k, a, b, A_log, dt_bias)
    for h in range(H):
        Mx = np.eye(dk)
        Sx = np.zeros((dk, dv))
        for t in range(T):
            kt = kh[0, t, 0][:, None]
            At = np.exp(g[0, t, h]) * (np.eye(dk) - be[0, t, h] * kt @ kt.T)
            Mx = At @ Mx
            Sx = At @ Sx + be[0, t, h] * kt @ v[0, t, h][None, :]
        np.testing.assert_allclose(M[0, h], Mx, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(S[0, h], Sx, rtol=1e-12, atol=1e-14)


def test_compose_and_prefix_reproduce_the_monolithic_run():
    """(M,S) of [0,T) = composition of the segments' summaries; the exclusive
    prefix gives each segment's initial state, and running each segment from it
    reproduces the monolithic o and h_T."""
    B, T, Hqk, H, dk, dv = 1, 96, 2, 4, 6, 5
    q, k, v = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk), rand(B, T, H, dv)
    a, b, A_log, dt_bias = _gates(B, T, H)
    h0 = rand(B, H, dk, dv)
    o, hT = oracle.fwd(q, k, v, a, b, A_log, dt_bias, h0=h0)
    Mw, Sw = oracle.summary(k, v, a, b, A_log, dt_bias)
    cuts = [0, 17, 64, 96]
    Ms, Ss = [], []
    for s0, s1 in zip(cuts[:-1], cuts[1:]):
        M, S = oracle.summary(k[:, s0:s1], v[:, s0:s1], a[:, s0:s1], b[:, s0:s1], A_log, dt_bias)
        Ms.append(M)
        Ss.append(S)
    Mc, Sc = oracle.compose(Ms[1], Ss[1], Ms[0], Ss[0])
    Mc, Sc = oracle.compose(Ms[2], Ss[2], Mc, Sc)
    np.testing.assert_allclose(Mc, Mw, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(Sc, Sw, rtol=1e-11, atol=1e-13)
    Hin, Hout = oracle.prefix(np.stack(Ms), np.stack(Ss), h0)
    np.testing.assert_allclose(Hin[0], h0, rtol=0, atol=0)
    np.testing.assert_allclose(Hout, hT, rtol=1e-11, atol=1e-12)
    for i, (s0, s1) in enumerate(zip(cuts[:-1], cuts[1:])):
        oi, hi = oracle.fwd(q[:, s0:s1], k[:, s0:s1], v[:, s0:s1], a[:, s0:s1], b[:, s0:s1],
                            A_log, dt_bias, h0=Hin[i])
        np.testing.assert_allclose(oi, o[:, s0:s1], rtol=1e-11, atol=1e-12)


def test_compose_is_associative_with_identity():
    dk, dv = 5, 3
    Ms = [rand(2, dk, dk) for _ in range(3)]
    Ss = [rand(2, dk, dv) for _ in range(3)]
    left = oracle.compose(Ms[2], Ss[2], *oracle.compose(Ms[1], Ss[1], Ms[0], Ss[0]))
    right = oracle.compose(*oracle.compose(Ms[2], Ss[2], Ms[1], Ss[1]), Ms[0], Ss[0])
    np.testing.assert_allclose(left[0], right[0], rtol=1e-12)
    np.testing.assert_allclose(left[1], right[1], rtol=1e-12)
    I = np.broadcast_to(np.eye(dk), (2, dk, dk))
    Z = np.zeros((2, dk, dv))
    ident = oracle.compose(Ms[0], Ss[0], I, Z)
    np.testing.assert_allclose(ident[0], Ms[0], rtol=0, atol=0)
    np.testing.assert_allclose(ident[1], Ss[0], rtol=0, atol=0)


# ------------------------------------------------------------------------ padding

def test_padding_matches_the_unpadded_run():
    """valid_len = L: o[:L] and h_T equal the L-token run, o[L:] = 0; gradients of
    valid tokens equal those of the L-token run, padded tokens get none."""
    B, T, Hqk, H, dk, dv = 2, 75, 1, 2, 6, 4
    L = [70, 75]
    q, k, v = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk), rand(B, T, H, dv)
    a, b, A_log, dt_bias = _gates(B, T, H)
    h0 = rand(B, H, dk, dv)
    dO, dHT = rand(B, T, H, dv), rand(B, H, dk, dv)
    o, hT = oracle.fwd(q, k, v, a, b, A_log, dt_bias, h0=h0, valid_len=L)
    grads = oracle.bwd(q, k, v, a, b, A_log, dt_bias, dO, dHT, h0=h0, valid_len=L)
    for bi, Lb in enumerate(L):
        sl = (slice(bi, bi + 1), slice(0, Lb))
        ou, hu = oracle.fwd(q[sl], k[sl], v[sl], a[sl], b[sl], A_log, dt_bias, h0=h0[bi:bi + 1])
        np.testing.assert_allclose(o[bi, :Lb], ou[0], rtol=1e-12, atol=1e-13)
        assert np.all(o[bi, Lb:] == 0)
        np.testing.assert_allclose(hT[bi], hu[0], rtol=1e-12, atol=1e-13)
        gu = oracle.bwd(q[sl], k[sl], v[sl], a[sl], b[sl], A_log, dt_bias, dO[sl],
                        dHT[bi:bi + 1], h0=h0[bi:bi + 1])
        for gp, gq in zip(grads[:5], gu[:5]):
            np.testing.assert_allclose(gp[bi, :Lb], gq[0], rtol=1e-11, atol=1e-12)
            assert np.all(gp[bi, Lb:] == 0)
        np.testing.assert_allclose(grads[5][bi], gu[5][0], rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------- gradients

def _loss_core(qh, kh, v, g, beta, h0, dO, dHT):
    o, hT = oracle.core_fwd(qh, kh, v, g, beta, h0)
    return float(np.sum(o * dO) + np.sum(hT * dHT))


def _fd(fun, x, eps=1e-6):
    grad = np.zeros_like(x)
    flat = x.reshape(-1)
    gflat = grad.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        flat[i] = old + eps
        fp = fun()
        flat[i] = old - eps
        fm = fun()
        flat[i] = old
        gflat[i] = (fp - fm) / (2 * eps)
    return grad


def test_core_gradients_match_finite_differences():
    B, T, Hqk, H, dk, dv = 1, 8, 1, 2, 4, 4
    qh, kh = rand(B, T, Hqk, dk), unit_rows(rand(B, T, Hqk, dk))
    v = rand(B, T, H, dv)
    g = -0.3 * np.abs(rand(B, T, H))
    beta = 1.0 / (1.0 + np.exp(-rand(B, T, H)))
    h0 = rand(B, H, dk, dv)
    dO, dHT = rand(B, T, H, dv), rand(B, H, dk, dv)
    dqh, dkh, dv_, dg, dbe, dH0 = oracle.core_bwd(qh, kh, v, g, beta, dO, dHT, h0=h0)
    f = lambda: _loss_core(qh, kh, v, g, beta, h0, dO, dHT)  # noqa: E731
    for x, gx in ((qh, dqh), (kh, dkh), (v, dv_), (g, dg), (beta, dbe), (h0, dH0)):
        np.testing.assert_allclose(gx, _fd(f, x), rtol=1e-6, atol=1e-8)


def test_full_gradients_match_finite_differences():
    """Raw q, k through the L2 norm and scale, summed over the V heads of a group."""
    B, T, Hqk, H, dk, dv = 2, 7, 1, 3, 4, 3
    q, k, v = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk), rand(B, T, H, dv)
    a, b, A_log, dt_bias = _gates(B, T, H, slow=False)
    h0 = rand(B, H, dk, dv)
    dO, dHT = rand(B, T, H, dv), rand(B, H, dk, dv)
    L = [7, 5]
    dq, dk_, dv_, dg, dbe, dH0 = oracle.bwd(q, k, v, a, b, A_log, dt_bias, dO, dHT, h0=h0,
                                            valid_len=L)

    def f():
        o, hT = oracle.fwd(q, k, v, a, b, A_log, dt_bias, h0=h0, valid_len=L)
        return float(np.sum(o * dO) + np.sum(hT * dHT))

    for x, gx in ((q, dq), (k, dk_), (v, dv_), (h0, dH0)):
        np.testing.assert_allclose(gx, _fd(f, x), rtol=1e-6, atol=1e-8)


def test_gate_gradients_chain_to_the_parameters():
    """dL/da_t = dg_t * dg_t/da_t and dL/db_t = dbeta_t * dbeta_t/db_t, with the
    prologue's own derivatives taken numerically; dL/dA_log, dL/ddt_bias likewise."""
    B, T, Hqk, H, dk, dv = 1, 6, 1, 2, 4, 3
    q, k, v = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk), rand(B, T, H, dv)
    a, b, A_log, dt_bias = _gates(B, T, H, slow=False)
    dO, dHT = rand(B, T, H, dv), rand(B, H, dk, dv)
    _, _, _, dg, dbe, _ = oracle.bwd(q, k, v, a, b, A_log, dt_bias, dO, dHT)

    def loss():
        o, hT = oracle.fwd(q, k, v, a, b, A_log, dt_bias)
        return float(np.sum(o * dO) + np.sum(hT * dHT))

    def gates():
        _, _, g, be = oracle.prologue(q, k, a, b, A_log, dt_bias)
        return g, be

    eps = 1e-6
    for x in (a, b, A_log, dt_bias):
        flat = x.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + eps
            lp, (gp, bp) = loss(), gates()
            flat[i] = old - eps
            lm, (gm, bm) = loss(), gates()
            flat[i] = old
            fd = (lp - lm) / (2 * eps)
            chain = np.sum(dg * (gp - gm) / (2 * eps)) + np.sum(dbe * (bp - bm) / (2 * eps))
            np.testing.assert_allclose(chain, fd, rtol=1e-5, atol=1e-8)


@pytest.mark.parametrize("valid_len", [None, [4, 6]])
def test_gate_parameter_gradients_match_finite_differences(valid_len):
    """oracle.gate_param_bwd (da, db, dA_log, ddt_bias from dg, dbeta) against central
    finite differences of the whole loss L = <dO, o> + <dHT, hT> in every gate input
    and parameter, with and without trailing padding."""
    B, T, Hqk, H, dk, dv = 2, 6, 1, 2, 4, 3
    q, k, v = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk), rand(B, T, H, dv)
    a, b, A_log, dt_bias = _gates(B, T, H, slow=True)
    dO, dHT = rand(B, T, H, dv), rand(B, H, dk, dv)
    vl = None if valid_len is None else np.array(valid_len, dtype=np.int32)
    _, _, _, dg, dbe, _ = oracle.bwd(q, k, v, a, b, A_log, dt_bias, dO, dHT, valid_len=vl)
    da, db, dA, ddt = oracle.gate_param_bwd(a, b, A_log, dt_bias, dg, dbe, valid_len=vl)

    def loss():
        o, hT = oracle.fwd(q, k, v, a, b, A_log, dt_bias, valid_len=vl)
        return float(np.sum(o * dO) + np.sum(hT * dHT))

    eps = 1e-6
    for x, grad in ((a, da), (b, db), (A_log, dA), (dt_bias, ddt)):
        flat, gflat = x.reshape(-1), grad.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + eps
            lp = loss()
            flat[i] = old - eps
            lm = loss()
            flat[i] = old
            np.testing.assert_allclose(gflat[i], (lp - lm) / (2 * eps), rtol=1e-5, atol=1e-8)


def test_gradient_summary_and_reverse_prefix_reproduce_dH0():
    """D of a segment = dH_in with dH_out = 0; the reverse prefix of (M^T, D) over
    segments gives the monolithic dH0, and per-segment backward from dH_out[i]
    gives the monolithic token gradients."""
    B, T, Hqk, H, dk, dv = 1, 80, 1, 2, 5, 4
    q, k, v = rand(B, T, Hqk, dk), rand(B, T, Hqk, dk), rand(B, T, H, dv)
    a, b, A_log, dt_bias = _gates(B, T, H)
    h0 = rand(B, H, dk, dv)
    dO, dHT = rand(B, T, H, dv), rand(B, H, dk, dv)
    full = oracle.bwd(q, k, v, a, b, A_log, dt_bias, dO, dHT, h0=h0)
    cuts = [0, 30, 64, 80]
    segs = list(zip(cuts[:-1], cuts[1:]))
    Ms, Ss, Ds = [], [], []
    for s0, s1 in segs:
        sl = (slice(None), slice(s0, s1))
        M, S = oracle.summary(k[sl], v[sl], a[sl], b[sl], A_log, dt_bias)
        D = oracle.summary_bwd(q[sl], k[sl], a[sl], b[sl], A_log, dt_bias, dO[sl])
        zero = oracle.bwd(q[sl], k[sl], v[sl], a[sl], b[sl], A_log, dt_bias, dO[sl], None,
                          h0=rand(B, H, dk, dv))[5]
        np.testing.assert_allclose(D, zero, rtol=1e-11, atol=1e-12)
        Ms.append(M)
        Ss.append(S)
        Ds.append(D)
    Hin, _ = oracle.prefix(np.stack(Ms), np.stack(Ss), h0)
    dHout, dH0 = oracle.prefix_bwd(np.stack(Ms), np.stack(Ds), dHT)
    np.testing.assert_allclose(dH0, full[5], rtol=1e-11, atol=1e-12)
    for i, (s0, s1) in enumerate(segs):
        sl = (slice(None), slice(s0, s1))
        gi = oracle.bwd(q[sl], k[sl], v[sl], a[sl], b[sl], A_log, dt_bias, dO[sl], dHout[i],
                        h0=Hin[i])
        for gseg, gfull in zip(gi[:5], full[:5]):
            np.testing.assert_allclose(gseg, gfull[:, s0:s1], rtol=1e-10, atol=1e-11)


def test_empty_sequence():
    B, T, Hqk, H, dk, dv = 2, 0, 1, 2, 4, 3
    q, k, v = np.zeros((B, T, Hqk, dk)), np.zeros((B, T, Hqk, dk)), np.zeros((B, T, H, dv))
    a = b = np.zeros((B, T, H))
    h0 = rand(B, H, dk, dv)
    o, hT = oracle.fwd(q, k, v, a, b, np.zeros(H), np.zeros(H), h0=h0)
    assert o.shape == (B, 0, H, dv)
    np.testing.assert_allclose(hT, h0, rtol=0, atol=0)
    M, S = oracle.summary(k, v, a, b, np.zeros(H), np.zeros(H))
    np.testing.assert_allclose(M, np.broadcast_to(np.eye(dk), M.shape), rtol=0, atol=0)
    assert np.all(S == 0)
