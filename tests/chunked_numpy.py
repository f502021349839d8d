"""A second, chunked fp64 formulation of the GDN forward -- test-only.

It pins the oracle (a token-by-token recurrence) against an independent
formulation: the chunked form with cumulative gates inside a chunk, the
triangular system (I + tril(diag(beta) K K^T o Gamma, -1)), and the inter-chunk
state pass.  Written with numpy/scipy primitives only; it imports nothing from
the oracle or from the CUDA library.
"""
import numpy as np
from scipy.linalg import solve_triangular


def chunked_fwd(qh, kh, v, g, beta, h0=None, C=64):
    """qh, kh [B,T,Hqk,dk]; v [B,T,H,dv]; g, beta [B,T,H]; h0 [B,H,dk,dv] -> (o, hT)."""
    B, T, Hqk, dk = qh.shape
    H, dv = v.shape[2], v.shape[3]
    r = H // Hqk
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else h0[b, h].copy()
            for t0 in range(0, T, C):
                t1 = min(T, t0 + C)
                Q = qh[b, t0:t1, h // r]
                K = kh[b, t0:t1, h // r]
                V = v[b, t0:t1, h]
                be = beta[b, t0:t1, h]
                G = np.cumsum(g[b, t0:t1, h])
                gam = np.exp(G)
                n = t1 - t0
                Gam = np.exp(G[:, None] - G[None, :])
                lower = np.tril(np.ones((n, n)), -1)
                A = lower * (be[:, None] * (K @ K.T) * Gam)
                IA = np.eye(n) + A
                W = solve_triangular(IA, (be * gam)[:, None] * K, lower=True, unit_diagonal=True)
                U = solve_triangular(IA, be[:, None] * V, lower=True, unit_diagonal=True)
                Vn = U - W @ S
                P = np.tril(Q @ K.T * Gam)
                o[b, t0:t1, h] = gam[:, None] * (Q @ S) + P @ Vn
                Kt = np.exp(G[-1] - G)[:, None] * K
                S = gam[-1] * S + Kt.T @ Vn
            hT[b, h] = S
    return o, hT
