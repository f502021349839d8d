"""Pins of the gated RMSNorm oracle (oracle/rmsnorm.py) to things other than itself.

- With the gate replaced by silu(z) = 1 (z chosen so), the output equals torch's rms_norm
  (a library routine) times w, in fp64.
- A worked row by hand: o = (3, 4), eps = 0: rms = sqrt(12.5).
- With eps = 0 the output does not change when o is scaled by c > 0.
- The backward matches central finite differences of the forward (fp64, tiny sizes).
"""
import numpy as np
import pytest
import torch

import oracle


def _silu(z):
    return z / (1.0 + np.exp(-z))


def test_matches_torch_rms_norm():
    rng = np.random.default_rng(1)
    o = rng.standard_normal((3, 5, 16))
    w = rng.standard_normal(16)
    # silu(z) = 1: z solves z sigmoid(z) = 1 (z ~ 1.2785), found by bisection here
    lo, hi = 0.0, 3.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        lo, hi = (mid, hi) if _silu(mid) < 1.0 else (lo, mid)
    z = np.full_like(o, 0.5 * (lo + hi))
    y = oracle.rmsnorm_gated_fwd(o, z, w, eps=1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(o), (16,), torch.from_numpy(w),
                                       eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_worked_row():
    y = oracle.rmsnorm_gated_fwd(np.array([3.0, 4.0]), np.array([2.0, -1.0]),
                                 np.array([1.0, 2.0]), eps=0.0)
    rms = np.sqrt(12.5)
    np.testing.assert_allclose(y, [3.0 / rms * 1.0 * _silu(2.0), 4.0 / rms * 2.0 * _silu(-1.0)],
                               rtol=1e-14)


def test_scale_invariance_without_eps():
    rng = np.random.default_rng(2)
    o, z, w = rng.standard_normal((4, 8)), rng.standard_normal((4, 8)), rng.standard_normal(8)
    np.testing.assert_allclose(oracle.rmsnorm_gated_fwd(7.5 * o, z, w, eps=0.0),
                               oracle.rmsnorm_gated_fwd(o, z, w, eps=0.0), rtol=1e-12)


@pytest.mark.parametrize("shape", [(2, 3, 6), (5, 4)])
def test_backward_matches_finite_differences(shape):
    rng = np.random.default_rng(len(shape))
    o, z = rng.standard_normal(shape), rng.standard_normal(shape)
    w, dy = rng.standard_normal(shape[-1]), rng.standard_normal(shape)
    eps_n, h = 1e-6, 1e-6
    do, dz, dw = oracle.rmsnorm_gated_bwd(o, z, w, dy, eps=eps_n)

    def loss(o_, z_, w_):
        return float(np.sum(oracle.rmsnorm_gated_fwd(o_, z_, w_, eps=eps_n) * dy))

    def fd(arr, f):
        g = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            g[idx] = (f(p) - f(m)) / (2 * h)
        return g

    np.testing.assert_allclose(do, fd(o, lambda v: loss(v, z, w)), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dz, fd(z, lambda v: loss(o, v, w)), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dw, fd(w, lambda v: loss(o, z, v)), rtol=1e-6, atol=1e-7)
