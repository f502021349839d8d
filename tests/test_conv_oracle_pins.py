"""Pins of the Conv1D + SiLU oracle (oracle/conv.py) to things other than itself.

- The pre-activation with no halo and no bias is numpy's full discrete convolution of
  each channel with its reversed taps, cut to the first T outputs (a library routine).
- K = 1 is the elementwise map y = silu(w x + bias) (closed form).
- The backward matches central finite differences of the forward (fp64, tiny sizes).
- Splitting a row into two segments, the second fed the first's last K - 1 tokens as its
  halo, gives the unsplit outputs; the second segment's dhalo added to the first's last
  K - 1 token gradients gives the unsplit dx (the left-halo exchange of the "p2p" mode of
  "linear attention cp #1035" and its reverse).
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _silu(a):
    return a / (1.0 + np.exp(-a))


def _draw(rng, B, T, C, K, halo=True, bias=True):
    x = rng.standard_normal((B, T, C))
    w = rng.standard_normal((C, K)) * 0.5
    b = rng.standard_normal(C) * 0.3 if bias else None
    h = rng.standard_normal((B, K - 1, C)) if halo else None
    return x, w, b, h


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_preactivation_is_numpy_convolution(K):
    rng = np.random.default_rng(10 + K)
    x, w, _, _ = _draw(rng, 2, 37, 5, K, halo=False, bias=False)
    y = oracle.conv_silu_fwd(x, w)
    for bi in range(2):
        for c in range(5):
            a = np.convolve(x[bi, :, c], w[c, ::-1])[:37]
            np.testing.assert_allclose(y[bi, :, c], _silu(a), rtol=1e-13, atol=1e-13)


def test_k1_is_elementwise():
    rng = np.random.default_rng(3)
    x, w, b, _ = _draw(rng, 2, 9, 6, 1, halo=False)
    y = oracle.conv_silu_fwd(x, w, b)
    np.testing.assert_allclose(y, _silu(x * w[:, 0] + b), rtol=1e-13, atol=1e-13)


def test_halo_enters_as_the_tokens_before_zero():
    rng = np.random.default_rng(4)
    x, w, b, h = _draw(rng, 1, 6, 3, 4)
    y = oracle.conv_silu_fwd(x, w, b, h)
    # token 0 reads halo rows 0..2 through taps 0..2 and x[0] through tap 3
    a0 = b + w[:, 0] * h[0, 0] + w[:, 1] * h[0, 1] + w[:, 2] * h[0, 2] + w[:, 3] * x[0, 0]
    np.testing.assert_allclose(y[0, 0], _silu(a0), rtol=1e-13)


@pytest.mark.parametrize("K,T", [(4, 7), (3, 2), (1, 5), (4, 1)])
def test_backward_matches_finite_differences(K, T):
    rng = np.random.default_rng(20 + K * 10 + T)
    x, w, b, h = _draw(rng, 2, T, 3, K, halo=K > 1)
    dy = rng.standard_normal((2, T, 3))
    dx, dw, db, dh = oracle.conv_silu_bwd(x, w, b, h, dy)
    eps = 1e-6

    def loss(x_, w_, b_, h_):
        return float(np.sum(oracle.conv_silu_fwd(x_, w_, b_, h_) * dy))

    def fd(arr, setter):
        g = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            g[idx] = (setter(p) - setter(m)) / (2 * eps)
        return g

    np.testing.assert_allclose(dx, fd(x, lambda v: loss(v, w, b, h)), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dw, fd(w, lambda v: loss(x, v, b, h)), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(db, fd(b, lambda v: loss(x, w, v, h)), rtol=1e-6, atol=1e-7)
    if h is not None:
        np.testing.assert_allclose(dh, fd(h, lambda v: loss(x, w, b, v)), rtol=1e-6, atol=1e-7)
    else:
        assert dh.shape == (2, 0, 3)


@pytest.mark.parametrize("T1", [1, 2, 5, 11])
def test_segments_compose_through_the_halo(T1):
    K, T = 4, 16
    rng = np.random.default_rng(40 + T1)
    x, w, b, h = _draw(rng, 2, T, 4, K)
    dy = rng.standard_normal((2, T, 4))
    y = oracle.conv_silu_fwd(x, w, b, h)
    dx, dw, db, dh = oracle.conv_silu_bwd(x, w, b, h, dy)
    xt = np.concatenate([h, x], axis=1)  # the second segment's halo: the K-1 tokens before T1
    h2 = xt[:, T1:T1 + K - 1]
    y1 = oracle.conv_silu_fwd(x[:, :T1], w, b, h)
    y2 = oracle.conv_silu_fwd(x[:, T1:], w, b, h2)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=1), y, rtol=1e-12, atol=1e-12)
    dx1, dw1, db1, dh1 = oracle.conv_silu_bwd(x[:, :T1], w, b, h, dy[:, :T1])
    dx2, dw2, db2, dh2 = oracle.conv_silu_bwd(x[:, T1:], w, b, h2, dy[:, T1:])
    g = np.concatenate([dh1, dx1], axis=1)  # gradient of x~ rows -(K-1) .. T1-1
    g[:, T1:T1 + K - 1] += dh2
    np.testing.assert_allclose(g[:, K - 1:], dx[:, :T1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g[:, :K - 1], dh, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dx2, dx[:, T1:], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw1 + dw2, dw, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(db1 + db2, db, rtol=1e-12, atol=1e-12)
