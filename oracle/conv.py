"""fp64 CPU oracle of the causal depthwise Conv1D + SiLU prologue -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this module; it shares no code with the CUDA library.

The pages name the step that feeds the core: a depthwise Conv1D over time on the projected
q, k, v ("linear attention cp #1035", section "What does this PR do": the "ulysses" mode runs
the depthwise Conv1D and the Gated DeltaNet on the full sequence; the "p2p" mode keeps the
local sequence shard and exchanges only the left halo that the Conv1D needs with the
neighbouring rank).  They leave the tap count and the activation open; this oracle takes the
plainest reading consistent with a causal depthwise convolution feeding the core: K taps per
channel (K = 4 in the layers the pages test), an optional per-channel bias, and SiLU.

Definition (one row b, channel c; x~ is x with the K - 1 halo tokens before token 0):
    x~[s] = x[s]                for 0 <= s < T
    x~[s] = halo[K - 1 + s]     for -(K - 1) <= s < 0   (zeros when no halo is given)
    a[t]  = bias + sum_{i=0}^{K-1} w[i] x~[t - (K - 1) + i]
    y[t]  = a[t] sigmoid(a[t])
Backward, from the chain rule on that definition:
    ds[t]    = dy[t] sigmoid(a[t]) (1 + a[t] (1 - sigmoid(a[t])))
    dx~[s]   = sum_i w[i] ds[s + (K - 1) - i]   over the t = s + (K - 1) - i in [0, T)
    dx       = dx~[0 .. T),   dhalo = dx~[-(K - 1) .. 0)
    dw[i]    = sum_{b, t} ds[t] x~[t - (K - 1) + i],   dbias = sum_{b, t} ds[t]
"""
from __future__ import annotations

import numpy as np


def _extended(x: np.ndarray, halo, K: int) -> np.ndarray:
    """x~ [B, T + K - 1, C]: the halo tokens (or zeros), then x."""
    B, T, C = x.shape
    h = np.zeros((B, K - 1, C)) if halo is None else np.asarray(halo, dtype=np.float64)
    if h.shape != (B, K - 1, C):
        raise ValueError(f"halo must be [B, K-1, C] = {(B, K - 1, C)}, got {h.shape}")
    return np.concatenate([h, x], axis=1)


def _preact(xt: np.ndarray, w: np.ndarray, bias, T: int) -> np.ndarray:
    K = w.shape[1]
    a = np.zeros((xt.shape[0], T, xt.shape[2]))
    for i in range(K):  # tap i reads token t - (K - 1) + i, i.e. row i + t of x~
        a += w[:, i] * xt[:, i:i + T, :]
    if bias is not None:
        a += np.asarray(bias, dtype=np.float64)
    return a


def _sigmoid(a: np.ndarray) -> np.ndarray:
    return 0.5 * (1.0 + np.tanh(0.5 * a))


def conv_silu_fwd(x, w, bias=None, halo=None) -> np.ndarray:
    """y [B, T, C] from x [B, T, C], w [C, K], bias [C] or None, halo [B, K-1, C] or None."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    a = _preact(_extended(x, halo, w.shape[1]), w, bias, x.shape[1])
    return a * _sigmoid(a)


def conv_silu_bwd(x, w, bias, halo, dy):
    """(dx [B,T,C], dw [C,K], dbias [C], dhalo [B,K-1,C]) for the forward above."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    B, T, C = x.shape
    K = w.shape[1]
    xt = _extended(x, halo, K)
    a = _preact(xt, w, bias, T)
    sg = _sigmoid(a)
    ds = dy * sg * (1.0 + a * (1.0 - sg))
    dxt = np.zeros_like(xt)
    dw = np.zeros((C, K))
    for i in range(K):
        dxt[:, i:i + T, :] += w[:, i] * ds
        dw[:, i] = np.sum(ds * xt[:, i:i + T, :], axis=(0, 1))
    return dxt[:, K - 1:, :], dw, ds.sum(axis=(0, 1)), dxt[:, :K - 1, :]
