"""fp64 CPU oracle of the gated RMSNorm epilogue on o -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this module; it shares no code with the CUDA library.

The pages place an RMSNorm with a gate after the core ("linear attention cp #1035", section
"What does this PR do": the output goes through RMSNorm, the gate and the output projection;
the test report names the module "RMSNormGated").  They leave the formula open; this oracle
takes the plainest reading: per row of D elements (one token and V head of o),
    n = o / sqrt(mean(o^2) + eps),   y = n * w * silu(z)
with w [D] a learned scale shared by all rows and z the gate tensor of o's shape.
Backward, from the chain rule on that definition (r = 1 / sqrt(mean(o^2) + eps)):
    dn = dy w silu(z)
    do = r (dn - n mean(dn n))
    dz = dy n w silu'(z),   silu'(z) = sigmoid(z) (1 + z (1 - sigmoid(z)))
    dw = sum over rows of dy n silu(z)
"""
from __future__ import annotations

import numpy as np


def _sigmoid(a):
    return 0.5 * (1.0 + np.tanh(0.5 * a))


def rmsnorm_gated_fwd(o, z, w, eps: float = 1e-6) -> np.ndarray:
    """y [..., D] from o, z [..., D] and w [D]."""
    o = np.asarray(o, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o * r * w * (z * _sigmoid(z))


def rmsnorm_gated_bwd(o, z, w, dy, eps: float = 1e-6):
    """(do, dz [..., D], dw [D]) for the forward above."""
    o = np.asarray(o, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    n = o * r
    s = _sigmoid(z)
    g = z * s
    dn = dy * w * g
    do = r * (dn - n * np.mean(dn * n, axis=-1, keepdims=True))
    dz = dy * n * w * s * (1.0 + z * (1.0 - s))
    dw = np.sum((dy * n * g).reshape(-1, o.shape[-1]), axis=0)
    return do, dz, dw
