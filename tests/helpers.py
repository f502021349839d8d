"""Shared test helpers: error metrics and head sampling (no method arithmetic)."""
import numpy as np
import torch

# Tolerances of the parity contract: bf16 I/O with fp32 accumulation, fp32 mode.
BF16_REL_L2 = 1e-2
BF16_MAX_REL = 1e-1
FP32_REL_L2 = 1e-5


def to64(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(x, ref):
    x, ref = to64(x), to64(ref)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0:
        return float(num)
    return float(num / den)


def max_rel(x, ref):
    x, ref = to64(x), to64(ref)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(x - ref)) if ref.size else 0.0
    return float(num / den) if den > 0 else float(num)


def assert_close(name, x, ref, dtype):
    x64, r64 = to64(x), to64(ref)
    assert np.all(np.isfinite(x64)), f"{name}: non-finite values"
    e2 = rel_l2(x64, r64)
    if dtype == torch.float32:
        assert e2 <= FP32_REL_L2, f"{name}: rel-L2 {e2:.3e} > {FP32_REL_L2}"
    else:
        em = max_rel(x64, r64)
        assert e2 <= BF16_REL_L2, f"{name}: rel-L2 {e2:.3e} > {BF16_REL_L2}"
        assert em <= BF16_MAX_REL, f"{name}: max-abs/ref-abs-max {em:.3e} > {BF16_MAX_REL}"
    return e2


def head_slice(inp: dict, hq0: int, nq: int, r: int) -> dict:
    """Inputs restricted to Q/K heads [hq0, hq0+nq) and their r V heads each."""
    h0, h1 = hq0 * r, (hq0 + nq) * r
    out = {}
    for key, val in inp.items():
        if val is None or key == "valid_len":
            out[key] = val
        elif key in ("q", "k"):
            out[key] = val[:, :, hq0:hq0 + nq]
        elif key in ("v", "dO"):
            out[key] = val[:, :, h0:h1]
        elif key in ("a", "b"):
            out[key] = val[:, :, h0:h1]
        elif key in ("A_log", "dt_bias"):
            out[key] = val[h0:h1]
        elif key in ("h0", "dHT"):
            out[key] = val[:, h0:h1]
        else:
            out[key] = val
    return out
