"""Seeded synthetic inputs for the Gated DeltaNet core.

This module holds none of the method's arithmetic: it only draws random tensors
with the shapes and distributions of the workloads (q, k, v, a, b ~ N(0,1);
A_log = log U(1,16); dt_bias ~ N(0,1); optional h0 ~ N(0, 0.1^2); output and
final-state gradients ~ N(0,1), optionally divided by sqrt(numel) as in the
"Linear Attention CP 融合算子 PR #1114 测试报告", section 4.1, which normalises
dO/dHT by tensor size).  It is shared by the tests, the benchmark and the smoke
check, which feed the same values to the CUDA library and to the CPU oracle.

Everything is drawn on the CPU with a seeded ``torch.Generator`` in fp32 and then
rounded once to the I/O dtype; the oracle reads the rounded values, so both sides
see identical inputs.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass
class Workload:
    """Shape and distribution recipe of one synthetic GDN problem."""

    name: str
    B: int
    T: int
    Hqk: int
    H: int
    dk: int
    dv: int
    dtype: torch.dtype = torch.bfloat16
    h0_std: Optional[float] = None          # None: no initial state
    grad_scale: str = "unit"                # "unit": N(0,1); "numel": N(0,1)/sqrt(numel)
    with_dHT: bool = False                  # draw a final-state gradient as well
    valid_len: Optional[list] = None        # per-row valid length (trailing padding)
    segments: int = 0                       # 0: library chooses
    decay_stress: bool = False              # dt_bias = -6 + N(0, 0.1^2): slow decay
    seed: int = 0
    extra: dict = field(default_factory=dict)


# The workloads of the pages' single-device GDN-core matrix (H=32 V heads from 16
# Q/K heads, head dim 128, chunk 64) plus a tiny fp32 case small enough for the
# oracle in a fraction of a second.
TINY = Workload("tiny_fp32_T128_h4x8_d16", B=1, T=128, Hqk=4, H=8, dk=16, dv=16,
                dtype=torch.float32, segments=2, seed=0)
FWD_8K = Workload("fwd_bf16_T8192_h16x32_d128", B=1, T=8192, Hqk=16, H=32, dk=128, dv=128,
                  seed=1)
STATEFUL_32K = Workload("fwdbwd_bf16_T32768_h16x32_d128_stateful", B=1, T=32768, Hqk=16,
                        H=32, dk=128, dv=128, h0_std=0.1, grad_scale="numel", with_dHT=True,
                        seed=2)
SEGMENTED_32K = Workload("segments8x4096_bf16_T32768_h16x32_d128", B=1, T=32768, Hqk=16,
                         H=32, dk=128, dv=128, h0_std=0.1, grad_scale="numel",
                         with_dHT=True, segments=8, seed=3)
PADDED_8K = Workload("padded_bf16_B2_T8192_valid7777", B=2, T=8192, Hqk=16, H=32, dk=128,
                     dv=128, valid_len=[7777, 7777], seed=4)
LONG_64K = Workload("fwdbwd_bf16_T65536_h16x32_d128_stateful", B=1, T=65536, Hqk=16, H=32,
                    dk=128, dv=128, h0_std=0.1, grad_scale="numel", with_dHT=True, seed=5)


def _normal(gen, shape):
    return torch.randn(*shape, generator=gen, dtype=torch.float32)


def make_inputs(w: Workload, *, T: Optional[int] = None, H: Optional[int] = None,
                Hqk: Optional[int] = None, seed: Optional[int] = None,
                decay_stress: Optional[bool] = None) -> dict:
    """Draw one problem on the CPU.  Returns a dict of CPU tensors.

    q, k [B,T,Hqk,dk] and v [B,T,H,dv], a, b [B,T,H] are in ``w.dtype``;
    A_log, dt_bias [H], h0 [B,H,dk,dv], dO [B,T,H,dv] (in ``w.dtype``) and
    dHT [B,H,dk,dv] are fp32 except dO.  ``valid_len`` is int32 [B] or None.
    """
    T = w.T if T is None else T
    H = w.H if H is None else H
    Hqk = w.Hqk if Hqk is None else Hqk
    seed = w.seed if seed is None else seed
    stress = w.decay_stress if decay_stress is None else decay_stress
    gen = torch.Generator().manual_seed(seed)
    B, dk, dv = w.B, w.dk, w.dv
    out = {}
    out["q"] = _normal(gen, (B, T, Hqk, dk)).to(w.dtype)
    out["k"] = _normal(gen, (B, T, Hqk, dk)).to(w.dtype)
    out["v"] = _normal(gen, (B, T, H, dv)).to(w.dtype)
    out["a"] = _normal(gen, (B, T, H)).to(w.dtype)
    out["b"] = _normal(gen, (B, T, H)).to(w.dtype)
    out["A_log"] = torch.empty(H).uniform_(1.0, 16.0, generator=gen).log()
    if stress:
        out["dt_bias"] = -6.0 + 0.1 * _normal(gen, (H,))
    else:
        out["dt_bias"] = _normal(gen, (H,))
    out["h0"] = (w.h0_std * _normal(gen, (B, H, dk, dv))) if w.h0_std else None
    dO = _normal(gen, (B, T, H, dv))
    dHT = _normal(gen, (B, H, dk, dv)) if w.with_dHT else None
    if w.grad_scale == "numel":
        dO = dO / (max(dO.numel(), 1) ** 0.5)
        if dHT is not None:
            dHT = dHT / (dHT.numel() ** 0.5)
    out["dO"] = dO.to(w.dtype)
    out["dHT"] = dHT
    if w.valid_len is not None:
        out["valid_len"] = torch.tensor([min(int(x), T) for x in w.valid_len], dtype=torch.int32)
    else:
        out["valid_len"] = None
    return out


def make_varlen_inputs(w: Workload, lengths, *, seed: Optional[int] = None) -> dict:
    """A packed row of len(lengths) sequences: q, k, v, a, b, dO of one row (B = 1) of
    T = sum(lengths) tokens as in make_inputs, h0 and dHT [N,H,dk,dv] (one per sequence,
    when the workload has them) and cu_seqlens int32 [N + 1] (the running offsets)."""
    import dataclasses
    lengths = [int(x) for x in lengths]
    T = sum(lengths)
    w1 = dataclasses.replace(w, B=1, T=T, valid_len=None)
    out = make_inputs(w1, seed=seed)
    seed = w.seed if seed is None else seed
    gen = torch.Generator().manual_seed(seed + 7919)
    N = len(lengths)
    out["h0"] = (w.h0_std * _normal(gen, (N, w.H, w.dk, w.dv))) if w.h0_std else None
    if w.with_dHT:
        dHT = _normal(gen, (N, w.H, w.dk, w.dv))
        out["dHT"] = dHT / (dHT.numel() ** 0.5) if w.grad_scale == "numel" else dHT
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + x)
    out["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32)
    return out


def length_mix(total: int, n: int, *, seed: int = 0, min_len: int = 1) -> list:
    """n sequence lengths that sum to total, drawn around total / n (uniform cut points of
    the row, at least min_len each): a packed batch of training samples of mixed length."""
    gen = torch.Generator().manual_seed(seed)
    free = total - n * min_len
    if free < 0:
        raise ValueError("total too small for n sequences of min_len")
    cuts = sorted(torch.randint(0, free + 1, (n - 1,), generator=gen).tolist())
    edges = [0] + cuts + [free]
    return [edges[i + 1] - edges[i] + min_len for i in range(n)]


def to_numpy64(inputs: dict) -> dict:
    """The exact (already rounded) values as float64 numpy arrays, for the oracle."""
    res = {}
    for key, val in inputs.items():
        if val is None:
            res[key] = None
        elif key in ("valid_len", "cu_seqlens"):
            res[key] = val.numpy().astype("int32")
        else:
            res[key] = val.to(torch.float64).numpy()
    return res


def make_conv_inputs(B: int, T: int, C: int, K: int, dtype=torch.bfloat16, *, seed: int = 0,
                     halo: bool = True, bias: bool = True, T_stride: Optional[int] = None) -> dict:
    """Seeded inputs of the Conv1D + SiLU prologue, on the CPU: x, dy [B, T_stride, C] in
    `dtype` (T_stride >= T tokens per row, N(0, 1)), w [C, K] fp32 (N(0, 0.25)), bias [C]
    fp32 (N(0, 0.01)) or None, halo [B, K-1, C] in `dtype` (N(0, 1)) or None.  C is the
    channel count of the projected q, k, v the convolution runs over (2 Hqk dk + H dv)."""
    Ts = T if T_stride is None else T_stride
    gen = torch.Generator().manual_seed(seed)
    out = {"x": _normal(gen, (B, Ts, C)).to(dtype),
           "w": 0.5 * _normal(gen, (C, K)),
           "bias": 0.1 * _normal(gen, (C,)) if bias else None,
           "halo": _normal(gen, (B, K - 1, C)).to(dtype) if (halo and K > 1) else None,
           "dy": _normal(gen, (B, Ts, C)).to(dtype)}
    return out


def make_rmsnorm_inputs(shape, dtype=torch.bfloat16, *, seed: int = 0) -> dict:
    """Seeded inputs of the gated RMSNorm epilogue, on the CPU: o, z, dy of `shape`
    ([B, T, H, dv]) in `dtype`, N(0, 1); w [dv] fp32, 1 + N(0, 0.1^2)."""
    gen = torch.Generator().manual_seed(seed)
    return {"o": _normal(gen, shape).to(dtype), "z": _normal(gen, shape).to(dtype),
            "w": 1.0 + 0.1 * _normal(gen, (shape[-1],)), "dy": _normal(gen, shape).to(dtype)}
