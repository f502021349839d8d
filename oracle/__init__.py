"""fp64 CPU oracle for the Gated DeltaNet core -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
and imports nothing from it.  The arithmetic lives in ``gdn_oracle.c`` (plain C,
fp64, OpenMP over (batch, head)); this module compiles it with gcc and calls it
through ctypes on numpy float64 arrays.

Every function follows the definition written at the top of ``gdn_oracle.c``:
the gated delta rule named by "linear attention cp #1035" (section "What does
this PR do") and by the "Linear Attention CP 融合算子 PR #1114 测试报告"
(sections 4.1 and 5.2), and the affine segment summary H_out = M @ H_in + S with
its prefix merge from PR #1035 ("p2p" and "all_gather" modes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into liboracle.so (gcc, -O2, OpenMP) if stale."""
    with _lock:
        stale = force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
                   "-Wno-unused-function", _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("Hqk", ctypes.c_int64),
                ("H", ctypes.c_int64), ("dk", ctypes.c_int64), ("dv", ctypes.c_int64),
                ("l2norm", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("eps", ctypes.c_double), ("scale", ctypes.c_double)]


_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int32)
_P = ctypes.POINTER(_Problem)


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        for name, args in {
            "oracle_prologue": [_P, _D, _D, _D, _D, _D, _D, _I, _D, _D, _D, _D],
            "oracle_core_fwd": [_P, _D, _D, _D, _D, _D, _D, _I, _D, _D, ctypes.c_int],
            "oracle_core_bwd": [_P, _D, _D, _D, _D, _D, _D, _I, _D, _D, _D, _D, _D, _D, _D,
                                _D, ctypes.c_int],
            "oracle_fwd": [_P, _D, _D, _D, _D, _D, _D, _D, _D, _I, _D, _D, ctypes.c_int],
            "oracle_bwd": [_P, _D, _D, _D, _D, _D, _D, _D, _D, _I, _D, _D, _D, _D, _D, _D,
                           _D, _D, ctypes.c_int],
            "oracle_summary": [_P, _D, _D, _D, _D, _D, _D, _I, _D, _D, ctypes.c_int],
            "oracle_summary_bwd": [_P, _D, _D, _D, _D, _D, _D, _I, _D, _D, ctypes.c_int],
            "oracle_compose": [ctypes.c_int64] * 3 + [_D] * 6,
            "oracle_prefix": [ctypes.c_int64] * 4 + [_D] * 5,
            "oracle_prefix_bwd": [ctypes.c_int64] * 4 + [_D] * 5,
            "oracle_gate_param_bwd": [_P, _D, _D, _D, _D, _I, _D, _D, _D, _D, _D, _D],
        }.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return a


def _ptr(a):
    if a is None:
        return None
    if a.dtype == np.int32:
        return a.ctypes.data_as(_I)
    return a.ctypes.data_as(_D)


def _vl(valid_len):
    if valid_len is None:
        return None
    return np.ascontiguousarray(np.asarray(valid_len, dtype=np.int32))


def _problem(q_or_k, v, l2norm=True, eps=1e-6, scale=None):
    B, T, Hqk, dk = q_or_k.shape
    H, dv = v.shape[2], v.shape[3]
    if scale is None or scale <= 0:
        scale = 1.0 / float(np.sqrt(dk))
    return _Problem(B, T, Hqk, H, dk, dv, 1 if l2norm else 0, 0, float(eps), float(scale))


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: oracle rejected its arguments (code {rc})")


def prologue(q, k, a, b, A_log, dt_bias, valid_len=None, *, H=None, dv=1, l2norm=True,
             eps=1e-6, scale=None):
    """q_hat, k_hat [B,T,Hqk,dk], g, beta [B,T,H] (padded tokens: g = beta = 0)."""
    q, k, a, b = _f64(q), _f64(k), _f64(a), _f64(b)
    A_log, dt_bias = _f64(A_log), _f64(dt_bias)
    B, T, Hqk, dk = q.shape
    H = a.shape[2]
    p = _problem(q, np.zeros((B, T, H, dv)), l2norm, eps, scale)
    qh, kh = np.empty_like(q), np.empty_like(k)
    g, be = np.empty_like(a), np.empty_like(a)
    vl = _vl(valid_len)
    _check(_load().oracle_prologue(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(a), _ptr(b),
                                   _ptr(A_log), _ptr(dt_bias), _ptr(vl), _ptr(qh), _ptr(kh),
                                   _ptr(g), _ptr(be)), "prologue")
    return qh, kh, g, be


def core_fwd(qh, kh, v, g, beta, h0=None, valid_len=None, nthreads=0):
    """Recurrence over prepared q_hat, k_hat, g, beta: returns (o, h_T)."""
    qh, kh, v, g, beta, h0 = map(_f64, (qh, kh, v, g, beta, h0))
    p = _problem(qh, v, l2norm=False, scale=1.0)
    B, T, H, dv = v.shape
    o = np.empty((B, T, H, dv))
    hT = np.empty((B, H, p.dk, dv))
    vl = _vl(valid_len)
    _check(_load().oracle_core_fwd(ctypes.byref(p), _ptr(qh), _ptr(kh), _ptr(v), _ptr(g),
                                   _ptr(beta), _ptr(h0), _ptr(vl), _ptr(o), _ptr(hT),
                                   nthreads), "core_fwd")
    return o, hT


def core_bwd(qh, kh, v, g, beta, dO, dHT=None, h0=None, valid_len=None, nthreads=0):
    """Gradients of <dO,o> + <dHT,h_T> w.r.t. q_hat, k_hat (Q/K heads), v, g, beta, h0."""
    qh, kh, v, g, beta, h0, dO, dHT = map(_f64, (qh, kh, v, g, beta, h0, dO, dHT))
    p = _problem(qh, v, l2norm=False, scale=1.0)
    B, T, H, dv = v.shape
    dqh, dkh = np.empty_like(qh), np.empty_like(kh)
    dv_ = np.empty_like(v)
    dg, dbe = np.empty_like(g), np.empty_like(g)
    dH0 = np.empty((B, H, p.dk, dv))
    vl = _vl(valid_len)
    _check(_load().oracle_core_bwd(ctypes.byref(p), _ptr(qh), _ptr(kh), _ptr(v), _ptr(g),
                                   _ptr(beta), _ptr(h0), _ptr(vl), _ptr(dO), _ptr(dHT),
                                   _ptr(dqh), _ptr(dkh), _ptr(dv_), _ptr(dg), _ptr(dbe),
                                   _ptr(dH0), nthreads), "core_bwd")
    return dqh, dkh, dv_, dg, dbe, dH0


def fwd(q, k, v, a, b, A_log, dt_bias, h0=None, valid_len=None, *, l2norm=True, eps=1e-6,
        scale=None, nthreads=0):
    """GDN forward from raw inputs: returns (o [B,T,H,dv], h_T [B,H,dk,dv])."""
    q, k, v, a, b, A_log, dt_bias, h0 = map(_f64, (q, k, v, a, b, A_log, dt_bias, h0))
    p = _problem(q, v, l2norm, eps, scale)
    B, T, H, dv = v.shape
    o = np.empty((B, T, H, dv))
    hT = np.empty((B, H, p.dk, dv))
    vl = _vl(valid_len)
    _check(_load().oracle_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                              _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(vl), _ptr(o),
                              _ptr(hT), nthreads), "fwd")
    return o, hT


def bwd(q, k, v, a, b, A_log, dt_bias, dO, dHT=None, h0=None, valid_len=None, *, l2norm=True,
        eps=1e-6, scale=None, nthreads=0):
    """GDN backward from raw inputs: returns (dq, dk, dv, dg, dbeta, dH0)."""
    q, k, v, a, b, A_log, dt_bias, h0, dO, dHT = map(
        _f64, (q, k, v, a, b, A_log, dt_bias, h0, dO, dHT))
    p = _problem(q, v, l2norm, eps, scale)
    B, T, H, dv = v.shape
    dq, dk = np.empty_like(q), np.empty_like(k)
    dv_ = np.empty_like(v)
    dg, dbe = np.empty_like(a), np.empty_like(a)
    dH0 = np.empty((B, H, p.dk, dv))
    vl = _vl(valid_len)
    _check(_load().oracle_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                              _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(vl), _ptr(dO),
                              _ptr(dHT), _ptr(dq), _ptr(dk), _ptr(dv_), _ptr(dg), _ptr(dbe),
                              _ptr(dH0), nthreads), "bwd")
    return dq, dk, dv_, dg, dbe, dH0


def summary(k, v, a, b, A_log, dt_bias, valid_len=None, *, l2norm=True, eps=1e-6, nthreads=0):
    """Affine summary of the whole sequence: (M [B,H,dk,dk], S [B,H,dk,dv])."""
    k, v, a, b, A_log, dt_bias = map(_f64, (k, v, a, b, A_log, dt_bias))
    p = _problem(k, v, l2norm, eps, None)
    B, T, H, dv = v.shape
    M = np.empty((B, H, p.dk, p.dk))
    S = np.empty((B, H, p.dk, dv))
    vl = _vl(valid_len)
    _check(_load().oracle_summary(ctypes.byref(p), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                  _ptr(A_log), _ptr(dt_bias), _ptr(vl), _ptr(M), _ptr(S),
                                  nthreads), "summary")
    return M, S


def summary_bwd(q, k, a, b, A_log, dt_bias, dO, valid_len=None, *, l2norm=True, eps=1e-6,
                scale=None, nthreads=0):
    """Gradient summary D = d<dO, o>/dH_in  [B,H,dk,dv]."""
    q, k, a, b, A_log, dt_bias, dO = map(_f64, (q, k, a, b, A_log, dt_bias, dO))
    B, T, H, dv = dO.shape
    p = _problem(q, dO, l2norm, eps, scale)
    D = np.empty((B, H, p.dk, dv))
    vl = _vl(valid_len)
    _check(_load().oracle_summary_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(a), _ptr(b),
                                      _ptr(A_log), _ptr(dt_bias), _ptr(vl), _ptr(dO), _ptr(D),
                                      nthreads), "summary_bwd")
    return D


def gate_param_bwd(a, b, A_log, dt_bias, dg, dbeta, valid_len=None):
    """Gradients of the gate parameters from dg, dbeta [B,T,H]: (da, db [B,T,H],
    dA_log, ddt_bias [H]) through g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)."""
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    dg, dbeta = _f64(dg), _f64(dbeta)
    B, T, H = a.shape
    p = _problem(np.zeros((B, T, H, 1)), np.zeros((B, T, H, 1)))
    da, db = np.empty_like(a), np.empty_like(a)
    dA, ddt = np.empty(H), np.empty(H)
    _check(_load().oracle_gate_param_bwd(ctypes.byref(p), _ptr(a), _ptr(b), _ptr(A_log),
                                         _ptr(dt_bias), _ptr(_vl(valid_len)), _ptr(dg),
                                         _ptr(dbeta), _ptr(da), _ptr(db), _ptr(dA), _ptr(ddt)),
           "gate_param_bwd")
    return da, db, dA, ddt


def compose(M2, S2, M1, S1):
    """(M2 M1, M2 S1 + S2), batched over the leading dimensions."""
    M2, S2, M1, S1 = map(_f64, (M2, S2, M1, S1))
    dk, dv = S1.shape[-2], S1.shape[-1]
    n = int(np.prod(S1.shape[:-2])) if S1.ndim > 2 else 1
    M = np.empty_like(M1)
    S = np.empty_like(S1)
    _check(_load().oracle_compose(n, dk, dv, _ptr(M2), _ptr(S2), _ptr(M1), _ptr(S1), _ptr(M),
                                  _ptr(S)), "compose")
    return M, S


def prefix(M, S, h0=None):
    """Exclusive prefix over segments: M [P,...,dk,dk], S [P,...,dk,dv] -> (H_in, H_out)."""
    M, S, h0 = map(_f64, (M, S, h0))
    P = S.shape[0]
    dk, dv = S.shape[-2], S.shape[-1]
    n = int(np.prod(S.shape[1:-2])) if S.ndim > 3 else 1
    Hin = np.empty_like(S)
    Hout = np.empty(S.shape[1:])
    _check(_load().oracle_prefix(n, P, dk, dv, _ptr(M), _ptr(S), _ptr(h0), _ptr(Hin),
                                 _ptr(Hout)), "prefix")
    return Hin, Hout


def prefix_bwd(M, D, dHT=None):
    """Reverse exclusive prefix of state gradients -> (dH_out [P,...], dH0 [...])."""
    M, D, dHT = map(_f64, (M, D, dHT))
    P = D.shape[0]
    dk, dv = D.shape[-2], D.shape[-1]
    n = int(np.prod(D.shape[1:-2])) if D.ndim > 3 else 1
    dHout = np.empty_like(D)
    dH0 = np.empty(D.shape[1:])
    _check(_load().oracle_prefix_bwd(n, P, dk, dv, _ptr(M), _ptr(D), _ptr(dHT), _ptr(dHout),
                                     _ptr(dH0)), "prefix_bwd")
    return dHout, dH0


# The causal depthwise Conv1D + SiLU prologue (numpy, fp64): see oracle/conv.py.
from .conv import conv_silu_bwd, conv_silu_fwd  # noqa: E402,F401
# The gated RMSNorm epilogue on o (numpy, fp64): see oracle/rmsnorm.py.
from .rmsnorm import rmsnorm_gated_bwd, rmsnorm_gated_fwd  # noqa: E402,F401


# ------------------------------------------------------------ packed variable-length rows
#
# The test report of "Linear Attention CP 融合算子 PR #1114" (section 5.2) covers
# variable-length training samples through trailing padding of each batch row.  Packing
# several samples into one row generalises it: sequence i is the tokens
# cu_seqlens[i] .. cu_seqlens[i+1]-1 of the row and runs the gated delta rule on its own,
# from its own initial state h0[i] (zero when h0 is None), exactly as if it were a batch
# row of its own; nothing flows across a boundary.  These functions are that definition:
# one call of the single-sequence oracle above per packed sequence.


def seq_bounds(cu_seqlens, T):
    """[(start, end)] of every packed sequence; cu_seqlens: N + 1 non-decreasing offsets
    from 0 to T."""
    cu = np.asarray(cu_seqlens, dtype=np.int64).ravel()
    if cu.size < 1 or cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must run from 0 to T without decreasing")
    return [(int(cu[i]), int(cu[i + 1])) for i in range(cu.size - 1)]


def _one(x, i):
    return None if x is None else x[i:i + 1]


def core_fwd_varlen(qh, kh, v, g, beta, cu_seqlens, h0=None, nthreads=0):
    """Packed rows (B = 1) over prepared q_hat, k_hat, g, beta: (o [1,T,H,dv],
    h_T [N,H,dk,dv]) with h0 [N,H,dk,dv] or None."""
    qh, kh, v, g, beta, h0 = map(_f64, (qh, kh, v, g, beta, h0))
    _, T, H, dv = v.shape
    bounds = seq_bounds(cu_seqlens, T)
    o = np.empty_like(v)
    hT = np.empty((len(bounds), H, qh.shape[3], dv))
    for i, (s, e) in enumerate(bounds):
        o[:, s:e], hT[i:i + 1] = core_fwd(qh[:, s:e], kh[:, s:e], v[:, s:e], g[:, s:e],
                                          beta[:, s:e], _one(h0, i), nthreads=nthreads)
    return o, hT


def fwd_varlen(q, k, v, a, b, A_log, dt_bias, cu_seqlens, h0=None, *, l2norm=True, eps=1e-6,
               scale=None, nthreads=0):
    """Packed rows (B = 1) from raw inputs: (o [1,T,H,dv], h_T [N,H,dk,dv])."""
    q, k, v, a, b, A_log, dt_bias, h0 = map(_f64, (q, k, v, a, b, A_log, dt_bias, h0))
    _, T, H, dv = v.shape
    bounds = seq_bounds(cu_seqlens, T)
    o = np.empty_like(v)
    hT = np.empty((len(bounds), H, q.shape[3], dv))
    for i, (s, e) in enumerate(bounds):
        o[:, s:e], hT[i:i + 1] = fwd(q[:, s:e], k[:, s:e], v[:, s:e], a[:, s:e], b[:, s:e],
                                     A_log, dt_bias, h0=_one(h0, i), l2norm=l2norm, eps=eps,
                                     scale=scale, nthreads=nthreads)
    return o, hT


def bwd_varlen(q, k, v, a, b, A_log, dt_bias, cu_seqlens, dO, dHT=None, h0=None, *,
               l2norm=True, eps=1e-6, scale=None, nthreads=0):
    """Gradients of sum_t <dO_t, o_t> + sum_i <dHT[i], h_T[i]> over packed rows:
    (dq, dk [1,T,Hqk,dk], dv [1,T,H,dv], dg, dbeta [1,T,H], dH0 [N,H,dk,dv])."""
    q, k, v, a, b, A_log, dt_bias, h0, dO, dHT = map(
        _f64, (q, k, v, a, b, A_log, dt_bias, h0, dO, dHT))
    _, T, H, dv = v.shape
    bounds = seq_bounds(cu_seqlens, T)
    dq, dk, dv_ = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    dg, dbe = np.empty_like(a), np.empty_like(a)
    dH0 = np.empty((len(bounds), H, q.shape[3], dv))
    for i, (s, e) in enumerate(bounds):
        r = bwd(q[:, s:e], k[:, s:e], v[:, s:e], a[:, s:e], b[:, s:e], A_log, dt_bias,
                dO[:, s:e], _one(dHT, i), h0=_one(h0, i), l2norm=l2norm, eps=eps, scale=scale,
                nthreads=nthreads)
        dq[:, s:e], dk[:, s:e], dv_[:, s:e], dg[:, s:e], dbe[:, s:e], dH0[i:i + 1] = r
    return dq, dk, dv_, dg, dbe, dH0
