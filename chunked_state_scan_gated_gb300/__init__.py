"""GB300 Gated DeltaNet core: Python binding of the C ABI in include/gdn.h.

Argument marshalling only.  Every step of the computation runs in the CUDA
library ``libgdn.so`` (hand-written sm_103a kernels); PyTorch provides device
memory and the stream.  If the library is missing the calls raise: there is no
CPU fallback.

The functions keep the C names (``gdn_fwd``, ``gdn_bwd``, ``gdn_summary``,
``gdn_summary_bwd``, ``gdn_compose``, ``gdn_prefix_compose``,
``gdn_prefix_compose_bwd``, ``gdn_apply_state``, ``gdn_apply_state_bwd``,
``gdn_gate_param_bwd``, ``gdn_query_support``, ``gdn_resolved_segments``, ``gdn_workspace_size``,
``gdn_check_device_status``) and
take torch tensors in the token-major layouts of the header: q, k
[B,T,Hqk,dk]; v [B,T,H,dv]; a, b [B,T,H]; A_log, dt_bias [H] fp32; states
[B,H,dk,dv] fp32.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE, GDN_ERR_CUDA, \
    GDN_ERR_DEVICE_TIMEOUT = range(6)
GDN_FP32, GDN_BF16 = 0, 1
GDN_OP_FWD, GDN_OP_BWD, GDN_OP_SUMMARY, GDN_OP_SUMMARY_BWD, GDN_OP_FWD_CTX, GDN_OP_BWD_CTX = \
    range(6)

# Every symbol include/gdn.h declares (checked by the CPU test suite).
EXPORTS = (
    "gdn_status_string", "gdn_abi_version", "gdn_problem_init", "gdn_query_support",
    "gdn_resolved_segments", "gdn_workspace_size", "gdn_fwd", "gdn_bwd", "gdn_gate_param_bwd", "gdn_summary", "gdn_summary_bwd",
    "gdn_compose", "gdn_prefix_compose", "gdn_prefix_compose_bwd", "gdn_apply_state",
    "gdn_apply_state_bwd", "gdn_check_device_status", "gdn_kernel_info", "gdn_fwd_kernel",
    "gdn_bwd_kernel", "gdn_fwd_noalloc", "gdn_noalloc_check_device_status", "gdn_ctx_size",
    "gdn_fwd_ctx", "gdn_bwd_ctx",
    "gdn_fwd_ctx_kernel", "gdn_bwd_ctx_kernel", "gdn_conv_silu_fwd", "gdn_fwd_conv",
    "gdn_conv_silu_bwd_workspace_size", "gdn_conv_silu_bwd", "gdn_rmsnorm_gated_fwd",
    "gdn_rmsnorm_gated_bwd_workspace_size", "gdn_rmsnorm_gated_bwd",
    "gdn_varlen_workspace_size", "gdn_fwd_varlen", "gdn_bwd_varlen",
    "gdn_varlen_check_device_status",
)


class GDNError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)}")


class Problem(ctypes.Structure):
    """Mirror of ``gdn_problem`` (include/gdn.h)."""

    _fields_ = [("dtype", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("B", ctypes.c_int64), ("T", ctypes.c_int64), ("T_stride", ctypes.c_int64),
                ("Hqk", ctypes.c_int64), ("H", ctypes.c_int64), ("dk", ctypes.c_int64),
                ("dv", ctypes.c_int64), ("l2norm_qk", ctypes.c_int32), ("l2_eps", ctypes.c_float),
                ("scale", ctypes.c_float), ("segments", ctypes.c_int32)]


class ConvProblem(ctypes.Structure):
    """Mirror of ``gdn_conv_problem`` (include/gdn.h)."""

    _fields_ = [("dtype", ctypes.c_int32), ("K", ctypes.c_int32), ("B", ctypes.c_int64),
                ("T", ctypes.c_int64), ("C", ctypes.c_int64), ("T_stride", ctypes.c_int64)]


class ConvQkv(ctypes.Structure):
    """Mirror of ``gdn_conv_qkv`` (include/gdn.h)."""

    _fields_ = [("K", ctypes.c_int32), ("x", ctypes.c_void_p * 3), ("w", ctypes.c_void_p * 3),
                ("bias", ctypes.c_void_p * 3), ("halo", ctypes.c_void_p * 3),
                ("y", ctypes.c_void_p * 3)]


class RmsNormProblem(ctypes.Structure):
    """Mirror of ``gdn_rmsnorm_problem`` (include/gdn.h)."""

    _fields_ = [("dtype", ctypes.c_int32), ("D", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("eps", ctypes.c_float)]


_lock = threading.Lock()
_lib = None
_VP = ctypes.c_void_p
_PP = ctypes.POINTER(Problem)
_I64 = ctypes.c_int64
_CPP = ctypes.POINTER(ConvProblem)
_RPP = ctypes.POINTER(RmsNormProblem)


def load_library(path: str | None = None):
    """Load libgdn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"GDN CUDA library not found at {p}; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(p)
        sig = {
            "gdn_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "gdn_abi_version": ([], ctypes.c_int32),
            "gdn_problem_init": ([_PP], None),
            "gdn_query_support": ([_PP], ctypes.c_int),
            "gdn_workspace_size": ([_PP, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)],
                                   ctypes.c_int),
            "gdn_resolved_segments": ([_PP, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
                                      ctypes.c_int),
            "gdn_gate_param_bwd": ([_PP] + [_VP] * 11 + [_VP], ctypes.c_int),
            "gdn_fwd": ([_PP] + [_VP] * 12 + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_apply_state": ([_PP] + [_VP] * 12 + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_bwd": ([_PP] + [_VP] * 18 + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_apply_state_bwd": ([_PP] + [_VP] * 18 + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_summary": ([_PP] + [_VP] * 10 + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_summary_bwd": ([_PP] + [_VP] * 10 + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_compose": ([_I64] * 3 + [_VP] * 7, ctypes.c_int),
            "gdn_prefix_compose": ([_I64] * 4 + [_VP] * 6, ctypes.c_int),
            "gdn_prefix_compose_bwd": ([_I64] * 4 + [_VP] * 6, ctypes.c_int),
            "gdn_check_device_status": ([_VP, _VP], ctypes.c_int),
            "gdn_noalloc_check_device_status": ([_VP], ctypes.c_int),
            "gdn_kernel_info": ([_PP, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.POINTER(ctypes.c_int32),
                                 ctypes.POINTER(ctypes.c_char_p)], ctypes.c_int),
            "gdn_fwd_kernel": ([_PP, ctypes.c_int32] + [_VP] * 12 + [ctypes.c_size_t, _VP],
                               ctypes.c_int),
            "gdn_bwd_kernel": ([_PP, ctypes.c_int32] + [_VP] * 18 + [ctypes.c_size_t, _VP],
                               ctypes.c_int),
            "gdn_fwd_noalloc": ([_PP] + [_VP] * 12, ctypes.c_int),
            "gdn_ctx_size": ([_PP, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
            "gdn_fwd_ctx": ([_PP] + [_VP] * 12 + [ctypes.c_size_t, _VP, ctypes.c_size_t, _VP],
                            ctypes.c_int),
            "gdn_bwd_ctx": ([_PP] + [_VP] * 8 + [ctypes.c_size_t] + [_VP] * 10
                            + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_fwd_ctx_kernel": ([_PP, ctypes.c_int32] + [_VP] * 12
                                   + [ctypes.c_size_t, _VP, ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_bwd_ctx_kernel": ([_PP, ctypes.c_int32] + [_VP] * 8 + [ctypes.c_size_t]
                                   + [_VP] * 10 + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_conv_silu_fwd": ([_CPP] + [_VP] * 6, ctypes.c_int),
            "gdn_fwd_conv": ([_PP, ctypes.POINTER(ConvQkv)] + [_VP] * 8
                             + [_VP, ctypes.c_size_t, _VP, ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_conv_silu_bwd_workspace_size": ([_CPP, ctypes.POINTER(ctypes.c_size_t)],
                                                 ctypes.c_int),
            "gdn_conv_silu_bwd": ([_CPP] + [_VP] * 10 + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_rmsnorm_gated_fwd": ([_RPP] + [_VP] * 5, ctypes.c_int),
            "gdn_rmsnorm_gated_bwd_workspace_size": ([_RPP, ctypes.POINTER(ctypes.c_size_t)],
                                                     ctypes.c_int),
            "gdn_rmsnorm_gated_bwd": ([_RPP] + [_VP] * 8 + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_varlen_workspace_size": ([_PP, _VP, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
            "gdn_fwd_varlen": ([_PP, _VP, _VP, ctypes.c_int32] + [_VP] * 11
                               + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_bwd_varlen": ([_PP, _VP, _VP, ctypes.c_int32] + [_VP] * 17
                               + [ctypes.c_size_t, _VP], ctypes.c_int),
            "gdn_varlen_check_device_status": ([_VP, _PP, _VP, ctypes.c_int32, ctypes.c_int32,
                                                _VP], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().gdn_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != GDN_OK:
        raise GDNError(fn, status)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("GDN tensors must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("GDN tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return GDN_BF16
    if dt == torch.float32:
        return GDN_FP32
    raise ValueError(f"unsupported I/O dtype {dt}")


def make_problem(q_or_k: torch.Tensor, v_or_dO: torch.Tensor, *, T: int | None = None,
                 T_stride: int = 0, segments: int = 0, l2norm: bool = True, eps: float = 1e-6,
                 scale: float = 0.0) -> Problem:
    B, Tq, Hqk, dk = q_or_k.shape
    H, dv = v_or_dO.shape[2], v_or_dO.shape[3]
    p = Problem()
    load_library().gdn_problem_init(ctypes.byref(p))
    p.dtype = _dtype_code(q_or_k.dtype)
    p.B, p.T, p.T_stride = B, (Tq if T is None else T), T_stride
    p.Hqk, p.H, p.dk, p.dv = Hqk, H, dk, dv
    p.l2norm_qk = 1 if l2norm else 0
    p.l2_eps = eps
    p.scale = scale
    p.segments = segments
    return p


def gdn_query_support(problem: Problem) -> int:
    return load_library().gdn_query_support(ctypes.byref(problem))


def gdn_workspace_size(problem: Problem, op: int) -> int:
    n = ctypes.c_size_t(0)
    _check("gdn_workspace_size",
           load_library().gdn_workspace_size(ctypes.byref(problem), op, ctypes.byref(n)))
    return n.value


def gdn_resolved_segments(problem: Problem, op: int) -> int:
    """Segments the call of `op` splits T into (problem.segments, or the automatic choice)."""
    n = ctypes.c_int32(0)
    _check("gdn_resolved_segments",
           load_library().gdn_resolved_segments(ctypes.byref(problem), op, ctypes.byref(n)))
    return n.value


def workspace(problem: Problem, op: int, device=None) -> torch.Tensor:
    """A caller-owned workspace buffer for `op` (uint8, 256-byte aligned by torch)."""
    n = gdn_workspace_size(problem, op)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _ws(problem, op, ws, device):
    if ws is None:
        ws = workspace(problem, op, device)
    return ws


def gdn_fwd(q, k, v, a, b, A_log, dt_bias, h0=None, valid_len=None, *, segments=0,
            l2norm=True, eps=1e-6, scale=0.0, o=None, hT=None, want_hT=True, ws=None,
            stream=None, problem=None):
    """Forward: returns (o [B,T,H,dv] in q.dtype, hT [B,H,dk,dv] fp32 or None)."""
    p = problem or make_problem(q, v, segments=segments, l2norm=l2norm, eps=eps, scale=scale)
    B, T, H, dv = v.shape
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_hT:
        hT = torch.empty((B, H, q.shape[3], dv), dtype=torch.float32, device=q.device)
    ws = _ws(p, GDN_OP_FWD, ws, q.device)
    _check("gdn_fwd", load_library().gdn_fwd(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
        _ptr(dt_bias), _ptr(h0), _ptr(valid_len), _ptr(o), _ptr(hT), _ptr(ws), ws.numel(),
        _stream(stream)))
    return o, hT


GDN_NOALLOC_SCRATCH_BYTES = 64 << 20


def gdn_fwd_noalloc(q, k, v, a, b, A_log, dt_bias, h0=None, valid_len=None, *, o, hT=None,
                    segments=0, l2norm=True, eps=1e-6, scale=0.0, stream=None, problem=None):
    """Forward into caller-given outputs with no workspace: the library's static
    device scratch (GDN_NOALLOC_SCRATCH_BYTES) is used instead.  For callers that
    cannot allocate device memory; o (and hT if wanted) must be preallocated."""
    p = problem or make_problem(q, v, segments=segments, l2norm=l2norm, eps=eps, scale=scale)
    _check("gdn_fwd_noalloc", load_library().gdn_fwd_noalloc(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
        _ptr(dt_bias), _ptr(h0), _ptr(valid_len), _ptr(o), _ptr(hT), _stream(stream)))
    return o, hT


def gdn_apply_state(q, k, v, a, b, A_log, dt_bias, Hin, valid_len=None, **kw):
    """Forward of a segment from its incoming state Hin (required)."""
    if Hin is None:
        raise ValueError("gdn_apply_state needs Hin")
    p = kw.pop("problem", None) or make_problem(q, v, segments=kw.pop("segments", 0),
                                                 l2norm=kw.pop("l2norm", True),
                                                 eps=kw.pop("eps", 1e-6),
                                                 scale=kw.pop("scale", 0.0))
    B, T, H, dv = v.shape
    o = kw.pop("o", None)
    hT = kw.pop("hT", None)
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and kw.pop("want_hT", True):
        hT = torch.empty((B, H, q.shape[3], dv), dtype=torch.float32, device=q.device)
    ws = _ws(p, GDN_OP_FWD, kw.pop("ws", None), q.device)
    _check("gdn_apply_state", load_library().gdn_apply_state(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
        _ptr(dt_bias), _ptr(Hin), _ptr(valid_len), _ptr(o), _ptr(hT), _ptr(ws), ws.numel(),
        _stream(kw.pop("stream", None))))
    return o, hT


def _bwd_common(name, q, k, v, a, b, A_log, dt_bias, h0, valid_len, dO, dHT, want_dH0, kw):
    p = kw.pop("problem", None) or make_problem(q, v, segments=kw.pop("segments", 0),
                                                 l2norm=kw.pop("l2norm", True),
                                                 eps=kw.pop("eps", 1e-6),
                                                 scale=kw.pop("scale", 0.0))
    B, T, H, dv = v.shape
    def out(name, make):
        t = kw.pop(name, None)
        return make() if t is None else t

    dq = out("dq", lambda: torch.empty_like(q))
    dk = out("dk", lambda: torch.empty_like(k))
    dv_ = out("dv", lambda: torch.empty_like(v))
    dg = out("dg", lambda: torch.empty((B, T, H), dtype=torch.float32, device=q.device))
    dbeta = out("dbeta", lambda: torch.empty((B, T, H), dtype=torch.float32, device=q.device))
    dH0 = kw.pop("dH0", None)
    if dH0 is None and want_dH0:
        dH0 = torch.empty((B, H, q.shape[3], dv), dtype=torch.float32, device=q.device)
    ws = _ws(p, GDN_OP_BWD, kw.pop("ws", None), q.device)
    fn = getattr(load_library(), name)
    _check(name, fn(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
                    _ptr(dt_bias), _ptr(h0), _ptr(valid_len), _ptr(dO), _ptr(dHT), _ptr(dq),
                    _ptr(dk), _ptr(dv_), _ptr(dg), _ptr(dbeta), _ptr(dH0), _ptr(ws), ws.numel(),
                    _stream(kw.pop("stream", None))))
    return dq, dk, dv_, dg, dbeta, dH0


def gdn_bwd(q, k, v, a, b, A_log, dt_bias, dO, dHT=None, h0=None, valid_len=None, *,
            want_dH0=True, **kw):
    """Backward: returns (dq, dk, dv, dg, dbeta, dH0)."""
    return _bwd_common("gdn_bwd", q, k, v, a, b, A_log, dt_bias, h0, valid_len, dO, dHT,
                       want_dH0, kw)


def gdn_apply_state_bwd(q, k, v, a, b, A_log, dt_bias, Hin, dO, dHout=None, valid_len=None,
                        **kw):
    """Backward of a segment run from Hin: (dq, dk, dv, dg, dbeta, dHin)."""
    if Hin is None:
        raise ValueError("gdn_apply_state_bwd needs Hin")
    return _bwd_common("gdn_apply_state_bwd", q, k, v, a, b, A_log, dt_bias, Hin, valid_len, dO,
                       dHout, True, kw)


def gdn_ctx_size(problem: Problem) -> int:
    """Bytes of the forward context of gdn_fwd_ctx / gdn_bwd_ctx."""
    n = ctypes.c_size_t(0)
    _check("gdn_ctx_size", load_library().gdn_ctx_size(ctypes.byref(problem), ctypes.byref(n)))
    return n.value


def ctx_buffer(problem: Problem, device=None) -> torch.Tensor:
    """A caller-owned forward context buffer (uint8)."""
    return torch.empty(gdn_ctx_size(problem), dtype=torch.uint8, device=device or "cuda")


def gdn_fwd_ctx(q, k, v, a, b, A_log, dt_bias, h0=None, valid_len=None, *, ctx=None,
                segments=0, l2norm=True, eps=1e-6, scale=0.0, o=None, hT=None, want_hT=True,
                ws=None, stream=None, problem=None):
    """Forward that also keeps the segment transitions and start states:
    returns (o, hT, ctx) with ctx for gdn_bwd_ctx."""
    p = problem or make_problem(q, v, segments=segments, l2norm=l2norm, eps=eps, scale=scale)
    B, T, H, dv = v.shape
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_hT:
        hT = torch.empty((B, H, q.shape[3], dv), dtype=torch.float32, device=q.device)
    ctx = ctx if ctx is not None else ctx_buffer(p, q.device)
    ws = _ws(p, GDN_OP_FWD_CTX, ws, q.device)
    _check("gdn_fwd_ctx", load_library().gdn_fwd_ctx(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
        _ptr(dt_bias), _ptr(h0), _ptr(valid_len), _ptr(o), _ptr(hT), _ptr(ctx), ctx.numel(),
        _ptr(ws), ws.numel(), _stream(stream)))
    return o, hT, ctx


def gdn_bwd_ctx(q, k, v, a, b, A_log, dt_bias, ctx, dO, dHT=None, valid_len=None, *,
                want_dH0=True, **kw):
    """Backward from a gdn_fwd_ctx context: returns (dq, dk, dv, dg, dbeta, dH0)."""
    p = kw.pop("problem", None) or make_problem(q, v, segments=kw.pop("segments", 0),
                                                 l2norm=kw.pop("l2norm", True),
                                                 eps=kw.pop("eps", 1e-6),
                                                 scale=kw.pop("scale", 0.0))
    B, T, H, dv = v.shape
    dq = kw.pop("dq", None)
    dq = torch.empty_like(q) if dq is None else dq
    dk = kw.pop("dk", None)
    dk = torch.empty_like(k) if dk is None else dk
    dv_ = kw.pop("dv", None)
    dv_ = torch.empty_like(v) if dv_ is None else dv_
    dg = kw.pop("dg", None)
    dg = torch.empty((B, T, H), dtype=torch.float32, device=q.device) if dg is None else dg
    dbeta = kw.pop("dbeta", None)
    dbeta = torch.empty((B, T, H), dtype=torch.float32, device=q.device) if dbeta is None else dbeta
    dH0 = kw.pop("dH0", None)
    if dH0 is None and want_dH0:
        dH0 = torch.empty((B, H, q.shape[3], dv), dtype=torch.float32, device=q.device)
    ws = _ws(p, GDN_OP_BWD_CTX, kw.pop("ws", None), q.device)
    _check("gdn_bwd_ctx", load_library().gdn_bwd_ctx(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
        _ptr(dt_bias), _ptr(ctx), ctx.numel(), _ptr(valid_len), _ptr(dO), _ptr(dHT), _ptr(dq),
        _ptr(dk), _ptr(dv_), _ptr(dg), _ptr(dbeta), _ptr(dH0), _ptr(ws), ws.numel(),
        _stream(kw.pop("stream", None))))
    if kw:
        raise TypeError(f"unexpected arguments {sorted(kw)}")
    return dq, dk, dv_, dg, dbeta, dH0


def gdn_gate_param_bwd(a, b, A_log, dt_bias, dg, dbeta, valid_len=None, *, da=None, db=None,
                       dA_log=None, ddt_bias=None, stream=None, problem=None):
    """Gate-parameter gradients from dg, dbeta: (da, db [B,T,H] fp32, dA_log, ddt_bias [H] fp32)."""
    B, T, H = a.shape
    if problem is None:
        d = 128 if a.dtype == torch.bfloat16 else 16
        problem = Problem()
        load_library().gdn_problem_init(ctypes.byref(problem))
        problem.dtype = _dtype_code(a.dtype)
        problem.B, problem.T, problem.Hqk, problem.H, problem.dk, problem.dv = B, T, H, H, d, d
    f32 = dict(dtype=torch.float32, device=a.device)
    da = da if da is not None else torch.empty((B, T, H), **f32)
    db = db if db is not None else torch.empty((B, T, H), **f32)
    dA_log = dA_log if dA_log is not None else torch.empty((H,), **f32)
    ddt_bias = ddt_bias if ddt_bias is not None else torch.empty((H,), **f32)
    _check("gdn_gate_param_bwd", load_library().gdn_gate_param_bwd(
        ctypes.byref(problem), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(valid_len),
        _ptr(dg), _ptr(dbeta), _ptr(da), _ptr(db), _ptr(dA_log), _ptr(ddt_bias),
        _stream(stream)))
    return da, db, dA_log, ddt_bias


def gdn_summary(k, v, a, b, A_log, dt_bias, valid_len=None, *, l2norm=True, eps=1e-6, M=None,
                S=None, ws=None, stream=None, problem=None):
    """Segment summary (M [B,H,dk,dk], S [B,H,dk,dv]) fp32."""
    p = problem or make_problem(k, v, l2norm=l2norm, eps=eps)
    B, T, H, dv = v.shape
    dk = k.shape[3]
    M = M if M is not None else torch.empty((B, H, dk, dk), dtype=torch.float32, device=k.device)
    S = S if S is not None else torch.empty((B, H, dk, dv), dtype=torch.float32, device=k.device)
    ws = _ws(p, GDN_OP_SUMMARY, ws, k.device)
    _check("gdn_summary", load_library().gdn_summary(
        ctypes.byref(p), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
        _ptr(valid_len), _ptr(M), _ptr(S), _ptr(ws), ws.numel(), _stream(stream)))
    return M, S


def gdn_summary_bwd(q, k, a, b, A_log, dt_bias, dO, valid_len=None, *, l2norm=True, eps=1e-6,
                    scale=0.0, D=None, ws=None, stream=None, problem=None):
    """Gradient summary D = d<dO, o>/dH_in [B,H,dk,dv] fp32."""
    p = problem or make_problem(q, dO, l2norm=l2norm, eps=eps, scale=scale)
    B, T, H, dv = dO.shape
    D = D if D is not None else torch.empty((B, H, q.shape[3], dv), dtype=torch.float32,
                                            device=q.device)
    ws = _ws(p, GDN_OP_SUMMARY_BWD, ws, q.device)
    _check("gdn_summary_bwd", load_library().gdn_summary_bwd(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
        _ptr(valid_len), _ptr(dO), _ptr(D), _ptr(ws), ws.numel(), _stream(stream)))
    return D


def gdn_compose(M2, S2, M1, S1, *, M=None, S=None, stream=None):
    """(M2 M1, M2 S1 + S2), batched over the leading dims."""
    dk, dv = S1.shape[-2], S1.shape[-1]
    n = S1.numel() // (dk * dv)
    M = M if M is not None else torch.empty_like(M1)
    S = S if S is not None else torch.empty_like(S1)
    _check("gdn_compose", load_library().gdn_compose(n, dk, dv, _ptr(M2), _ptr(S2), _ptr(M1),
                                                     _ptr(S1), _ptr(M), _ptr(S),
                                                     _stream(stream)))
    return M, S


def gdn_prefix_compose(M, S, h0=None, *, want_Hout=True, Hin=None, Hout=None, stream=None):
    """Exclusive prefix over the leading (segment) dim -> (Hin [P,...], Hout [...])."""
    P = S.shape[0]
    dk, dv = S.shape[-2], S.shape[-1]
    n = S.numel() // (P * dk * dv) if P else 0
    Hin = Hin if Hin is not None else torch.empty_like(S)
    if Hout is None and want_Hout:
        Hout = torch.empty(S.shape[1:], dtype=torch.float32, device=S.device)
    _check("gdn_prefix_compose", load_library().gdn_prefix_compose(
        n, P, dk, dv, _ptr(M), _ptr(S), _ptr(h0), _ptr(Hin), _ptr(Hout), _stream(stream)))
    return Hin, Hout


def gdn_prefix_compose_bwd(M, D, dHT=None, *, want_dH0=True, dHout=None, dH0=None, stream=None):
    """Reverse exclusive prefix of state gradients -> (dHout [P,...], dH0 [...])."""
    P = D.shape[0]
    dk, dv = D.shape[-2], D.shape[-1]
    n = D.numel() // (P * dk * dv) if P else 0
    dHout = dHout if dHout is not None else torch.empty_like(D)
    if dH0 is None and want_dH0:
        dH0 = torch.empty(D.shape[1:], dtype=torch.float32, device=D.device)
    _check("gdn_prefix_compose_bwd", load_library().gdn_prefix_compose_bwd(
        n, P, dk, dv, _ptr(M), _ptr(D), _ptr(dHT), _ptr(dHout), _ptr(dH0), _stream(stream)))
    return dHout, dH0


def gdn_kernel_info(problem: Problem, op: int):
    """Names of the kernels `op` (GDN_OP_FWD / GDN_OP_BWD) launches, in order."""
    lib = load_library()
    count = ctypes.c_int32(0)
    _check("gdn_kernel_info", lib.gdn_kernel_info(ctypes.byref(problem), op, -1,
                                                  ctypes.byref(count), None))
    names = []
    for i in range(count.value):
        nm = ctypes.c_char_p()
        _check("gdn_kernel_info", lib.gdn_kernel_info(ctypes.byref(problem), op, i, None,
                                                      ctypes.byref(nm)))
        names.append(nm.value.decode())
    return names


def gdn_fwd_kernel(index, q, k, v, a, b, A_log, dt_bias, h0, valid_len, o, hT, ws, *,
                   problem, stream=None):
    """Launch only kernel `index` of gdn_fwd (after a full gdn_fwd on the same workspace)."""
    _check("gdn_fwd_kernel", load_library().gdn_fwd_kernel(
        ctypes.byref(problem), index, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
        _ptr(dt_bias), _ptr(h0), _ptr(valid_len), _ptr(o), _ptr(hT), _ptr(ws), ws.numel(),
        _stream(stream)))


def gdn_bwd_kernel(index, q, k, v, a, b, A_log, dt_bias, h0, valid_len, dO, dHT, dq, dk, dv,
                   dg, dbeta, dH0, ws, *, problem, stream=None):
    """Launch only kernel `index` of gdn_bwd (after a full gdn_bwd on the same workspace)."""
    _check("gdn_bwd_kernel", load_library().gdn_bwd_kernel(
        ctypes.byref(problem), index, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
        _ptr(dt_bias), _ptr(h0), _ptr(valid_len), _ptr(dO), _ptr(dHT), _ptr(dq), _ptr(dk),
        _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dH0), _ptr(ws), ws.numel(), _stream(stream)))


def gdn_fwd_ctx_kernel(index, q, k, v, a, b, A_log, dt_bias, h0, valid_len, o, hT, ctx, ws, *,
                       problem, stream=None):
    """Launch only kernel `index` of gdn_fwd_ctx (after a full gdn_fwd_ctx)."""
    _check("gdn_fwd_ctx_kernel", load_library().gdn_fwd_ctx_kernel(
        ctypes.byref(problem), index, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
        _ptr(dt_bias), _ptr(h0), _ptr(valid_len), _ptr(o), _ptr(hT), _ptr(ctx), ctx.numel(),
        _ptr(ws), ws.numel(), _stream(stream)))


def gdn_bwd_ctx_kernel(index, q, k, v, a, b, A_log, dt_bias, ctx, valid_len, dO, dHT, dq, dk,
                       dv, dg, dbeta, dH0, ws, *, problem, stream=None):
    """Launch only kernel `index` of gdn_bwd_ctx (after a full gdn_bwd_ctx)."""
    _check("gdn_bwd_ctx_kernel", load_library().gdn_bwd_ctx_kernel(
        ctypes.byref(problem), index, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
        _ptr(dt_bias), _ptr(ctx), ctx.numel(), _ptr(valid_len), _ptr(dO), _ptr(dHT), _ptr(dq),
        _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dH0), _ptr(ws), ws.numel(),
        _stream(stream)))


def gdn_noalloc_check_device_status(stream=None) -> int:
    """Synchronise, read and clear the status word of gdn_fwd_noalloc's static scratch."""
    return load_library().gdn_noalloc_check_device_status(_stream(stream))


def gdn_check_device_status(ws, stream=None) -> int:
    """Synchronous: status recorded on the device by the last call that used `ws`."""
    return load_library().gdn_check_device_status(_ptr(ws), _stream(stream))


class GDNCore(torch.autograd.Function):
    """Autograd wrapper: forward = gdn_fwd, backward = gdn_bwd (recomputes, saves inputs only)."""

    @staticmethod
    def forward(ctx, q, k, v, a, b, A_log, dt_bias, h0, valid_len, segments):
        o, hT = gdn_fwd(q, k, v, a, b, A_log, dt_bias, h0, valid_len, segments=segments)
        ctx.save_for_backward(q, k, v, a, b, A_log, dt_bias, h0, valid_len)
        ctx.segments = segments
        return o, hT

    @staticmethod
    def backward(ctx, dO, dHT):
        if any(ctx.needs_input_grad[3:7]):
            raise NotImplementedError(
                "GDNCore returns dg and dbeta through gdn_bwd; gradients w.r.t. a, b, A_log "
                "and dt_bias are not computed by this operator")
        q, k, v, a, b, A_log, dt_bias, h0, valid_len = ctx.saved_tensors
        dq, dk, dv, dg, dbeta, dH0 = gdn_bwd(
            q, k, v, a, b, A_log, dt_bias, dO.contiguous(),
            None if dHT is None else dHT.contiguous(), h0, valid_len,
            want_dH0=h0 is not None, segments=ctx.segments)
        # dg and dbeta are w.r.t. g and beta; the parameter chain to a, b,
        # A_log, dt_bias is not part of this operator.
        return dq, dk, dv, None, None, None, None, dH0, None, None


# ------------------------------------------------ causal depthwise Conv1D + SiLU prologue

def make_conv_problem(x: torch.Tensor, K: int, *, T: int | None = None,
                      T_stride: int = 0) -> ConvProblem:
    """Problem for x [B, T_stride, C] (tokens [0, T) of each row) and K taps."""
    B, Tx, C = x.shape
    p = ConvProblem()
    p.dtype = _dtype_code(x.dtype)
    p.K = K
    p.B, p.T, p.C, p.T_stride = B, (Tx if T is None else T), C, T_stride
    return p


def gdn_conv_silu_bwd_workspace_size(problem: ConvProblem) -> int:
    n = ctypes.c_size_t(0)
    _check("gdn_conv_silu_bwd_workspace_size", load_library().gdn_conv_silu_bwd_workspace_size(
        ctypes.byref(problem), ctypes.byref(n)))
    return n.value


def gdn_conv_silu_fwd(x, w, bias=None, halo=None, *, y=None, stream=None, problem=None):
    """y = silu(causal depthwise conv of x with w [C, K] (+ bias [C]), the K - 1 tokens of
    halo [B, K-1, C] before token 0).  x [B, T, C] bf16 or fp32; w, bias fp32."""
    p = problem or make_conv_problem(x, w.shape[1])
    y = y if y is not None else torch.empty_like(x)
    _check("gdn_conv_silu_fwd", load_library().gdn_conv_silu_fwd(
        ctypes.byref(p), _ptr(x), _ptr(w), _ptr(bias), _ptr(halo), _ptr(y), _stream(stream)))
    return y


def gdn_fwd_conv(x, w, a, b, A_log, dt_bias, h0=None, valid_len=None, *,
                 bias=(None, None, None), halo=(None, None, None), y=None, with_ctx=True,
                 ctx=None, segments=0, l2norm=True, eps=1e-6, scale=0.0, o=None, hT=None,
                 want_hT=True, ws=None, stream=None, problem=None):
    """The Conv1D + SiLU of x = (x_q, x_k, x_v) (layouts of q, k, v) with taps
    w = (w_q, w_k, w_v) [channels, K] fused into the forward (gdn_fwd_ctx when with_ctx,
    else gdn_fwd).  Returns (o, hT, ctx or None, (q, k, v)) with q, k, v the activated
    inputs the backward takes."""
    xq, xk, xv = x
    p = problem or make_problem(xq, xv, segments=segments, l2norm=l2norm, eps=eps, scale=scale)
    B, T, H, dv = xv.shape
    y = tuple(y) if y is not None else tuple(torch.empty_like(t) for t in x)
    cv = ConvQkv()
    cv.K = int(w[0].shape[1])
    for i in range(3):
        cv.x[i] = _ptr(x[i])
        cv.w[i] = _ptr(w[i])
        cv.bias[i] = _ptr(bias[i])
        cv.halo[i] = _ptr(halo[i])
        cv.y[i] = _ptr(y[i])
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=xq.dtype, device=xq.device)
    if hT is None and want_hT:
        hT = torch.empty((B, H, xq.shape[3], dv), dtype=torch.float32, device=xq.device)
    if with_ctx:
        ctx = ctx if ctx is not None else ctx_buffer(p, xq.device)
    else:
        ctx = None
    ws = _ws(p, GDN_OP_FWD_CTX if with_ctx else GDN_OP_FWD, ws, xq.device)
    _check("gdn_fwd_conv", load_library().gdn_fwd_conv(
        ctypes.byref(p), ctypes.byref(cv), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
        _ptr(h0), _ptr(valid_len), _ptr(o), _ptr(hT), _ptr(ctx),
        ctx.numel() if ctx is not None else 0, _ptr(ws), ws.numel(), _stream(stream)))
    return o, hT, ctx, y


def gdn_conv_silu_bwd(x, w, bias, halo, dy, *, want_dbias=True, want_dhalo=True, dx=None,
                      dw=None, dbias=None, dhalo=None, ws=None, stream=None, problem=None):
    """(dx [B,T,C], dw [C,K] fp32, dbias [C] fp32 or None, dhalo [B,K-1,C] or None).

    With a problem whose T_stride exceeds T, only tokens [0, T) of each row of dx are
    written; a dx allocated here (like x) leaves the rest of each row uninitialised."""
    p = problem or make_conv_problem(x, w.shape[1])
    B, _, C = x.shape
    K = w.shape[1]
    f32 = dict(dtype=torch.float32, device=x.device)
    dx = dx if dx is not None else torch.empty_like(x)
    dw = dw if dw is not None else torch.empty((C, K), **f32)
    if want_dbias and dbias is None:
        dbias = torch.empty((C,), **f32)
    if want_dhalo and dhalo is None and K > 1:
        dhalo = torch.empty((B, K - 1, C), dtype=x.dtype, device=x.device)
    if ws is None:
        ws = torch.empty(max(gdn_conv_silu_bwd_workspace_size(p), 16), dtype=torch.uint8,
                         device=x.device)
    _check("gdn_conv_silu_bwd", load_library().gdn_conv_silu_bwd(
        ctypes.byref(p), _ptr(x), _ptr(w), _ptr(bias), _ptr(halo), _ptr(dy), _ptr(dx), _ptr(dw),
        _ptr(dbias), _ptr(dhalo), _ptr(ws), ws.numel(), _stream(stream)))
    return dx, dw, dbias, dhalo


# ------------------------------------------------------- gated RMSNorm epilogue on o

def make_rmsnorm_problem(o: torch.Tensor, eps: float = 1e-6) -> RmsNormProblem:
    """Problem for o [..., D]: every leading index is a row."""
    p = RmsNormProblem()
    p.dtype = _dtype_code(o.dtype)
    p.D = o.shape[-1]
    p.rows = o.numel() // max(o.shape[-1], 1)
    p.eps = eps
    return p


def gdn_rmsnorm_gated_bwd_workspace_size(problem: RmsNormProblem) -> int:
    n = ctypes.c_size_t(0)
    _check("gdn_rmsnorm_gated_bwd_workspace_size",
           load_library().gdn_rmsnorm_gated_bwd_workspace_size(ctypes.byref(problem),
                                                                ctypes.byref(n)))
    return n.value


def gdn_rmsnorm_gated_fwd(o, z, w, eps=1e-6, *, y=None, stream=None, problem=None):
    """y = o / sqrt(mean(o^2) + eps) * w * silu(z) over the last dim; o, z bf16 or fp32."""
    p = problem or make_rmsnorm_problem(o, eps)
    y = y if y is not None else torch.empty_like(o)
    _check("gdn_rmsnorm_gated_fwd", load_library().gdn_rmsnorm_gated_fwd(
        ctypes.byref(p), _ptr(o), _ptr(z), _ptr(w), _ptr(y), _stream(stream)))
    return y


def gdn_rmsnorm_gated_bwd(o, z, w, dy, eps=1e-6, *, d_o=None, dz=None, dw=None, ws=None,
                          stream=None, problem=None):
    """(do, dz in o's dtype, dw [D] fp32)."""
    p = problem or make_rmsnorm_problem(o, eps)
    d_o = d_o if d_o is not None else torch.empty_like(o)
    dz = dz if dz is not None else torch.empty_like(z)
    dw = dw if dw is not None else torch.empty((o.shape[-1],), dtype=torch.float32,
                                               device=o.device)
    if ws is None:
        ws = torch.empty(max(gdn_rmsnorm_gated_bwd_workspace_size(p), 16), dtype=torch.uint8,
                         device=o.device)
    _check("gdn_rmsnorm_gated_bwd", load_library().gdn_rmsnorm_gated_bwd(
        ctypes.byref(p), _ptr(o), _ptr(z), _ptr(w), _ptr(dy), _ptr(d_o), _ptr(dz), _ptr(dw),
        _ptr(ws), ws.numel(), _stream(stream)))
    return d_o, dz, dw


# ------------------------------------------------------------ packed variable-length rows

class Varlen:
    """The offsets of a packed row: a host int32 copy (sizes the launches) and a device
    copy (read by the kernels), both [N + 1], from 0 to T."""

    def __init__(self, cu_seqlens, device="cuda"):
        host = torch.as_tensor(cu_seqlens, dtype=torch.int32).reshape(-1).cpu().contiguous()
        self.host = host
        self.n = int(host.numel()) - 1
        if self.n < 0:
            raise ValueError("cu_seqlens needs at least one offset")
        self.dev = host.to(device)

    def host_ptr(self):
        return ctypes.c_void_p(self.host.data_ptr())


def _varlen_of(cu_seqlens, device):
    return cu_seqlens if isinstance(cu_seqlens, Varlen) else Varlen(cu_seqlens, device)


def gdn_varlen_workspace_size(problem: Problem, cu: Varlen, op: int) -> int:
    n = ctypes.c_size_t(0)
    _check("gdn_varlen_workspace_size", load_library().gdn_varlen_workspace_size(
        ctypes.byref(problem), cu.host_ptr(), cu.n, op, ctypes.byref(n)))
    return n.value


def varlen_workspace(problem: Problem, cu: Varlen, op: int, device=None) -> torch.Tensor:
    n = gdn_varlen_workspace_size(problem, cu, op)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device or "cuda")


def gdn_fwd_varlen(q, k, v, a, b, A_log, dt_bias, cu_seqlens, h0=None, *, segments=0,
                   l2norm=True, eps=1e-6, scale=0.0, o=None, hT=None, want_hT=True, ws=None,
                   stream=None, problem=None):
    """Packed rows (B = 1): q, k [1,T,Hqk,dk], v [1,T,H,dv], a, b [1,T,H]; sequence i is
    tokens cu_seqlens[i] .. cu_seqlens[i+1]-1, run from h0[i] ([N,H,dk,dv] or None).
    Returns (o [1,T,H,dv], hT [N,H,dk,dv] fp32 or None)."""
    cu = _varlen_of(cu_seqlens, q.device)
    p = problem or make_problem(q, v, segments=segments, l2norm=l2norm, eps=eps, scale=scale)
    _, T, H, dv = v.shape
    if o is None:
        o = torch.empty((1, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_hT:
        hT = torch.empty((cu.n, H, q.shape[3], dv), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = varlen_workspace(p, cu, GDN_OP_FWD, q.device)
    _check("gdn_fwd_varlen", load_library().gdn_fwd_varlen(
        ctypes.byref(p), _ptr(cu.dev), cu.host_ptr(), cu.n, _ptr(q), _ptr(k), _ptr(v), _ptr(a),
        _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(o), _ptr(hT), _ptr(ws), ws.numel(),
        _stream(stream)))
    return o, hT


def gdn_bwd_varlen(q, k, v, a, b, A_log, dt_bias, cu_seqlens, dO, dHT=None, h0=None, *,
                   segments=0, l2norm=True, eps=1e-6, scale=0.0, want_dH0=True, ws=None,
                   stream=None, problem=None):
    """Backward of gdn_fwd_varlen: (dq, dk, dv, dg, dbeta, dH0 [N,H,dk,dv] or None)."""
    cu = _varlen_of(cu_seqlens, q.device)
    p = problem or make_problem(q, v, segments=segments, l2norm=l2norm, eps=eps, scale=scale)
    _, T, H, dv = v.shape
    dq, dk, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg = torch.empty((1, T, H), dtype=torch.float32, device=q.device)
    dbeta = torch.empty_like(dg)
    dH0 = torch.empty((cu.n, H, q.shape[3], dv), dtype=torch.float32,
                      device=q.device) if want_dH0 else None
    if ws is None:
        ws = varlen_workspace(p, cu, GDN_OP_BWD, q.device)
    _check("gdn_bwd_varlen", load_library().gdn_bwd_varlen(
        ctypes.byref(p), _ptr(cu.dev), cu.host_ptr(), cu.n, _ptr(q), _ptr(k), _ptr(v), _ptr(a),
        _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(dO), _ptr(dHT), _ptr(dq), _ptr(dk),
        _ptr(dv_), _ptr(dg), _ptr(dbeta), _ptr(dH0), _ptr(ws), ws.numel(), _stream(stream)))
    return dq, dk, dv_, dg, dbeta, dH0


def gdn_varlen_check_device_status(ws, problem: Problem, cu: Varlen, op: int,
                                   stream=None) -> int:
    """Synchronises and reads/clears the status words of a varlen call's workspace."""
    return load_library().gdn_varlen_check_device_status(
        _ptr(ws), ctypes.byref(problem), cu.host_ptr(), cu.n, op, _stream(stream))
