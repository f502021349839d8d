"""CPU checks of the C ABI: the library builds, loads and exports every symbol
include/gdn.h declares, and host-side validation returns the documented status
before any launch (no GPU needed: these calls never reach CUDA)."""
import ctypes
import os
import re
import subprocess

import pytest

import chunked_state_scan_gated_gb300 as gdn
from chunked_state_scan_gated_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdn.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|gdn_status|int32_t|void|size_t)\s+"
                                 r"(gdn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("gdn_fwd", "gdn_bwd", "gdn_summary", "gdn_summary_bwd", "gdn_compose",
                 "gdn_prefix_compose", "gdn_prefix_compose_bwd", "gdn_apply_state",
                 "gdn_apply_state_bwd", "gdn_query_support", "gdn_workspace_size"):
        assert must in names
    assert set(names) == set(gdn.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.gdn_abi_version() == 1


def test_status_strings(lib):
    for code, name in enumerate(["GDN_OK", "GDN_ERR_INVALID_ARG", "GDN_ERR_UNSUPPORTED",
                                 "GDN_ERR_WORKSPACE", "GDN_ERR_CUDA", "GDN_ERR_DEVICE_TIMEOUT"]):
        assert gdn.status_string(code) == name


def problem(**kw):
    p = gdn.Problem()
    gdn.load_library().gdn_problem_init(ctypes.byref(p))
    p.B, p.T, p.Hqk, p.H, p.dk, p.dv = 1, 8192, 16, 32, 128, 128
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_problem_defaults(lib):
    p = problem()
    assert p.dtype == gdn.GDN_BF16 and p.chunk == 64 and p.l2norm_qk == 1
    assert abs(p.l2_eps - 1e-6) < 1e-12 and p.scale == 0 and p.segments == 0


@pytest.mark.parametrize("kw,status", [
    ({}, gdn.GDN_OK),
    ({"chunk": 32}, gdn.GDN_ERR_UNSUPPORTED),                    # fail fast: chunk != 64
    ({"dk": 64}, gdn.GDN_ERR_UNSUPPORTED),                       # bf16 needs head dim 128
    ({"dtype": gdn.GDN_FP32, "dk": 64, "dv": 32}, gdn.GDN_OK),   # fp32 path takes it
    ({"dtype": gdn.GDN_FP32, "dk": 24}, gdn.GDN_ERR_UNSUPPORTED),
    ({"dtype": gdn.GDN_FP32, "dk": 256}, gdn.GDN_ERR_UNSUPPORTED),
    ({"H": 24}, gdn.GDN_ERR_INVALID_ARG),                        # H % Hqk != 0
    ({"Hqk": 0}, gdn.GDN_ERR_INVALID_ARG),
    ({"T": -1}, gdn.GDN_ERR_INVALID_ARG),
    ({"T_stride": 100}, gdn.GDN_ERR_INVALID_ARG),                # stride < T
    ({"T_stride": 9000}, gdn.GDN_OK),
    ({"segments": 129}, gdn.GDN_ERR_INVALID_ARG),                # more segments than chunks
    ({"segments": 128}, gdn.GDN_OK),
    ({"l2_eps": -1.0}, gdn.GDN_ERR_INVALID_ARG),
    ({"dtype": 7}, gdn.GDN_ERR_INVALID_ARG),
    ({"T": 0}, gdn.GDN_OK),
    ({"B": 0}, gdn.GDN_OK),
])
def test_query_support(lib, kw, status):
    assert gdn.gdn_query_support(problem(**kw)) == status


def test_workspace_size(lib):
    p = problem()
    sizes = [gdn.gdn_workspace_size(p, op) for op in range(4)]
    assert all(s >= 256 for s in sizes)
    assert sizes[gdn.GDN_OP_BWD] > sizes[gdn.GDN_OP_FWD]
    n = ctypes.c_size_t(0)
    assert lib.gdn_workspace_size(ctypes.byref(p), 9, ctypes.byref(n)) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_workspace_size(ctypes.byref(p), 0, None) == gdn.GDN_ERR_INVALID_ARG


A = 1 << 20      # a 16-byte aligned stand-in address; validation fails before any use


def fwd_args(**over):
    args = dict(q=A, k=A, v=A, a=A, b=A, A_log=A, dt_bias=A, h0=None, valid_len=None, o=A,
                hT=None, ws=A, ws_bytes=1 << 40)
    args.update(over)
    return args


def call_fwd(lib, p, args):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.gdn_fwd(ctypes.byref(p), vp(args["q"]), vp(args["k"]), vp(args["v"]),
                       vp(args["a"]), vp(args["b"]), vp(args["A_log"]), vp(args["dt_bias"]),
                       vp(args["h0"]), vp(args["valid_len"]), vp(args["o"]), vp(args["hT"]),
                       vp(args["ws"]), args["ws_bytes"], None)


@pytest.mark.parametrize("over,status", [
    ({"q": None}, gdn.GDN_ERR_INVALID_ARG),
    ({"o": None}, gdn.GDN_ERR_INVALID_ARG),
    ({"k": A + 2}, gdn.GDN_ERR_INVALID_ARG),          # misaligned
    ({"h0": A + 8}, gdn.GDN_ERR_INVALID_ARG),
    ({"ws": None}, gdn.GDN_ERR_WORKSPACE),
    ({"ws_bytes": 1024}, gdn.GDN_ERR_WORKSPACE),
    ({"ws": A + 16}, gdn.GDN_ERR_INVALID_ARG),        # workspace must be 256-byte aligned
])
def test_fwd_validation_fails_before_launch(lib, over, status):
    assert call_fwd(lib, problem(), fwd_args(**over)) == status


def test_unsupported_shape_is_refused_before_pointers(lib):
    assert call_fwd(lib, problem(chunk=128), fwd_args()) == gdn.GDN_ERR_UNSUPPORTED


def test_bwd_and_summary_validation(lib):
    p = problem()
    vp = ctypes.c_void_p
    base = [vp(A)] * 7 + [None, None, vp(A), None]       # ..., h0, valid_len, dO, dHT
    outs_bad = [None] + [vp(A)] * 4 + [None]
    assert lib.gdn_bwd(ctypes.byref(p), *base, *outs_bad, vp(A), 1 << 40,
                       None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_summary(ctypes.byref(p), vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), None,
                           None, vp(A), vp(A), 1 << 40, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_apply_state(ctypes.byref(p), *[vp(A)] * 7, None, None, vp(A), None, vp(A),
                               1 << 40, None) == gdn.GDN_ERR_INVALID_ARG     # Hin required


def test_compose_prefix_validation(lib):
    vp = ctypes.c_void_p
    assert lib.gdn_compose(-1, 4, 4, *[vp(A)] * 6, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_compose(2, 256, 4, *[vp(A)] * 6, None) == gdn.GDN_ERR_UNSUPPORTED
    assert lib.gdn_compose(2, 4, 4, None, *[vp(A)] * 5, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_prefix_compose(2, 0, 4, 4, vp(A), vp(A), None, vp(A), None,
                                  None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_prefix_compose_bwd(2, 3, 4, 4, vp(A), vp(A + 4), None, vp(A), None,
                                      None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_check_device_status(None, None) == gdn.GDN_ERR_INVALID_ARG


def test_ctx_size_and_validation(lib):
    """The forward context holds M and H_in of every resolved segment and, on the bf16
    tensor-core path, per chunk the prologue's outputs -- rq/rk (Hqk x 128 fp32), and per V head
    the W, U images (16 KB each), the P, T images (8 KB each) and 64 fp32 gates -- and the bf16
    image of the chunk-start state of every V head (32 KB); a missing, short or misaligned
    context is refused before any launch."""
    NC = 8192 // 64
    pro = NC * (16 * 128 * 4 + 32 * (16384 + 16384 + 8192 + 8192 + 64 * 4 + 32768))
    for seg in (0, 1, 5):
        p = problem(segments=seg)
        P = gdn.gdn_resolved_segments(p, gdn.GDN_OP_FWD)
        assert P == gdn.gdn_resolved_segments(p, gdn.GDN_OP_BWD)
        assert P == gdn.gdn_resolved_segments(p, gdn.GDN_OP_FWD_CTX)
        assert gdn.gdn_ctx_size(p) == P * 1 * 32 * (128 * 128 + 128 * 128) * 4 + pro
        # the prologue images move from the workspaces into the context
        for op, op_ctx in ((gdn.GDN_OP_FWD, gdn.GDN_OP_FWD_CTX),
                           (gdn.GDN_OP_BWD, gdn.GDN_OP_BWD_CTX)):
            assert gdn.gdn_workspace_size(p, op_ctx) < gdn.gdn_workspace_size(p, op)
        p32 = problem(segments=seg, dtype=gdn.GDN_FP32)
        P32 = gdn.gdn_resolved_segments(p32, gdn.GDN_OP_FWD)
        assert gdn.gdn_ctx_size(p32) == P32 * 1 * 32 * (128 * 128 + 128 * 128) * 4
        assert gdn.gdn_workspace_size(p32, gdn.GDN_OP_FWD_CTX) == \
            gdn.gdn_workspace_size(p32, gdn.GDN_OP_FWD)
    p = problem()
    need = gdn.gdn_ctx_size(p)
    vp = ctypes.c_void_p
    fwd = [vp(A)] * 7 + [None, None, vp(A), None]      # q .. dt_bias, h0, valid_len, o, hT
    for ctx, n in ((None, need), (A, need - 4), (A + 8, need)):
        st = lib.gdn_fwd_ctx(ctypes.byref(p), *fwd, None if ctx is None else vp(ctx), n,
                             vp(A), 1 << 40, None)
        assert st == gdn.GDN_ERR_INVALID_ARG
        st = lib.gdn_bwd_ctx(ctypes.byref(p), *[vp(A)] * 7, None if ctx is None else vp(ctx), n,
                             None, vp(A), None, *[vp(A)] * 5, None, vp(A), 1 << 40, None)
        assert st == gdn.GDN_ERR_INVALID_ARG
    names = gdn.gdn_kernel_info(p, gdn.GDN_OP_BWD_CTX)
    assert "summary_pair_tc" not in names and "grad_tc" in names      # no forward summaries
    assert "prep_tc" not in names                                      # nor the prologue
    assert "dstates_chain_tc" in names and "states_pair_tc" not in names  # nor the states
    assert "prep_tc" in gdn.gdn_kernel_info(p, gdn.GDN_OP_BWD)
    assert gdn.gdn_kernel_info(p, gdn.GDN_OP_FWD_CTX)[-1] == "apply_chain_tc"


def test_conv_validation_and_workspace(lib):
    """Host-side checks of the Conv1D + SiLU calls (no launch reaches CUDA)."""
    A = 1 << 20  # a 16-byte-aligned fake device address; validation fails before any use

    def prob(**kw):
        p = gdn.ConvProblem()
        p.dtype, p.K, p.B, p.T, p.C, p.T_stride = gdn.GDN_BF16, 4, 2, 300, 256, 0
        for k, v in kw.items():
            setattr(p, k, v)
        return p

    n = ctypes.c_size_t(0)
    assert lib.gdn_conv_silu_bwd_workspace_size(ctypes.byref(prob()), ctypes.byref(n)) == 0
    assert n.value == 2 * 3 * 256 * 5 * 4  # 2 rows x 3 tiles of 128 tokens x C x (K + 1) fp32
    assert lib.gdn_conv_silu_bwd_workspace_size(ctypes.byref(prob()), None) == \
        gdn.GDN_ERR_INVALID_ARG
    vp = ctypes.c_void_p
    for kw, status in (({"K": 5}, gdn.GDN_ERR_UNSUPPORTED), ({"K": 0}, gdn.GDN_ERR_UNSUPPORTED),
                       ({"C": 6}, gdn.GDN_ERR_UNSUPPORTED), ({"C": 12}, gdn.GDN_ERR_UNSUPPORTED),
                       ({"C": 0}, gdn.GDN_ERR_INVALID_ARG),
                       ({"T": -1}, gdn.GDN_ERR_INVALID_ARG),
                       ({"T_stride": 10}, gdn.GDN_ERR_INVALID_ARG),
                       ({"dtype": 7}, gdn.GDN_ERR_INVALID_ARG)):
        p = prob(**kw)
        assert lib.gdn_conv_silu_fwd(ctypes.byref(p), vp(A), vp(A), None, None, vp(A),
                                     None) == status, kw
        assert lib.gdn_conv_silu_bwd(ctypes.byref(p), vp(A), vp(A), None, None, vp(A), vp(A),
                                     vp(A), None, None, vp(A), 1 << 30, None) == status, kw
    p = prob()
    # null or misaligned required pointers
    assert lib.gdn_conv_silu_fwd(ctypes.byref(p), None, vp(A), None, None, vp(A), None) == \
        gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_conv_silu_fwd(ctypes.byref(p), vp(A + 8), vp(A), None, None, vp(A), None) == \
        gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_conv_silu_fwd(ctypes.byref(p), vp(A), None, None, None, vp(A), None) == \
        gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_conv_silu_bwd(ctypes.byref(p), vp(A), vp(A), None, None, None, vp(A), vp(A),
                                 None, None, vp(A), 1 << 30, None) == gdn.GDN_ERR_INVALID_ARG
    # workspace too small or missing
    assert lib.gdn_conv_silu_bwd(ctypes.byref(p), vp(A), vp(A), None, None, vp(A), vp(A), vp(A),
                                 None, None, vp(A), n.value - 16, None) == gdn.GDN_ERR_WORKSPACE
    assert lib.gdn_conv_silu_bwd(ctypes.byref(p), vp(A), vp(A), None, None, vp(A), vp(A), vp(A),
                                 None, None, None, 0, None) == gdn.GDN_ERR_WORKSPACE


def test_rmsnorm_validation_and_workspace(lib):
    """Host-side checks of the gated RMSNorm calls (no launch reaches CUDA)."""
    A = 1 << 20
    vp = ctypes.c_void_p

    def prob(**kw):
        p = gdn.RmsNormProblem()
        p.dtype, p.D, p.rows, p.eps = gdn.GDN_BF16, 128, 1000, 1e-6
        for k, v in kw.items():
            setattr(p, k, v)
        return p

    n = ctypes.c_size_t(0)
    assert lib.gdn_rmsnorm_gated_bwd_workspace_size(ctypes.byref(prob()), ctypes.byref(n)) == 0
    assert n.value == 63 * 128 * 4  # ceil(1000 / 16 rows per CTA step) CTAs x D fp32
    # the backward's grid is capped (a fixed count: dw does not depend on the device)
    big = ctypes.c_size_t(0)
    assert lib.gdn_rmsnorm_gated_bwd_workspace_size(ctypes.byref(prob(rows=1 << 20)),
                                                     ctypes.byref(big)) == 0
    assert big.value == 608 * 128 * 4
    for kw, status in (({"D": 6}, gdn.GDN_ERR_UNSUPPORTED), ({"D": 516}, gdn.GDN_ERR_UNSUPPORTED),
                       ({"D": 0}, gdn.GDN_ERR_INVALID_ARG), ({"rows": -1}, gdn.GDN_ERR_INVALID_ARG),
                       ({"eps": -1.0}, gdn.GDN_ERR_INVALID_ARG),
                       ({"dtype": 9}, gdn.GDN_ERR_INVALID_ARG)):
        p = prob(**kw)
        assert lib.gdn_rmsnorm_gated_fwd(ctypes.byref(p), vp(A), vp(A), vp(A), vp(A),
                                         None) == status, kw
        assert lib.gdn_rmsnorm_gated_bwd(ctypes.byref(p), vp(A), vp(A), vp(A), vp(A), vp(A),
                                         vp(A), vp(A), vp(A), 1 << 30, None) == status, kw
    p = prob()
    assert lib.gdn_rmsnorm_gated_fwd(ctypes.byref(p), vp(A), None, vp(A), vp(A), None) == \
        gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_rmsnorm_gated_fwd(ctypes.byref(p), vp(A), vp(A + 4), vp(A), vp(A), None) == \
        gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_rmsnorm_gated_bwd(ctypes.byref(p), vp(A), vp(A), vp(A), vp(A), vp(A), vp(A),
                                     vp(A), vp(A), n.value - 16, None) == gdn.GDN_ERR_WORKSPACE


def test_varlen_validation_and_workspace(lib):
    """Host-side checks of the packed variable-length calls (no launch reaches CUDA)."""
    A = 1 << 20
    vp = ctypes.c_void_p
    p = problem(T=500, Hqk=1, H=2)

    def ws(cu, op, prob=p):
        arr = (ctypes.c_int32 * len(cu))(*cu)
        n = ctypes.c_size_t(0)
        st = lib.gdn_varlen_workspace_size(ctypes.byref(prob), arr, len(cu) - 1, op,
                                           ctypes.byref(n))
        return st, n.value

    cu = [0, 1, 64, 64, 129, 319, 500]
    st_f, nf = ws(cu, gdn.GDN_OP_FWD)
    st_b, nb = ws(cu, gdn.GDN_OP_BWD)
    assert st_f == gdn.GDN_OK and st_b == gdn.GDN_OK and nb > nf > 0
    # the padded batch [6, 190] of the inputs and output is inside the workspace
    assert nf >= 6 * 190 * (2 * 128 + 2 * 128 + 2 + 2 + 2 * 128) * 2
    for bad in ([1, 500], [0, 400], [0, 300, 200, 500], [0, 501]):
        assert ws(bad, gdn.GDN_OP_FWD)[0] == gdn.GDN_ERR_INVALID_ARG, bad
    assert ws(cu, gdn.GDN_OP_SUMMARY)[0] == gdn.GDN_ERR_INVALID_ARG
    assert ws(cu, gdn.GDN_OP_FWD, problem(B=2, T=500, Hqk=1, H=2))[0] == gdn.GDN_ERR_INVALID_ARG
    assert ws([0], gdn.GDN_OP_FWD, problem(T=0, Hqk=1, H=2))[0] == gdn.GDN_OK
    # an unsupported shape fails as it does for gdn_fwd
    assert ws(cu, gdn.GDN_OP_FWD, problem(T=500, Hqk=1, H=2, dk=64))[0] == \
        gdn.GDN_ERR_UNSUPPORTED
    arr = (ctypes.c_int32 * 3)(0, 300, 200)
    st = lib.gdn_fwd_varlen(ctypes.byref(problem(T=200, Hqk=1, H=2)), vp(A), arr, 2,
                            *[vp(A)] * 5, vp(A), vp(A), None, vp(A), None, vp(A), 1 << 40, None)
    assert st == gdn.GDN_ERR_INVALID_ARG
    arr = (ctypes.c_int32 * 3)(0, 100, 200)
    st = lib.gdn_fwd_varlen(ctypes.byref(problem(T=200, Hqk=1, H=2)), vp(A), arr, 2,
                            *[vp(A)] * 5, vp(A), vp(A), None, vp(A), None, vp(A), 16, None)
    assert st == gdn.GDN_ERR_WORKSPACE


STRUCTS = {  # C struct name -> (ctypes mirror, its fields as named in the header)
    "gdn_problem": (gdn.Problem, [f for f, _ in gdn.Problem._fields_]),
    "gdn_conv_problem": (gdn.ConvProblem, [f for f, _ in gdn.ConvProblem._fields_]),
    "gdn_conv_qkv": (gdn.ConvQkv, [f for f, _ in gdn.ConvQkv._fields_]),
    "gdn_rmsnorm_problem": (gdn.RmsNormProblem, [f for f, _ in gdn.RmsNormProblem._fields_]),
}


def test_struct_layouts_match_the_header(tmp_path):
    """sizeof and every field offset of the public structs, as gcc lays them out from
    include/gdn.h, equal those of the binding's ctypes mirrors."""
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "gdn.h"', "int main(void) {"]
    for name, (_, fields) in STRUCTS.items():
        lines.append(f'  printf("{name} size %zu\\n", sizeof({name}));')
        for f in fields:
            lines.append(f'  printf("{name} {f} %zu\\n", offsetof({name}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {}
    for line in out.splitlines():
        name, key, val = line.split()
        got[(name, key)] = int(val)
    for name, (cls, fields) in STRUCTS.items():
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for f in fields:
            assert got[(name, f)] == getattr(cls, f).offset, (name, f)


def call_fwd_conv(lib, p, cv, ws=None, ws_bytes=0):
    vp = ctypes.c_void_p
    return lib.gdn_fwd_conv(ctypes.byref(p), None if cv is None else ctypes.byref(cv),
                            *[vp(A)] * 4, None, None, vp(A), None, None, 0,
                            None if ws is None else vp(ws), ws_bytes, None)


def conv_qkv(**over):
    cv = gdn.ConvQkv()
    cv.K = over.pop("K", 4)
    for i in range(3):
        cv.x[i] = A
        cv.w[i] = A
        cv.y[i] = A + (1 << 30) + i * (1 << 28)   # clear of every x
    for key, (i, val) in over.items():
        getattr(cv, key)[i] = val
    return cv


@pytest.mark.parametrize("over,status", [
    ({"x": (0, None)}, gdn.GDN_ERR_INVALID_ARG),
    ({"w": (2, None)}, gdn.GDN_ERR_INVALID_ARG),
    ({"y": (1, None)}, gdn.GDN_ERR_INVALID_ARG),
    ({"bias": (0, A + 4)}, gdn.GDN_ERR_INVALID_ARG),     # misaligned
    ({"halo": (2, A + 8)}, gdn.GDN_ERR_INVALID_ARG),
    ({"y": (1, A + 64)}, gdn.GDN_ERR_INVALID_ARG),       # y overlaps its x
    ({"K": 5}, gdn.GDN_ERR_UNSUPPORTED),
    ({"K": 0}, gdn.GDN_ERR_UNSUPPORTED),
    ({}, gdn.GDN_ERR_WORKSPACE),                          # valid up to the missing workspace
])
def test_fwd_conv_validation_fails_before_launch(lib, over, status):
    assert call_fwd_conv(lib, problem(), conv_qkv(**over)) == status


def test_fwd_conv_needs_its_description(lib):
    assert call_fwd_conv(lib, problem(), None) == gdn.GDN_ERR_INVALID_ARG
