"""GPU parity of the Conv1D + SiLU fused into the forward (gdn_fwd_conv, through the C ABI).

Two references:
  * the fp64 oracles composed as the pages put the steps ("linear attention cp #1035",
    section "What does this PR do": the depthwise Conv1D feeds q, k, v of the Gated
    DeltaNet): oracle.conv_silu_fwd on each of x_q, x_k, x_v, then oracle.fwd on the three
    results, compared at the bf16 bars (rel-L2 <= 1e-2, max-abs / ref-abs-max <= 1e-1);
  * the stand-alone Conv1D (gdn_conv_silu_fwd) followed by gdn_fwd_ctx / gdn_fwd, which the
    fused call must reproduce bit for bit (same operation order on the same bf16 inputs):
    the activated q, k, v, o, h_T and the whole training-step context.
Cases span several chunks and a ragged tail, every tap count, with and without halo and
bias, grouped heads (r = 1, 2, 4), padded rows, and the bench's head layout at T = 8192 (the
persistent prologue walking many chunks per CTA).
"""
import pytest
import torch

import oracle
import chunked_state_scan_gated_gb300 as gdn
from chunked_state_scan_gated_gb300 import inputs as gi
from tests.helpers import assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load_library()


def make_case(B, T, Hqk, H, K, *, halo, bias, seed, valid_len=None, d=128,
              dtype=torch.bfloat16):
    """Core inputs of the shape plus, per q, k, v, the Conv1D inputs x (layout of q, k, v),
    taps w [channels, K], bias and halo (all seeded, on the CPU)."""
    w = gi.Workload("conv_fused", B=B, T=T, Hqk=Hqk, H=H, dk=d, dv=d, dtype=dtype, h0_std=0.1,
                    valid_len=valid_len, seed=seed)
    core = gi.make_inputs(w)
    conv = []
    for i, heads in enumerate((Hqk, Hqk, H)):
        c = gi.make_conv_inputs(B, T, heads * d, K, dtype, seed=seed * 10 + i, halo=halo,
                                bias=bias)
        conv.append({"x": c["x"].view(B, T, heads, d), "w": c["w"], "bias": c["bias"],
                     "halo": c["halo"]})
    return core, conv


def cuda(t):
    return t.cuda() if torch.is_tensor(t) else t


def zero_ctx(core):
    """A zero-filled context buffer: the context has alignment gaps that no call writes."""
    p = gdn.make_problem(core["q"], core["v"])
    return torch.zeros(gdn.gdn_ctx_size(p), dtype=torch.uint8, device="cuda")


def same_bytes(name, a_, b_):
    eq = a_ == b_
    if not bool(eq.all()):
        bad = torch.nonzero(~eq).flatten()
        raise AssertionError(f"{name}: {bad.numel()} of {eq.numel()} bytes differ, first at "
                             f"{int(bad[0])}, last at {int(bad[-1])}")


def run_fused(core, conv, with_ctx=True):
    d = {k: cuda(v) for k, v in core.items()}
    x = tuple(cuda(c["x"]) for c in conv)
    w = tuple(cuda(c["w"]) for c in conv)
    bias = tuple(cuda(c["bias"]) for c in conv)
    halo = tuple(cuda(c["halo"]) for c in conv)
    o, hT, ctx, y = gdn.gdn_fwd_conv(x, w, d["a"], d["b"], d["A_log"], d["dt_bias"], d["h0"],
                                     d["valid_len"], bias=bias, halo=halo, with_ctx=with_ctx,
                                     ctx=zero_ctx(core) if with_ctx else None)
    torch.cuda.synchronize()
    return o, hT, ctx, y


def run_separate(core, conv, with_ctx=True):
    d = {k: cuda(v) for k, v in core.items()}
    y = []
    for c in conv:
        x = cuda(c["x"])
        B, T, heads, _ = x.shape
        yi = gdn.gdn_conv_silu_fwd(x.reshape(B, T, -1), cuda(c["w"]), cuda(c["bias"]),
                                   cuda(c["halo"]))
        y.append(yi.view(x.shape))
    args = (y[0], y[1], y[2], d["a"], d["b"], d["A_log"], d["dt_bias"], d["h0"], d["valid_len"])
    if with_ctx:
        o, hT, ctx = gdn.gdn_fwd_ctx(*args, ctx=zero_ctx(core))
    else:
        o, hT = gdn.gdn_fwd(*args)[:2]
        ctx = None
    torch.cuda.synchronize()
    return o, hT, ctx, tuple(y)


def live_tokens(valid_len, T, B):
    """Tokens of each row that sit in a chunk holding a valid token."""
    if valid_len is None:
        return [T] * B
    return [min(T, (int(L) + 63) // 64 * 64) for L in valid_len]


CASES = [  # B, T, Hqk, H, K, halo, bias, valid_len
    (2, 190, 2, 4, 4, True, True, None),
    (1, 320, 2, 2, 2, False, True, None),
    (1, 100, 1, 4, 1, False, False, None),
    (2, 200, 2, 4, 3, True, True, [130, 200]),
    (1, 64, 2, 4, 4, True, False, None),
    (1, 1, 2, 4, 4, True, True, None),            # one token: every tap but one is halo
    (2, 130, 2, 4, 4, True, True, [0, 70]),       # a row of padding only
]
IDS = [f"B{c[0]}_T{c[1]}_h{c[2]}x{c[3]}_K{c[4]}{'_halo' if c[5] else ''}"
       f"{'_bias' if c[6] else ''}{'_padded' if c[7] else ''}" for c in CASES]


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_fused_conv_matches_oracle(case):
    B, T, Hqk, H, K, halo, bias, vl = case
    core, conv = make_case(B, T, Hqk, H, K, halo=halo, bias=bias, seed=B * 100 + T + K,
                           valid_len=vl)
    o, hT, _, y = run_fused(core, conv)
    ry = []
    for c in conv:
        x = to64(c["x"])
        Bx, Tx, heads, _ = x.shape
        r = oracle.conv_silu_fwd(x.reshape(Bx, Tx, -1), to64(c["w"]), to64(c["bias"]),
                                 to64(c["halo"]))
        ry.append(r.reshape(x.shape))
    ends = live_tokens(vl, T, B)
    for name, yi, ri in zip("qkv", y, ry):
        for bb, end in enumerate(ends):
            assert_close(f"y_{name}[{bb}]", yi[bb, :end], ri[bb, :end], torch.bfloat16)
            assert not torch.any(yi[bb, end:] != 0), f"y_{name}[{bb}] past the live chunks"
    ro, rhT = oracle.fwd(ry[0], ry[1], ry[2], to64(core["a"]), to64(core["b"]),
                         to64(core["A_log"]), to64(core["dt_bias"]), to64(core["h0"]),
                         core["valid_len"])
    if vl is None:
        assert_close("o", o, ro, torch.bfloat16)
    else:
        for bb, L in enumerate(vl):
            assert_close(f"o[{bb}]", o[bb, :L], ro[bb, :L], torch.bfloat16)
    assert_close("hT", hT, rhT, torch.bfloat16)


@pytest.mark.parametrize("with_ctx", [True, False], ids=["ctx", "no_ctx"])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_fused_conv_equals_separate_passes(case, with_ctx):
    B, T, Hqk, H, K, halo, bias, vl = case
    core, conv = make_case(B, T, Hqk, H, K, halo=halo, bias=bias, seed=B * 100 + T + K + 7,
                           valid_len=vl)
    o, hT, ctx, y = run_fused(core, conv, with_ctx)
    so, shT, sctx, sy = run_separate(core, conv, with_ctx)
    for bb, end in enumerate(live_tokens(vl, T, B)):
        for name, a_, b_ in zip("qkv", y, sy):
            assert torch.equal(a_[bb, :end], b_[bb, :end]), f"y_{name}[{bb}] differs"
    assert torch.equal(o, so)
    assert torch.equal(hT, shT)
    if with_ctx:
        same_bytes("ctx", ctx, sctx)
    else:
        assert ctx is None


def test_fused_conv_bench_heads_8k_and_backward():
    """H = 32 from 16 Q/K heads, T = 8192, K = 4 with halo and bias: the fused forward equals
    the separate passes bit for bit, and the training-step backward from its context equals
    the backward from the separate passes' context."""
    core, conv = make_case(1, 8192, 16, 32, 4, halo=True, bias=True, seed=11)
    o, hT, ctx, y = run_fused(core, conv)
    so, shT, sctx, sy = run_separate(core, conv)
    for name, a_, b_ in zip("qkv", y, sy):
        assert torch.equal(a_, b_), f"y_{name} differs"
    assert torch.equal(o, so) and torch.equal(hT, shT)
    same_bytes("ctx", ctx, sctx)
    d = {k: cuda(v) for k, v in core.items()}
    g1 = gdn.gdn_bwd_ctx(y[0], y[1], y[2], d["a"], d["b"], d["A_log"], d["dt_bias"], ctx,
                         d["dO"], d["dHT"])
    g2 = gdn.gdn_bwd_ctx(sy[0], sy[1], sy[2], d["a"], d["b"], d["A_log"], d["dt_bias"], sctx,
                         d["dO"], d["dHT"])
    torch.cuda.synchronize()
    for name, a_, b_ in zip(("dq", "dk", "dv", "dg", "dbeta", "dH0"), g1, g2):
        assert torch.equal(a_, b_), f"{name} differs"


def test_fused_conv_rejects_bad_arguments():
    core, conv = make_case(1, 128, 2, 4, 4, halo=True, bias=True, seed=3)
    d = {k: cuda(v) for k, v in core.items()}
    x = tuple(cuda(c["x"]) for c in conv)
    w = tuple(cuda(c["w"]) for c in conv)
    # y overlapping its x
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_fwd_conv(x, w, d["a"], d["b"], d["A_log"], d["dt_bias"], y=(x[0], x[1], x[2]))
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG
    # five taps
    w5 = tuple(torch.zeros((t.shape[0], 5), dtype=torch.float32, device="cuda") for t in w)
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_fwd_conv(x, w5, d["a"], d["b"], d["A_log"], d["dt_bias"])
    assert e.value.status == gdn.GDN_ERR_UNSUPPORTED


def test_fused_conv_row_stride():
    """Rows T_stride = 200 tokens apart, T = 150 of them used: the fused call reads x and
    writes y (and o) in those rows only, as the separate passes do."""
    B, T, Ts, Hqk, H, K = 2, 150, 200, 2, 4, 4
    core, conv = make_case(B, Ts, Hqk, H, K, halo=True, bias=True, seed=21)
    d = {k: cuda(v) for k, v in core.items()}
    x = tuple(cuda(c["x"]) for c in conv)
    w = tuple(cuda(c["w"]) for c in conv)
    bias = tuple(cuda(c["bias"]) for c in conv)
    halo = tuple(cuda(c["halo"]) for c in conv)
    p = gdn.make_problem(d["q"], d["v"], T=T, T_stride=Ts)
    o = torch.zeros_like(d["v"])
    y = tuple(torch.zeros_like(t) for t in x)
    o, hT, _, y = gdn.gdn_fwd_conv(x, w, d["a"], d["b"], d["A_log"], d["dt_bias"], d["h0"],
                                   bias=bias, halo=halo, y=y, o=o, with_ctx=False, problem=p)
    sy = []
    for xi, wi, bi, hi in zip(x, w, bias, halo):
        cp = gdn.make_conv_problem(xi.reshape(B, Ts, -1), K, T=T, T_stride=Ts)
        yi = torch.zeros_like(xi)
        gdn.gdn_conv_silu_fwd(xi.reshape(B, Ts, -1), wi, bi, hi, y=yi.view(B, Ts, -1),
                              problem=cp)
        sy.append(yi)
    so = torch.zeros_like(d["v"])
    so, shT = gdn.gdn_fwd(sy[0], sy[1], sy[2], d["a"], d["b"], d["A_log"], d["dt_bias"],
                          d["h0"], o=so, problem=p)[:2]
    torch.cuda.synchronize()
    for name, a_, b_ in zip("qkv", y, sy):
        assert torch.equal(a_, b_), f"y_{name} differs"
        assert not torch.any(a_[:, T:] != 0), f"y_{name} written past T"
    assert torch.equal(o, so) and torch.equal(hT, shT)


def test_fused_conv_fp32_cuda_core_route():
    """fp32 (CUDA-core path, d = 32): the call runs the stand-alone Conv1D, then the forward;
    checked against the composed fp64 oracles at the fp32 bar (rel-L2 <= 1e-5)."""
    B, T, Hqk, H, K = 1, 150, 2, 4, 3
    core, conv = make_case(B, T, Hqk, H, K, halo=True, bias=True, seed=31, d=32,
                           dtype=torch.float32)
    o, hT, ctx, y = run_fused(core, conv)
    ry = []
    for c in conv:
        x = to64(c["x"])
        r = oracle.conv_silu_fwd(x.reshape(B, T, -1), to64(c["w"]), to64(c["bias"]),
                                 to64(c["halo"]))
        ry.append(r.reshape(x.shape))
    for name, yi, ri in zip("qkv", y, ry):
        assert_close(f"y_{name}", yi, ri, torch.float32)
    ro, rhT = oracle.fwd(ry[0], ry[1], ry[2], to64(core["a"]), to64(core["b"]),
                         to64(core["A_log"]), to64(core["dt_bias"]), to64(core["h0"]))
    assert_close("o", o, ro, torch.float32)
    assert_close("hT", hT, rhT, torch.float32)
