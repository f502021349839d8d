"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle.

Small cases are compared element by element on every output; the full-size
workloads (T = 8K, 32K, 64K with H = 32, dk = dv = 128, bf16) are compared on
sampled Q/K groups (the oracle computes them one by one) plus properties that
hold at any size (finite outputs, zero output and gradients on padded tokens,
segment composition equal to the monolithic run).

Bars: fp32 I/O rel-L2 <= 1e-5; bf16 I/O rel-L2 <= 1e-2 and
max-abs / ref-abs-max <= 1e-1 per tensor (the acceptance bar of the
"Linear Attention CP 融合算子 PR #1114 测试报告", section 4.2: worst rel-L2
5.86e-3 against a 1e-2 threshold, all tensors finite).
"""
import numpy as np
import pytest
import torch

import oracle
import chunked_state_scan_gated_gb300 as gdn
from chunked_state_scan_gated_gb300 import inputs as gi
from tests.helpers import assert_close, head_slice, to64

pytestmark = pytest.mark.gpu

NAMES_BWD = ("dq", "dk", "dv", "dg", "dbeta", "dH0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load_library()


def dev(inp):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}


def np64(inp):
    return gi.to_numpy64(inp)


def oracle_fwd(n, **kw):
    return oracle.fwd(n["q"], n["k"], n["v"], n["a"], n["b"], n["A_log"], n["dt_bias"],
                      h0=n["h0"], valid_len=n["valid_len"], **kw)


def oracle_bwd(n, **kw):
    return oracle.bwd(n["q"], n["k"], n["v"], n["a"], n["b"], n["A_log"], n["dt_bias"], n["dO"],
                      n["dHT"], h0=n["h0"], valid_len=n["valid_len"], **kw)


def gpu_fwd(d, segments=0):
    return gdn.gdn_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                       d["h0"], d["valid_len"], segments=segments)


def gpu_bwd(d, segments=0):
    return gdn.gdn_bwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                       d["dO"], d["dHT"], d["h0"], d["valid_len"], segments=segments)


def check_fwd_bwd(w, inp, segments=0, sample=None, bwd=True):
    """Run GPU fwd (+bwd) on the whole problem; compare all or sampled Q/K groups."""
    d = dev(inp)
    o, hT = gpu_fwd(d, segments)
    grads = gpu_bwd(d, segments) if bwd else None
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    r = w.H // w.Hqk
    groups = [(0, w.Hqk)] if sample is None else [(hq, 1) for hq in sample]
    for hq0, nq in groups:
        n = np64(head_slice(inp, hq0, nq, r))
        h0s, h1s = hq0 * r, (hq0 + nq) * r
        ro, rhT = oracle_fwd(n)
        assert_close("o", o[:, :, h0s:h1s], ro, w.dtype)
        assert_close("hT", hT[:, h0s:h1s], rhT, w.dtype)
        if bwd:
            ref = oracle_bwd(n)
            got = (grads[0][:, :, hq0:hq0 + nq], grads[1][:, :, hq0:hq0 + nq],
                   grads[2][:, :, h0s:h1s], grads[3][:, :, h0s:h1s], grads[4][:, :, h0s:h1s],
                   grads[5][:, h0s:h1s] if grads[5] is not None else None)
            for name, g, rg in zip(NAMES_BWD, got, ref):
                if name == "dH0" and inp["h0"] is None:
                    continue
                assert_close(name, g, rg, w.dtype)
    return o, hT, grads


# ------------------------------------------------------------- fp32, full compare

SMALL = [
    # name, B, T, Hqk, H, dk, dv, segments, h0_std, valid_len, stress
    ("cfg0_tiny", 1, 128, 4, 8, 16, 16, 2, None, None, False),
    ("cfg0_tiny_stress", 1, 128, 4, 8, 16, 16, 2, 0.1, None, True),
    ("T1", 1, 1, 2, 4, 32, 32, 0, 0.1, None, True),
    ("T63", 1, 63, 2, 4, 32, 32, 0, 0.1, None, True),
    ("T64", 1, 64, 2, 4, 32, 32, 1, 0.1, None, True),
    ("T65", 2, 65, 2, 4, 32, 32, 2, 0.1, None, True),
    ("T200_seg3", 1, 200, 1, 3, 32, 48, 3, 0.1, None, True),
    ("dk64_dv32", 1, 150, 1, 2, 64, 32, 0, 0.1, None, True),
    ("d128_fp32", 1, 300, 2, 4, 128, 128, 2, 0.1, None, True),
    ("padded", 2, 130, 1, 2, 32, 32, 2, 0.1, [70, 130], True),
    ("padded_mid_chunk", 2, 200, 2, 4, 16, 16, 3, 0.1, [97, 3], False),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_fp32_fwd_bwd_matches_oracle(case):
    name, B, T, Hqk, H, dk, dv, seg, h0s, vl, stress = case
    w = gi.Workload(name, B=B, T=T, Hqk=Hqk, H=H, dk=dk, dv=dv, dtype=torch.float32,
                    h0_std=h0s, with_dHT=h0s is not None, valid_len=vl, decay_stress=stress,
                    seed=11)
    inp = gi.make_inputs(w)
    check_fwd_bwd(w, inp, segments=seg)


BF16_SMALL = [
    # name, B, T, Hqk, H, segments, h0_std, valid_len, stress
    ("bf16_T1", 1, 1, 1, 2, 0, 0.1, None, True),
    ("bf16_T63", 1, 63, 1, 2, 0, 0.1, None, True),
    ("bf16_T64", 1, 64, 1, 2, 1, None, None, False),
    ("bf16_T200_seg3", 2, 200, 1, 2, 3, 0.1, None, True),
    ("bf16_T320_seg2", 1, 320, 2, 4, 2, 0.1, None, True),
    ("bf16_padded", 2, 300, 1, 2, 2, 0.1, [300, 97], True),
    ("bf16_r4_default_decay", 1, 256, 1, 4, 2, 0.1, None, False),
]


PARAM_CASES = [  # name, dtype, B, T, H, valid_len
    ("fp32", torch.float32, 1, 130, 3, None),
    ("bf16_padded", torch.bfloat16, 2, 300, 4, [300, 97]),
    ("bf16_32k", torch.bfloat16, 1, 32768, 32, None),
]


@pytest.mark.parametrize("case", PARAM_CASES, ids=[c[0] for c in PARAM_CASES])
def test_gate_param_grads_match_oracle(case):
    """gdn_gate_param_bwd on given dg, dbeta (seeded, fp32) against the oracle's chain:
    both sides read the same values, the kernel computes in fp32 (fp32 tolerance)."""
    name, dtype, B, T, H, vl = case
    gen = torch.Generator().manual_seed(41)
    a = torch.randn(B, T, H, generator=gen).to(dtype)
    b = torch.randn(B, T, H, generator=gen).to(dtype)
    A_log = torch.log(torch.rand(H, generator=gen) * 15 + 1)
    dt_bias = torch.randn(H, generator=gen)
    dg = torch.randn(B, T, H, generator=gen)
    dbeta = torch.randn(B, T, H, generator=gen)
    vlt = None if vl is None else torch.tensor(vl, dtype=torch.int32)
    got = gdn.gdn_gate_param_bwd(a.cuda(), b.cuda(), A_log.cuda(), dt_bias.cuda(), dg.cuda(),
                                 dbeta.cuda(), None if vlt is None else vlt.cuda())
    torch.cuda.synchronize()
    ref = oracle.gate_param_bwd(to64(a), to64(b), to64(A_log), to64(dt_bias), to64(dg),
                                to64(dbeta), None if vl is None else np.array(vl, np.int32))
    for nm, g, r in zip(("da", "db", "dA_log", "ddt_bias"), got, ref):
        assert_close(nm, g, r, torch.float32)
    if vl is not None:
        for bi, Lb in enumerate(vl):
            assert (got[0][bi, Lb:] == 0).all() and (got[1][bi, Lb:] == 0).all()
    again = gdn.gdn_gate_param_bwd(a.cuda(), b.cuda(), A_log.cuda(), dt_bias.cuda(), dg.cuda(),
                                   dbeta.cuda(), None if vlt is None else vlt.cuda())
    for x, y in zip(got, again):  # fixed-order sums: bitwise repeatable
        assert torch.equal(x, y)


def test_gate_param_grads_end_to_end_bf16():
    """gdn_bwd -> gdn_gate_param_bwd against oracle.bwd -> oracle.gate_param_bwd."""
    w = gi.Workload("params_e2e", B=2, T=300, Hqk=1, H=2, dk=128, dv=128,
                    dtype=torch.bfloat16, h0_std=0.1, with_dHT=True, valid_len=[300, 150],
                    decay_stress=True, seed=23)
    inp = gi.make_inputs(w)
    d, n = dev(inp), np64(inp)
    grads = gpu_bwd(d)
    got = gdn.gdn_gate_param_bwd(d["a"], d["b"], d["A_log"], d["dt_bias"], grads[3], grads[4],
                                 d["valid_len"])
    torch.cuda.synchronize()
    rg = oracle_bwd(n)
    ref = oracle.gate_param_bwd(n["a"], n["b"], n["A_log"], n["dt_bias"], rg[3], rg[4],
                                n["valid_len"])
    for nm, g, r in zip(("da", "db", "dA_log", "ddt_bias"), got, ref):
        assert_close(nm, g, r, torch.bfloat16)


@pytest.mark.parametrize("case", BF16_SMALL, ids=[c[0] for c in BF16_SMALL])
def test_bf16_small_fwd_bwd_matches_oracle(case):
    name, B, T, Hqk, H, seg, h0s, vl, stress = case
    w = gi.Workload(name, B=B, T=T, Hqk=Hqk, H=H, dk=128, dv=128, dtype=torch.bfloat16,
                    h0_std=h0s, with_dHT=h0s is not None, valid_len=vl, decay_stress=stress,
                    seed=17)
    o, hT, g = check_fwd_bwd(w, gi.make_inputs(w), segments=seg)
    if vl is not None:
        for bi, Lb in enumerate(vl):
            assert (o[bi, Lb:] == 0).all()


@pytest.mark.parametrize("r, l2norm", [(1, True), (2, False), (4, False)],
                         ids=["r1_l2norm", "r2_raw_qk", "r4_raw_qk"])
def test_bf16_head_groups_and_raw_qk(r, l2norm):
    """dq, dk summed over each Q/K head's r V heads (r = 1, 2, 4), with and without the
    L2 norm of q and k (without it: q_hat = scale q, k_hat = k; the raw q, k are drawn
    small so that the recurrence stays contractive)."""
    w = gi.Workload(f"bf16_r{r}", B=2, T=200, Hqk=2, H=2 * r, dk=128, dv=128,
                    dtype=torch.bfloat16, h0_std=0.1, with_dHT=True, valid_len=[200, 133],
                    decay_stress=True, seed=41 + r)
    inp = gi.make_inputs(w)
    kw = {}
    if not l2norm:
        for nm in ("q", "k"):
            inp[nm] = (inp[nm].float() * 0.07).to(torch.bfloat16)
        kw = dict(l2norm=False, scale=0.5)
    d = dev(inp)
    o, hT = gdn.gdn_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                        d["h0"], d["valid_len"], segments=2, **kw)
    grads = gdn.gdn_bwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                        d["dO"], d["dHT"], d["h0"], d["valid_len"], segments=2, **kw)
    torch.cuda.synchronize()
    n = np64(inp)
    ro, rhT = oracle_fwd(n, **kw)
    assert_close("o", o, ro, w.dtype)
    assert_close("hT", hT, rhT, w.dtype)
    for name, g, rg in zip(NAMES_BWD, grads, oracle_bwd(n, **kw)):
        assert_close(name, g, rg, w.dtype)
    for bi, Lb in enumerate(w.valid_len):  # padded tokens: zero dq, dk
        assert (grads[0][bi, Lb:] == 0).all() and (grads[1][bi, Lb:] == 0).all()


@pytest.mark.parametrize("segments", [0, 2, 3])
def test_bf16_padding_only_chunks_are_skipped_and_zeroed(segments):
    """Rows with chunks of padding only (valid_len 0, 70, 191 of T = 320: the tensor-core
    kernels skip every chunk from ceil(valid_len / 64) on): every output and gradient
    matches the oracle, and every padded token's output and gradient is exactly zero even
    in output buffers that held NaN before the call (plain and training-step calls)."""
    w = gi.Workload("bf16_pad_chunks", B=3, T=320, Hqk=1, H=2, dk=128, dv=128,
                    dtype=torch.bfloat16, h0_std=0.1, with_dHT=True, valid_len=[0, 70, 191],
                    decay_stress=True, seed=47)
    inp = gi.make_inputs(w)
    d = dev(inp)
    n = np64(inp)
    fin = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"])
    nan = float("nan")
    o = torch.full_like(d["v"], nan)
    o, hT = gdn.gdn_fwd(*fin, d["h0"], d["valid_len"], segments=segments, o=o)
    outs = dict(dq=torch.full_like(d["q"], nan), dk=torch.full_like(d["k"], nan),
                dv=torch.full_like(d["v"], nan),
                dg=torch.full((3, 320, 2), nan, device="cuda"),
                dbeta=torch.full((3, 320, 2), nan, device="cuda"))
    grads = gdn.gdn_bwd(*fin, d["dO"], d["dHT"], d["h0"], d["valid_len"], segments=segments,
                        **outs)
    o2, hT2, ctx = gdn.gdn_fwd_ctx(*fin, d["h0"], d["valid_len"], segments=segments,
                                   o=torch.full_like(d["v"], nan))
    grads2 = gdn.gdn_bwd_ctx(*fin, ctx, d["dO"], d["dHT"], d["valid_len"], segments=segments)
    torch.cuda.synchronize()
    ro, rhT = oracle_fwd(n)
    rg = oracle_bwd(n)
    for oo, hh, gg in ((o, hT, grads), (o2, hT2, grads2)):
        assert_close("o", oo, ro, w.dtype)
        assert_close("hT", hh, rhT, w.dtype)
        for name, g, r in zip(NAMES_BWD, gg, rg):
            assert_close(name, g, r, w.dtype)
        for bi, Lb in enumerate(w.valid_len):
            for x in (oo, *gg[:5]):
                assert (x[bi, Lb:] == 0).all()
        torch.testing.assert_close(hh[0], d["h0"][0], rtol=0, atol=0)  # an empty row


def test_bf16_summary_matches_oracle():
    w = gi.Workload("bf16_summary", B=2, T=190, Hqk=1, H=2, dk=128, dv=128, dtype=torch.bfloat16,
                    decay_stress=True, valid_len=[190, 150], seed=18)
    inp = gi.make_inputs(w)
    n = np64(inp)
    d = dev(inp)
    M, S = gdn.gdn_summary(d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                           d["valid_len"])
    rM, rS = oracle.summary(n["k"], n["v"], n["a"], n["b"], n["A_log"], n["dt_bias"],
                            n["valid_len"])
    assert_close("M", M, rM, torch.bfloat16)
    assert_close("S", S, rS, torch.bfloat16)


def test_segment_counts_agree_fp32():
    w = gi.Workload("segcount", B=1, T=640, Hqk=2, H=4, dk=32, dv=32, dtype=torch.float32,
                    h0_std=0.1, with_dHT=True, decay_stress=True, seed=12)
    d = dev(gi.make_inputs(w))
    ref_o, ref_hT = gpu_fwd(d, 1)
    ref_g = gpu_bwd(d, 1)
    for P in (2, 3, 10):
        o, hT = gpu_fwd(d, P)
        g = gpu_bwd(d, P)
        assert_close(f"o P={P}", o, ref_o, torch.float32)
        assert_close(f"hT P={P}", hT, ref_hT, torch.float32)
        for name, a, b in zip(NAMES_BWD, g, ref_g):
            assert_close(f"{name} P={P}", a, b, torch.float32)


def test_summary_compose_prefix_apply_fp32():
    """Public segment calls: summaries, gradient summaries, compose, prefix,
    reverse prefix and per-segment apply/apply-backward against the oracle, and
    their composition against the monolithic run."""
    w = gi.Workload("segs", B=2, T=256, Hqk=2, H=4, dk=32, dv=32, dtype=torch.float32,
                    h0_std=0.1, with_dHT=True, decay_stress=True, seed=13)
    inp = gi.make_inputs(w)
    n = np64(inp)
    d = dev(inp)
    cuts = [0, 64, 128, 192, 256]
    Ms, Ss, Ds = [], [], []
    for s0, s1 in zip(cuts[:-1], cuts[1:]):
        sl = {k: (v[:, s0:s1].contiguous() if k in ("q", "k", "v", "a", "b", "dO") else v)
              for k, v in d.items()}
        nl = {k: (v[:, s0:s1] if k in ("q", "k", "v", "a", "b", "dO") else v) for k, v in n.items()}
        M, S = gdn.gdn_summary(sl["k"], sl["v"], sl["a"], sl["b"], sl["A_log"], sl["dt_bias"])
        rM, rS = oracle.summary(nl["k"], nl["v"], nl["a"], nl["b"], nl["A_log"], nl["dt_bias"])
        assert_close("M", M, rM, torch.float32)
        assert_close("S", S, rS, torch.float32)
        D = gdn.gdn_summary_bwd(sl["q"], sl["k"], sl["a"], sl["b"], sl["A_log"], sl["dt_bias"],
                                sl["dO"])
        rD = oracle.summary_bwd(nl["q"], nl["k"], nl["a"], nl["b"], nl["A_log"], nl["dt_bias"],
                                nl["dO"])
        assert_close("D", D, rD, torch.float32)
        Ms.append(M)
        Ss.append(S)
        Ds.append(D)
    Mst, Sst, Dst = torch.stack(Ms), torch.stack(Ss), torch.stack(Ds)
    M01, S01 = gdn.gdn_compose(Ms[1], Ss[1], Ms[0], Ss[0])
    rM01, rS01 = oracle.compose(to64(Ms[1]), to64(Ss[1]), to64(Ms[0]), to64(Ss[0]))
    assert_close("compose M", M01, rM01, torch.float32)
    assert_close("compose S", S01, rS01, torch.float32)
    Hin, Hout = gdn.gdn_prefix_compose(Mst, Sst, d["h0"])
    rHin, rHout = oracle.prefix(to64(Mst), to64(Sst), n["h0"])
    assert_close("Hin", Hin, rHin, torch.float32)
    assert_close("Hout", Hout, rHout, torch.float32)
    dHout, dH0 = gdn.gdn_prefix_compose_bwd(Mst, Dst, d["dHT"])
    rdHout, rdH0 = oracle.prefix_bwd(to64(Mst), to64(Dst), n["dHT"])
    assert_close("dHout", dHout, rdHout, torch.float32)
    assert_close("dH0 (prefix)", dH0, rdH0, torch.float32)
    # monolithic references
    ro, rhT = oracle_fwd(n)
    rg = oracle_bwd(n)
    assert_close("dH0 (composed vs monolithic)", dH0, rg[5], torch.float32)
    assert_close("Hout vs hT", Hout, rhT, torch.float32)
    for i, (s0, s1) in enumerate(zip(cuts[:-1], cuts[1:])):
        sl = {k: (v[:, s0:s1].contiguous() if k in ("q", "k", "v", "a", "b", "dO") else v)
              for k, v in d.items()}
        o, hT = gdn.gdn_apply_state(sl["q"], sl["k"], sl["v"], sl["a"], sl["b"], sl["A_log"],
                                    sl["dt_bias"], Hin[i].contiguous())
        assert_close(f"o seg{i}", o, ro[:, s0:s1], torch.float32)
        g = gdn.gdn_apply_state_bwd(sl["q"], sl["k"], sl["v"], sl["a"], sl["b"], sl["A_log"],
                                    sl["dt_bias"], Hin[i].contiguous(), sl["dO"],
                                    dHout[i].contiguous())
        assert_close(f"dq seg{i}", g[0], rg[0][:, s0:s1], torch.float32)
        assert_close(f"dk seg{i}", g[1], rg[1][:, s0:s1], torch.float32)
        assert_close(f"dv seg{i}", g[2], rg[2][:, s0:s1], torch.float32)
        assert_close(f"dg seg{i}", g[3], rg[3][:, s0:s1], torch.float32)
        assert_close(f"dbeta seg{i}", g[4], rg[4][:, s0:s1], torch.float32)


def test_strided_segment_view_fp32():
    """A segment given by pointer offset + T_stride equals the contiguous copy."""
    w = gi.Workload("stride", B=2, T=192, Hqk=1, H=2, dk=16, dv=16, dtype=torch.float32,
                    h0_std=0.1, decay_stress=True, seed=14)
    d = dev(gi.make_inputs(w))
    s0, s1 = 64, 160
    sl = {k: (v[:, s0:s1].contiguous() if k in ("q", "k", "v", "a", "b") else v)
          for k, v in d.items()}
    M_ref, S_ref = gdn.gdn_summary(sl["k"], sl["v"], sl["a"], sl["b"], sl["A_log"],
                                   sl["dt_bias"])
    # same segment read in place from the full rows
    kk = d["k"][:, s0:]
    p = gdn.make_problem(kk, d["v"][:, s0:], T=s1 - s0, T_stride=w.T)
    M = torch.empty_like(M_ref)
    S = torch.empty_like(S_ref)
    ws = gdn.workspace(p, gdn.GDN_OP_SUMMARY)
    lib = gdn.load_library()
    import ctypes
    st = lib.gdn_summary(ctypes.byref(p), *[ctypes.c_void_p(t.data_ptr()) for t in (
        d["k"][:, s0:], d["v"][:, s0:], d["a"][:, s0:], d["b"][:, s0:])],
        ctypes.c_void_p(d["A_log"].data_ptr()), ctypes.c_void_p(d["dt_bias"].data_ptr()), None,
        ctypes.c_void_p(M.data_ptr()), ctypes.c_void_p(S.data_ptr()),
        ctypes.c_void_p(ws.data_ptr()), ws.numel(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == gdn.GDN_OK
    torch.testing.assert_close(M, M_ref, rtol=0, atol=0)
    torch.testing.assert_close(S, S_ref, rtol=0, atol=0)


def test_empty_inputs():
    for B, T in ((2, 0), (0, 5)):
        w = gi.Workload("empty", B=B, T=T, Hqk=1, H=2, dk=16, dv=16, dtype=torch.float32,
                        h0_std=0.1, with_dHT=True, seed=15)
        d = dev(gi.make_inputs(w))
        o, hT = gpu_fwd(d)
        assert o.shape == (B, T, 2, 16)
        torch.testing.assert_close(hT, d["h0"], rtol=0, atol=0)
        g = gpu_bwd(d)
        torch.testing.assert_close(g[5], d["dHT"], rtol=0, atol=0)
        M, S = gdn.gdn_summary(d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"])
        eye = torch.eye(16, device="cuda").expand_as(M)
        torch.testing.assert_close(M, eye, rtol=0, atol=0)
        assert (S == 0).all()


def test_valid_len_out_of_range_is_flagged():
    w = gi.Workload("flag", B=1, T=64, Hqk=1, H=1, dk=16, dv=16, dtype=torch.float32, seed=16)
    d = dev(gi.make_inputs(w))
    d["valid_len"] = torch.tensor([100], dtype=torch.int32, device="cuda")
    p = gdn.make_problem(d["q"], d["v"])
    ws = gdn.workspace(p, gdn.GDN_OP_FWD)
    gdn.gdn_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], None,
                d["valid_len"], ws=ws)
    assert gdn.gdn_check_device_status(ws) == gdn.GDN_ERR_INVALID_ARG
    assert gdn.gdn_check_device_status(ws) == gdn.GDN_OK     # cleared by the read
    d["valid_len"] = torch.tensor([64], dtype=torch.int32, device="cuda")
    gdn.gdn_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], None,
                d["valid_len"], ws=ws)
    assert gdn.gdn_check_device_status(ws) == gdn.GDN_OK


# ------------------------------------------------------------------ bf16 workloads

def test_cfg1_fwd_8k_bf16():
    w = gi.FWD_8K
    check_fwd_bwd(w, gi.make_inputs(w), sample=[0, 7, 15], bwd=False)


def test_cfg1_fwd_8k_bf16_decay_stress():
    w = gi.FWD_8K
    check_fwd_bwd(w, gi.make_inputs(w, decay_stress=True, seed=101), sample=[3, 12], bwd=False)


def test_cfg2_stateful_fwd_bwd_32k_bf16():
    w = gi.STATEFUL_32K
    check_fwd_bwd(w, gi.make_inputs(w), sample=[5])


def test_cfg2_stateful_32k_bf16_decay_stress_segment_counts():
    """Slow decay keeps the state alive across segments: P = 1 and P = 8 both
    match the oracle on a sampled group."""
    w = gi.STATEFUL_32K
    inp = gi.make_inputs(w, decay_stress=True, seed=102)
    for P in (1, 8):
        check_fwd_bwd(w, inp, segments=P, sample=[9])


def test_cfg3_segment_path_matches_monolithic_bf16():
    """8 segments of 4096 through the public summary / prefix / apply calls
    equal the monolithic run (and the oracle on a sampled group), forward and
    backward, with slow decay so the incoming states matter."""
    w = gi.SEGMENTED_32K
    inp = gi.make_inputs(w, decay_stress=True)
    d = dev(inp)
    o_ref, hT_ref = gpu_fwd(d)
    g_ref = gpu_bwd(d)
    L = 4096
    P = w.T // L
    seg = lambda x, i: x[:, i * L:(i + 1) * L].contiguous()  # noqa: E731
    keys = ("q", "k", "v", "a", "b", "dO")
    Ms, Ss, Ds = [], [], []
    for i in range(P):
        s = {k: seg(d[k], i) for k in keys}
        M, S = gdn.gdn_summary(s["k"], s["v"], s["a"], s["b"], d["A_log"], d["dt_bias"])
        D = gdn.gdn_summary_bwd(s["q"], s["k"], s["a"], s["b"], d["A_log"], d["dt_bias"], s["dO"])
        Ms.append(M)
        Ss.append(S)
        Ds.append(D)
    Mst, Sst, Dst = torch.stack(Ms), torch.stack(Ss), torch.stack(Ds)
    Hin, Hout = gdn.gdn_prefix_compose(Mst, Sst, d["h0"])
    dHout, dH0 = gdn.gdn_prefix_compose_bwd(Mst, Dst, d["dHT"])
    outs, grads = [], []
    for i in range(P):
        s = {k: seg(d[k], i) for k in keys}
        o, _ = gdn.gdn_apply_state(s["q"], s["k"], s["v"], s["a"], s["b"], d["A_log"],
                                   d["dt_bias"], Hin[i].contiguous(), want_hT=False)
        outs.append(o)
        grads.append(gdn.gdn_apply_state_bwd(s["q"], s["k"], s["v"], s["a"], s["b"],
                                             d["A_log"], d["dt_bias"], Hin[i].contiguous(),
                                             s["dO"], dHout[i].contiguous()))
    o_seg = torch.cat(outs, dim=1)
    assert_close("o segmented vs monolithic", o_seg, o_ref, torch.bfloat16)
    assert_close("hT segmented vs monolithic", Hout, hT_ref, torch.bfloat16)
    assert_close("dH0 segmented vs monolithic", dH0, g_ref[5], torch.bfloat16)
    for j, name in enumerate(NAMES_BWD[:5]):
        cat = torch.cat([g[j] for g in grads], dim=1)
        assert_close(f"{name} segmented vs monolithic", cat, g_ref[j], torch.bfloat16)
    # and both against the oracle on one sampled group
    r = w.H // w.Hqk
    hq = 4
    n = np64(head_slice(inp, hq, 1, r))
    ro, rhT = oracle_fwd(n)
    assert_close("o segmented vs oracle", o_seg[:, :, hq * r:(hq + 1) * r], ro, torch.bfloat16)
    assert_close("hT segmented vs oracle", Hout[:, hq * r:(hq + 1) * r], rhT, torch.bfloat16)
    # the segmented backward against the oracle's monolithic gradients, element by element
    rg = oracle_bwd(n)
    vs = slice(hq * r, (hq + 1) * r)
    for j, name in enumerate(NAMES_BWD[:5]):
        cat = torch.cat([g[j] for g in grads], dim=1)
        got = cat[:, :, hq:hq + 1] if name in ("dq", "dk") else cat[:, :, vs]
        assert_close(f"{name} segmented vs oracle", got, rg[j], torch.bfloat16)
    assert_close("dH0 segmented vs oracle", dH0[:, vs], rg[5], torch.bfloat16)
    assert_close("dHin of segment 0 vs oracle dH0", grads[0][5][:, vs], rg[5], torch.bfloat16)
    # every segment's gradient summary D against the oracle's
    for i in range(P):
        nl = {k: (n[k][:, i * L:(i + 1) * L] if k in keys else n[k]) for k in n}
        rD = oracle.summary_bwd(nl["q"], nl["k"], nl["a"], nl["b"], nl["A_log"], nl["dt_bias"],
                                nl["dO"])
        assert_close(f"D seg{i} vs oracle", Ds[i][:, vs], rD, torch.bfloat16)


def test_bf16_summary_bwd_matches_oracle():
    """The gradient summary D of a short bf16 segment (three chunks, a ragged tail)
    against the oracle, with slow decay so every chunk contributes."""
    w = gi.Workload("sumbwd", B=1, T=190, Hqk=1, H=2, dk=128, dv=128, decay_stress=True,
                    seed=41)
    inp = gi.make_inputs(w)
    n = np64(inp)
    d = dev(inp)
    D = gdn.gdn_summary_bwd(d["q"], d["k"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["dO"])
    rD = oracle.summary_bwd(n["q"], n["k"], n["a"], n["b"], n["A_log"], n["dt_bias"], n["dO"])
    assert_close("D", D, rD, torch.bfloat16)


def test_bf16_segmented_bwd_small_matches_oracle():
    """Two bf16 segments through the public summary / prefix / apply calls, forward
    and backward, compared with the oracle on every element (T = 190: a ragged tail)."""
    w = gi.Workload("segbwd", B=1, T=190, Hqk=1, H=2, dk=128, dv=128, h0_std=0.1,
                    with_dHT=True, decay_stress=True, seed=42)
    inp = gi.make_inputs(w)
    n = np64(inp)
    d = dev(inp)
    cuts = [0, 128, 190]
    keys = ("q", "k", "v", "a", "b", "dO")
    segs = [{k: d[k][:, s0:s1].contiguous() for k in keys} for s0, s1 in zip(cuts[:-1], cuts[1:])]
    Ms, Ss, Ds = [], [], []
    for s in segs:
        M, S = gdn.gdn_summary(s["k"], s["v"], s["a"], s["b"], d["A_log"], d["dt_bias"])
        Ms.append(M)
        Ss.append(S)
        Ds.append(gdn.gdn_summary_bwd(s["q"], s["k"], s["a"], s["b"], d["A_log"], d["dt_bias"],
                                      s["dO"]))
    Mst, Sst, Dst = torch.stack(Ms), torch.stack(Ss), torch.stack(Ds)
    Hin, Hout = gdn.gdn_prefix_compose(Mst, Sst, d["h0"])
    dHout, dH0 = gdn.gdn_prefix_compose_bwd(Mst, Dst, d["dHT"])
    outs, grads = [], []
    for i, s in enumerate(segs):
        outs.append(gdn.gdn_apply_state(s["q"], s["k"], s["v"], s["a"], s["b"], d["A_log"],
                                        d["dt_bias"], Hin[i].contiguous(), want_hT=False)[0])
        grads.append(gdn.gdn_apply_state_bwd(s["q"], s["k"], s["v"], s["a"], s["b"],
                                             d["A_log"], d["dt_bias"], Hin[i].contiguous(),
                                             s["dO"], dHout[i].contiguous()))
    ro, rhT = oracle_fwd(n)
    rg = oracle_bwd(n)
    assert_close("o", torch.cat(outs, dim=1), ro, torch.bfloat16)
    assert_close("hT", Hout, rhT, torch.bfloat16)
    for j, name in enumerate(NAMES_BWD[:5]):
        assert_close(name, torch.cat([g[j] for g in grads], dim=1), rg[j], torch.bfloat16)
    assert_close("dH0", dH0, rg[5], torch.bfloat16)
    assert_close("dHin of segment 0", grads[0][5], rg[5], torch.bfloat16)
    for i, (s0, s1) in enumerate(zip(cuts[:-1], cuts[1:])):
        nl = {k: (n[k][:, s0:s1] if k in keys else n[k]) for k in n}
        rD = oracle.summary_bwd(nl["q"], nl["k"], nl["a"], nl["b"], nl["A_log"], nl["dt_bias"],
                                nl["dO"])
        assert_close(f"D seg{i}", Ds[i], rD, torch.bfloat16)


def test_cfg4a_padded_batch_bf16():
    w = gi.PADDED_8K
    inp = gi.make_inputs(w, decay_stress=True)
    inp["dHT"] = None
    o, hT, g = check_fwd_bwd(w, inp, sample=[2])
    L = w.valid_len[0]
    assert (o[:, L:] == 0).all()
    for t in g[:5]:
        assert (t[:, L:] == 0).all()


def test_cfg4b_long_64k_fwd_bwd_bf16():
    w = gi.LONG_64K
    check_fwd_bwd(w, gi.make_inputs(w), sample=[11])


# ----------------------------------------------------------- determinism / stability

def test_repeat_runs_are_bitwise_identical_and_stable():
    """20 consecutive forward+backward runs: identical bits, finite, no memory
    growth (the test report's stability check, section 7)."""
    w = gi.FWD_8K
    d = dev(gi.make_inputs(gi.Workload("rep", B=1, T=8192, Hqk=16, H=32, dk=128, dv=128,
                                       h0_std=0.1, with_dHT=True, seed=21)))
    p = gdn.make_problem(d["q"], d["v"])
    wsf = gdn.workspace(p, gdn.GDN_OP_FWD)
    wsb = gdn.workspace(p, gdn.GDN_OP_BWD)
    ref = None
    mem0 = None
    for it in range(20):
        o, hT = gdn.gdn_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                            d["h0"], ws=wsf)
        g = gdn.gdn_bwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                        d["dO"], d["dHT"], d["h0"], ws=wsb)
        outs = (o, hT) + tuple(g)
        torch.cuda.synchronize()
        if ref is None:
            ref = [t.clone() for t in outs]
            mem0 = torch.cuda.memory_allocated()
            for t in ref:
                assert torch.isfinite(t.float()).all()
        else:
            for a, b in zip(outs, ref):
                assert torch.equal(a, b)
            del outs, o, hT, g
            assert torch.cuda.memory_allocated() <= mem0
    assert gdn.gdn_check_device_status(wsb) == gdn.GDN_OK
