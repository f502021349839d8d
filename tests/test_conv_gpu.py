"""GPU parity of the causal depthwise Conv1D + SiLU prologue (gdn_conv_silu_fwd / _bwd,
through the C ABI) against the fp64 oracle (oracle/conv.py).

Small cases compare every output element; the bench-size case (C = 8192 channels, the
projected q, k, v of H = 32, Hqk = 16, d = 128; T = 32768) compares sampled channels,
which are independent of one another in a depthwise convolution.  Bars as for the core:
fp32 rel-L2 <= 1e-5; bf16 rel-L2 <= 1e-2 and max-abs / ref-abs-max <= 1e-1.
"""
import numpy as np
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


def cuda(d):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}


def run_both(inp, T=None, T_stride=0):
    d = cuda(inp)
    K = inp["w"].shape[1]
    p = gdn.make_conv_problem(d["x"], K, T=T, T_stride=T_stride)
    y = gdn.gdn_conv_silu_fwd(d["x"], d["w"], d["bias"], d["halo"], problem=p)
    g = gdn.gdn_conv_silu_bwd(d["x"], d["w"], d["bias"], d["halo"], d["dy"], problem=p)
    torch.cuda.synchronize()
    return y, g


def oracle_of(inp, T):
    x, dy = to64(inp["x"])[:, :T], to64(inp["dy"])[:, :T]
    w, b, h = to64(inp["w"]), to64(inp["bias"]), to64(inp["halo"])
    return oracle.conv_silu_fwd(x, w, b, h), oracle.conv_silu_bwd(x, w, b, h, dy)


CASES = [  # dtype, B, T, C, K, halo, bias
    (torch.float32, 2, 300, 136, 4, True, True),
    (torch.float32, 1, 77, 8, 3, False, True),
    (torch.float32, 2, 513, 260, 2, True, False),
    (torch.float32, 1, 40, 12, 1, False, True),
    (torch.bfloat16, 2, 300, 136, 4, True, True),
    (torch.bfloat16, 3, 257, 512, 4, False, False),
    (torch.bfloat16, 1, 33, 128, 3, True, True),
    (torch.bfloat16, 2, 2, 64, 4, True, True),   # fewer tokens than halo rows
    (torch.bfloat16, 2, 1, 64, 4, True, True),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{'f32' if c[0] == torch.float32 else 'bf16'}"
                                             f"_B{c[1]}_T{c[2]}_C{c[3]}_K{c[4]}"
                                             f"{'_halo' if c[5] else ''}{'_bias' if c[6] else ''}"
                                             for c in CASES])
def test_conv_matches_oracle(case):
    dtype, B, T, C, K, halo, bias = case
    inp = gi.make_conv_inputs(B, T, C, K, dtype, seed=B * 1000 + T + K, halo=halo, bias=bias)
    y, (dx, dw, db, dh) = run_both(inp)
    ry, (rdx, rdw, rdb, rdh) = oracle_of(inp, T)
    assert_close("y", y, ry, dtype)
    assert_close("dx", dx, rdx, dtype)
    assert_close("dw", dw, rdw, dtype)
    assert_close("dbias", db, rdb, dtype)
    if K > 1:
        assert_close("dhalo", dh, rdh, dtype)
    else:
        assert dh is None


def test_conv_row_stride_and_segments():
    """A segment of longer rows (T_stride > T) fed the previous segment's last K - 1 tokens
    as its halo reproduces the unsplit run; its dhalo completes the first segment's dx."""
    B, T, C, K, T1 = 2, 700, 256, 4, 300
    inp = gi.make_conv_inputs(B, T, C, K, torch.float32, seed=7)
    d = cuda(inp)
    y, (dx, dw, db, dh) = run_both(inp)
    # first segment: tokens [0, T1) of the same buffers (row stride T)
    p1 = gdn.make_conv_problem(d["x"], K, T=T1, T_stride=T)
    y1 = torch.zeros_like(d["x"])
    gdn.gdn_conv_silu_fwd(d["x"], d["w"], d["bias"], d["halo"], y=y1, problem=p1)
    dx1 = torch.zeros_like(d["x"])
    _, dw1, db1, dh1 = gdn.gdn_conv_silu_bwd(d["x"], d["w"], d["bias"], d["halo"], d["dy"],
                                             dx=dx1, problem=p1)
    # second segment: its own buffers, halo = tokens T1-K+1 .. T1-1
    x2, dy2 = d["x"][:, T1:].contiguous(), d["dy"][:, T1:].contiguous()
    h2 = d["x"][:, T1 - K + 1:T1].contiguous()
    y2 = gdn.gdn_conv_silu_fwd(x2, d["w"], d["bias"], h2)
    dx2, dw2, db2, dh2 = gdn.gdn_conv_silu_bwd(x2, d["w"], d["bias"], h2, dy2)
    torch.cuda.synchronize()
    assert torch.equal(y1[:, :T1], y[:, :T1]) and (y1[:, T1:] == 0).all()
    torch.testing.assert_close(y2, y[:, T1:], rtol=1e-6, atol=1e-6)
    dx1[:, T1 - K + 1:T1] += dh2
    torch.testing.assert_close(dx1[:, :T1], dx[:, :T1], rtol=1e-5, atol=1e-5)
    assert (dx1[:, T1:] == 0).all()
    torch.testing.assert_close(dx2, dx[:, T1:], rtol=1e-6, atol=1e-6)
    torch.testing.assert_close(dh1, dh, rtol=1e-6, atol=1e-6)
    torch.testing.assert_close(dw1 + dw2, dw, rtol=1e-5, atol=1e-5)
    torch.testing.assert_close(db1 + db2, db, rtol=1e-5, atol=1e-5)


def test_conv_deterministic_and_empty():
    inp = gi.make_conv_inputs(2, 600, 128, 4, torch.bfloat16, seed=11)
    a = run_both(inp)
    b = run_both(inp)
    assert torch.equal(a[0], b[0])
    for u, v in zip(a[1], b[1]):
        assert torch.equal(u, v)
    # no tokens: nothing written forward; zero dw, dbias and dhalo backward
    d = cuda(gi.make_conv_inputs(2, 0, 64, 4, torch.bfloat16, seed=12))
    dx, dw, db, dh = gdn.gdn_conv_silu_bwd(d["x"], d["w"], d["bias"], d["halo"], d["dy"])
    torch.cuda.synchronize()
    assert (dw == 0).all() and (db == 0).all() and (dh == 0).all()


def test_conv_bench_size_sampled_channels():
    """B = 1, T = 32768, C = 8192 bf16 (the bench size), K = 4 with a halo: every output of
    32 sampled channels against the oracle, plus finiteness of everything."""
    B, T, C, K = 1, 32768, 8192, 4
    inp = gi.make_conv_inputs(B, T, C, K, torch.bfloat16, seed=5)
    y, (dx, dw, db, dh) = run_both(inp)
    for t in (y, dx, dw, db, dh):
        assert torch.isfinite(t.float()).all()
    cs = np.linspace(0, C - 1, 32).astype(int)
    sub = {k: (v[..., cs] if (torch.is_tensor(v) and k != "w") else v) for k, v in inp.items()}
    sub["w"] = inp["w"][cs]
    ry, (rdx, rdw, rdb, rdh) = oracle_of(sub, T)
    assert_close("y", y[..., cs], ry, torch.bfloat16)
    assert_close("dx", dx[..., cs], rdx, torch.bfloat16)
    assert_close("dw", dw[cs], rdw, torch.bfloat16)
    assert_close("dbias", db[cs], rdb, torch.bfloat16)
    assert_close("dhalo", dh[..., cs], rdh, torch.bfloat16)
