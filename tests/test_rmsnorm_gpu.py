"""GPU parity of the gated RMSNorm epilogue (gdn_rmsnorm_gated_fwd / _bwd, through the C
ABI) against the fp64 oracle (oracle/rmsnorm.py): every element of small cases, sampled
rows of the bench-size case (o of B = 1, T = 32768, H = 32, dv = 128; rows are independent,
and dw is checked as a whole against the oracle's sum over all rows).  Bars as for the core:
fp32 rel-L2 <= 1e-5; bf16 rel-L2 <= 1e-2 and max-abs / ref-abs-max <= 1e-1."""
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


def run(inp, eps=1e-6):
    d = {k: v.cuda() for k, v in inp.items()}
    y = gdn.gdn_rmsnorm_gated_fwd(d["o"], d["z"], d["w"], eps)
    g = gdn.gdn_rmsnorm_gated_bwd(d["o"], d["z"], d["w"], d["dy"], eps)
    torch.cuda.synchronize()
    return y, g


CASES = [(torch.float32, (2, 37, 3, 128)), (torch.float32, (1, 9, 2, 64)),
         (torch.float32, (3, 5, 260)), (torch.bfloat16, (2, 300, 4, 128)),
         (torch.bfloat16, (1, 17, 2, 512)), (torch.bfloat16, (4, 12)),
         (torch.bfloat16, (1, 1, 1, 128))]


@pytest.mark.parametrize("case", CASES, ids=[f"{'f32' if c[0] == torch.float32 else 'bf16'}_"
                                             + "x".join(map(str, c[1])) for c in CASES])
def test_rmsnorm_matches_oracle(case):
    dtype, shape = case
    inp = gi.make_rmsnorm_inputs(shape, dtype, seed=len(shape) * 100 + shape[-1])
    y, (do, dz, dw) = run(inp)
    o, z, w, dy = (to64(inp[k]) for k in ("o", "z", "w", "dy"))
    assert_close("y", y, oracle.rmsnorm_gated_fwd(o, z, w), dtype)
    rdo, rdz, rdw = oracle.rmsnorm_gated_bwd(o, z, w, dy)
    assert_close("do", do, rdo, dtype)
    assert_close("dz", dz, rdz, dtype)
    assert_close("dw", dw, rdw, dtype)


def test_rmsnorm_deterministic_and_empty():
    inp = gi.make_rmsnorm_inputs((2, 500, 4, 128), torch.bfloat16, seed=3)
    a, b = run(inp), run(inp)
    assert torch.equal(a[0], b[0])
    for u, v in zip(a[1], b[1]):
        assert torch.equal(u, v)
    e = gi.make_rmsnorm_inputs((0, 128), torch.bfloat16, seed=4)
    _, (_, _, dw) = run(e)
    assert (dw == 0).all()


def test_rmsnorm_bench_size_sampled_rows():
    shape = (1, 32768, 32, 128)
    inp = gi.make_rmsnorm_inputs(shape, torch.bfloat16, seed=6)
    y, (do, dz, dw) = run(inp)
    for t in (y, do, dz, dw):
        assert torch.isfinite(t.float()).all()
    ts = np.linspace(0, shape[1] - 1, 64).astype(int)
    sub = {k: (v[:, ts] if k != "w" else v) for k, v in inp.items()}
    o, z, w, dy = (to64(sub[k]) for k in ("o", "z", "w", "dy"))
    assert_close("y", y[:, ts], oracle.rmsnorm_gated_fwd(o, z, w), torch.bfloat16)
    rdo, rdz, _ = oracle.rmsnorm_gated_bwd(o, z, w, dy)
    assert_close("do", do[:, ts], rdo, torch.bfloat16)
    assert_close("dz", dz[:, ts], rdz, torch.bfloat16)
    # dw over all 1M rows: the oracle's sum in fp64, chunked to bound host memory
    ref = np.zeros(128)
    for t0 in range(0, shape[1], 4096):
        part = {k: to64(inp[k][:, t0:t0 + 4096]) for k in ("o", "z", "dy")}
        ref += oracle.rmsnorm_gated_bwd(part["o"], part["z"], to64(inp["w"]), part["dy"])[2]
    assert_close("dw", dw, ref, torch.bfloat16)
