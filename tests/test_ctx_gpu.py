"""GPU parity of the forward-context calls (gdn_fwd_ctx / gdn_bwd_ctx) through the C ABI.

gdn_fwd_ctx must give exactly gdn_fwd's outputs (it runs the same kernels, plus
the summary of the last segment); gdn_bwd_ctx must match the fp64 oracle under the
same bars as gdn_bwd, at small sizes on every element and at T = 32K on a sampled
Q/K group."""
import pytest
import torch

import chunked_state_scan_gated_gb300 as gdn
from chunked_state_scan_gated_gb300 import inputs as gi
from tests.helpers import assert_close, head_slice
from tests.test_parity_gpu import NAMES_BWD, dev, np64, oracle_bwd, oracle_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load_library()


def run_ctx(d, segments):
    o, hT = gdn.gdn_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                        d["h0"], d["valid_len"], segments=segments)
    o2, hT2, ctx = gdn.gdn_fwd_ctx(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"],
                                   d["dt_bias"], d["h0"], d["valid_len"], segments=segments)
    grads = gdn.gdn_bwd_ctx(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                            ctx, d["dO"], d["dHT"], d["valid_len"], segments=segments)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(hT, hT2)
    return o2, hT2, grads


def check(w, inp, segments, sample=None):
    d = dev(inp)
    o, hT, grads = run_ctx(d, segments)
    r = w.H // w.Hqk
    groups = [(0, w.Hqk)] if sample is None else [(hq, 1) for hq in sample]
    for hq0, nq in groups:
        n = np64(head_slice(inp, hq0, nq, r))
        h0s, h1s = hq0 * r, (hq0 + nq) * r
        ro, rhT = oracle_fwd(n)
        assert_close("o", o[:, :, h0s:h1s], ro, w.dtype)
        assert_close("hT", hT[:, h0s:h1s], rhT, w.dtype)
        ref = oracle_bwd(n)
        got = (grads[0][:, :, hq0:hq0 + nq], grads[1][:, :, hq0:hq0 + nq],
               grads[2][:, :, h0s:h1s], grads[3][:, :, h0s:h1s], grads[4][:, :, h0s:h1s],
               grads[5][:, h0s:h1s])
        for name, g, rg in zip(NAMES_BWD, got, ref):
            if name == "dH0" and inp["h0"] is None:
                continue
            assert_close(name, g, rg, w.dtype)
    return grads


CASES = [
    # name, dtype, B, T, Hqk, H, dk, segments, h0_std, valid_len, stress
    ("fp32_seg2", torch.float32, 1, 128, 4, 8, 16, 2, 0.1, None, True),
    ("fp32_seg1", torch.float32, 2, 65, 2, 4, 32, 1, 0.1, None, True),
    ("fp32_padded_seg3", torch.float32, 2, 200, 2, 4, 16, 3, 0.1, [97, 3], False),
    ("bf16_seg3", torch.bfloat16, 2, 200, 1, 2, 128, 3, 0.1, None, True),
    ("bf16_seg1_no_h0", torch.bfloat16, 1, 64, 1, 2, 128, 1, None, None, False),
    ("bf16_padded_seg2", torch.bfloat16, 2, 300, 1, 2, 128, 2, 0.1, [300, 97], True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_ctx_matches_oracle(case):
    name, dtype, B, T, Hqk, H, dk, seg, h0s, vl, stress = case
    w = gi.Workload(name, B=B, T=T, Hqk=Hqk, H=H, dk=dk, dv=dk, dtype=dtype, h0_std=h0s,
                    with_dHT=h0s is not None, valid_len=vl, decay_stress=stress, seed=29)
    grads = check(w, gi.make_inputs(w), seg)
    if vl is not None:
        for bi, Lb in enumerate(vl):
            assert (grads[2][bi, Lb:] == 0).all() and (grads[3][bi, Lb:] == 0).all()


def test_ctx_matches_recompute_bwd_bf16():
    """gdn_bwd_ctx and gdn_bwd agree (bf16 bars) on the same inputs."""
    w = gi.Workload("ctx_vs_bwd", B=1, T=640, Hqk=2, H=4, dk=128, dv=128, dtype=torch.bfloat16,
                    h0_std=0.1, with_dHT=True, decay_stress=True, seed=31)
    inp = gi.make_inputs(w)
    d = dev(inp)
    _, _, g_ctx = run_ctx(d, 4)
    g = gdn.gdn_bwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["dO"],
                    d["dHT"], d["h0"], d["valid_len"], segments=4)
    torch.cuda.synchronize()
    for name, x, y in zip(NAMES_BWD, g_ctx, g):
        assert_close(name, x, y.double().cpu().numpy(), torch.bfloat16)


def test_ctx_stateful_32k_bf16():
    w = gi.STATEFUL_32K
    check(w, gi.make_inputs(w, decay_stress=True, seed=103), 0, sample=[11])
