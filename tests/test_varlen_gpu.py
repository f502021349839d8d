"""GPU parity of the packed variable-length calls (gdn_fwd_varlen / gdn_bwd_varlen)
through the C ABI against the fp64 oracle's packed-row functions: every output and
gradient, at small sizes on every element (empty sequences, a one-token sequence,
sequences ending inside and on a chunk boundary), and on a 32K-token row of eight mixed
lengths at H = 32 on sampled Q/K groups."""
import pytest
import torch

import chunked_state_scan_gated_gb300 as gdn
from chunked_state_scan_gated_gb300 import inputs as gi
import oracle
from tests.helpers import assert_close, head_slice

pytestmark = pytest.mark.gpu

NAMES_BWD = ("dq", "dk", "dv", "dg", "dbeta", "dH0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load_library()


def dev(inp):
    return {k: (v.cuda() if torch.is_tensor(v) and k != "cu_seqlens" else v)
            for k, v in inp.items()}


def varlen_slice(inp, hq0, nq, r):
    """head_slice for packed inputs: states are [N, H, dk, dv]."""
    out = head_slice({k: v for k, v in inp.items() if k not in ("h0", "dHT", "cu_seqlens")},
                     hq0, nq, r)
    h0s, h1s = hq0 * r, (hq0 + nq) * r
    for key in ("h0", "dHT"):
        out[key] = None if inp[key] is None else inp[key][:, h0s:h1s]
    out["cu_seqlens"] = inp["cu_seqlens"]
    return out


def check(w, lengths, sample=None, with_bwd=True, segments=0):
    inp = gi.make_varlen_inputs(w, lengths)
    d = dev(inp)
    cu = gdn.Varlen(inp["cu_seqlens"])
    fin = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"])
    o, hT = gdn.gdn_fwd_varlen(*fin, cu, d["h0"], segments=segments)
    grads = gdn.gdn_bwd_varlen(*fin, cu, d["dO"], d["dHT"], d["h0"],
                               segments=segments) if with_bwd else None
    torch.cuda.synchronize()
    r = w.H // w.Hqk
    groups = [(0, w.Hqk)] if sample is None else [(hq, 1) for hq in sample]
    for hq0, nq in groups:
        n = gi.to_numpy64(varlen_slice(inp, hq0, nq, r))
        h0s, h1s = hq0 * r, (hq0 + nq) * r
        args = (n["q"], n["k"], n["v"], n["a"], n["b"], n["A_log"], n["dt_bias"],
                n["cu_seqlens"])
        ro, rhT = oracle.fwd_varlen(*args, h0=n["h0"])
        assert_close("o", o[:, :, h0s:h1s], ro, w.dtype)
        assert_close("hT", hT[:, h0s:h1s], rhT, w.dtype)
        if not with_bwd:
            continue
        ref = oracle.bwd_varlen(*args, n["dO"], n["dHT"], h0=n["h0"])
        got = (grads[0][:, :, hq0:hq0 + nq], grads[1][:, :, hq0:hq0 + nq],
               grads[2][:, :, h0s:h1s], grads[3][:, :, h0s:h1s], grads[4][:, :, h0s:h1s],
               grads[5][:, h0s:h1s])
        for name, g, rg in zip(NAMES_BWD, got, ref):
            assert_close(name, g, rg, w.dtype)
    return o, hT, grads


SMALL = [1, 63, 0, 64, 65, 190, 0, 117]   # 500 tokens, boundaries inside and on chunks


def test_varlen_bf16_small_matches_oracle():
    w = gi.Workload("varlen_bf16", B=1, T=0, Hqk=1, H=2, dk=128, dv=128, h0_std=0.1,
                    with_dHT=True, seed=61)
    check(w, SMALL)


def test_varlen_bf16_segmented_matches_oracle():
    """The padded batch split into time segments (prefix compose inside each row)."""
    w = gi.Workload("varlen_bf16_seg", B=1, T=0, Hqk=2, H=4, dk=128, dv=128, h0_std=0.1,
                    with_dHT=True, decay_stress=True, seed=62)
    check(w, [300, 5, 420, 129], segments=3)


def test_varlen_fp32_small_matches_oracle():
    w = gi.Workload("varlen_fp32", B=1, T=0, Hqk=2, H=4, dk=16, dv=32, dtype=torch.float32,
                    h0_std=0.1, with_dHT=True, seed=63)
    check(w, SMALL)


def test_varlen_without_states_and_single_sequence():
    """No h0 / dHT; one sequence over the whole row equals gdn_fwd on that row."""
    w = gi.Workload("varlen_plain", B=1, T=0, Hqk=1, H=2, dk=128, dv=128, seed=64)
    o, hT, _ = check(w, [7, 200, 33])
    inp = gi.make_varlen_inputs(w, [240])
    d = dev(inp)
    fin = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"])
    o1, hT1 = gdn.gdn_fwd_varlen(*fin, inp["cu_seqlens"], None)
    o2, hT2 = gdn.gdn_fwd(*fin, None, None)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(hT1, hT2)


def test_varlen_32k_mixed_lengths_sampled():
    """A 32K-token row of eight sequences of mixed length at the bench's head count."""
    w = gi.Workload("varlen_bf16_32k", B=1, T=0, Hqk=16, H=32, dk=128, dv=128, h0_std=0.1,
                    with_dHT=True, grad_scale="numel", seed=65)
    check(w, gi.length_mix(32768, 8, seed=65), sample=[11])


def test_varlen_device_offsets_disagreeing_with_host_are_reported():
    """A device copy of the offsets with a sequence longer than the host copy's longest is
    skipped (no access outside the buffers) and reported by the status call."""
    w = gi.Workload("varlen_bad", B=1, T=0, Hqk=1, H=2, dk=128, dv=128, seed=66)
    inp = gi.make_varlen_inputs(w, [100, 100])
    d = dev(inp)
    cu = gdn.Varlen(inp["cu_seqlens"])
    cu.dev = torch.tensor([0, 150, 200], dtype=torch.int32, device="cuda")
    p = gdn.make_problem(d["q"], d["v"])
    ws = gdn.varlen_workspace(p, cu, gdn.GDN_OP_FWD)
    fin = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"])
    gdn.gdn_fwd_varlen(*fin, cu, None, ws=ws, problem=p)
    assert gdn.gdn_varlen_check_device_status(ws, p, cu, gdn.GDN_OP_FWD) == \
        gdn.GDN_ERR_INVALID_ARG
    assert gdn.gdn_varlen_check_device_status(ws, p, cu, gdn.GDN_OP_FWD) == gdn.GDN_OK
