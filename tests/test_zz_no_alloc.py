"""gdn_fwd_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc or hand the library a workspace -- code that
runs while a stream is captured into a CUDA graph, or an operator plugin of an
inference runtime that offers no workspace hook.  gdn_fwd_noalloc serves them
with a fixed static device scratch array instead of a workspace.  These tests
call it through the C ABI and compare it with gdn_fwd on two calls in a row.
The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import chunked_state_scan_gated_gb300 as gdn
from chunked_state_scan_gated_gb300 import inputs as gi
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu


def vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(p, d, o, hT):
    lib = gdn.load_library()
    return lib.gdn_fwd_noalloc(ctypes.byref(p), vp(d["q"]), vp(d["k"]), vp(d["v"]), vp(d["a"]),
                               vp(d["b"]), vp(d["A_log"]), vp(d["dt_bias"]), vp(d["h0"]),
                               vp(d["valid_len"]), vp(o), vp(hT),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    gi.Workload("noalloc_fp32", B=1, T=128, Hqk=4, H=8, dk=16, dv=16, dtype=torch.float32,
                h0_std=0.1, segments=2, decay_stress=True, seed=31),
    gi.Workload("noalloc_bf16", B=2, T=500, Hqk=2, H=4, dk=128, dv=128, h0_std=0.1,
                valid_len=[500, 333], seed=32),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_noalloc_matches_workspace_forward_twice(w):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in gi.make_inputs(w).items()}
    p = gdn.make_problem(d["q"], d["v"], segments=w.segments)
    assert gdn.gdn_workspace_size(p, gdn.GDN_OP_FWD) <= gdn.GDN_NOALLOC_SCRATCH_BYTES
    ref_o, ref_hT = gdn.gdn_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"],
                                d["dt_bias"], d["h0"], d["valid_len"], segments=w.segments)
    for _ in range(2):
        o = torch.full_like(ref_o, float("nan"))
        hT = torch.full_like(ref_hT, float("nan"))
        assert call_noalloc(p, d, o, hT) == gdn.GDN_OK
        torch.cuda.synchronize()
        assert_close("o (no-alloc vs workspace)", o, ref_o, w.dtype)
        assert_close("hT (no-alloc vs workspace)", hT, ref_hT, w.dtype)


def test_noalloc_rejects_problems_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    q = torch.empty(1, 32768, 16, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.empty(1, 32768, 32, 128, dtype=torch.bfloat16, device="cuda")
    p = gdn.make_problem(q, v)
    assert gdn.gdn_workspace_size(p, gdn.GDN_OP_FWD) > gdn.GDN_NOALLOC_SCRATCH_BYTES
    d = {"q": q, "k": q, "v": v, "a": v, "b": v, "A_log": v, "dt_bias": v, "h0": None,
         "valid_len": None}
    assert call_noalloc(p, d, v, None) == gdn.GDN_ERR_UNSUPPORTED


def test_noalloc_device_status_reports_a_clamped_valid_len():
    """A valid_len outside [0, T] (a bad input made on the host, not a fault) is
    clamped by the kernels and recorded in the static scratch's status word, which
    gdn_noalloc_check_device_status reads and clears."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = gi.Workload("noalloc_flag", B=1, T=64, Hqk=1, H=1, dk=16, dv=16, dtype=torch.float32,
                    seed=33)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in gi.make_inputs(w).items()}
    p = gdn.make_problem(d["q"], d["v"])
    o = torch.empty_like(d["v"])
    hT = torch.empty(1, 1, 16, 16, device="cuda")
    assert gdn.gdn_noalloc_check_device_status() == gdn.GDN_OK   # clears earlier calls' word
    d["valid_len"] = torch.tensor([100], dtype=torch.int32, device="cuda")
    assert call_noalloc(p, d, o, hT) == gdn.GDN_OK
    assert gdn.gdn_noalloc_check_device_status() == gdn.GDN_ERR_INVALID_ARG
    assert gdn.gdn_noalloc_check_device_status() == gdn.GDN_OK   # cleared by the read
    d["valid_len"] = torch.tensor([64], dtype=torch.int32, device="cuda")
    assert call_noalloc(p, d, o, hT) == gdn.GDN_OK
    assert gdn.gdn_noalloc_check_device_status() == gdn.GDN_OK
