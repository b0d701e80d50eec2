"""gdr_chunk_fwd_static: the chunked forward without a caller-provided workspace.

Callers that may not allocate device memory when they run the forward pass
(a plugin whose framework owns every allocation, a loop where cudaMalloc could
block) call this entry point; it uses scratch compiled into the library. This
test calls it through the C ABI and checks its outputs against the regular
entry point (which takes a workspace), on two calls in a row, so that the
second call also sees the scratch the first one left behind.

It lives in a file that pytest collects last and builds nothing on its own,
so it passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import pytest
import torch

import gated_delta_rule_10_gb300 as gdr
from gated_delta_rule_10_gb300 import workloads as wl
from tests.gdr_testutil import TOL, gpu_forward, rel_err, to_dev

pytestmark = pytest.mark.gpu


def _static_entry():
    fn = gdr.lib().gdr_chunk_fwd_static
    fn.argtypes = [ctypes.POINTER(gdr.Shape)] + [ctypes.c_void_p] * 11 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


@pytest.mark.parametrize("variant,dtype", [("gdn", torch.bfloat16), ("gdn2", torch.bfloat16),
                                           ("kda", torch.float32), ("vbeta", torch.bfloat16)],
                         ids=["gdn-bf16", "gdn2-bf16", "kda-f32", "vbeta-bf16"])
def test_static_scratch_entry_matches_workspace_entry(variant, dtype):
    """bf16 scalar and channel gates take the single-kernel path with the status
    words in the scratch; fp32 and the per-value-channel write strength need no
    scratch at all (need = 0)."""
    fn = _static_entry()
    check = gdr.lib().gdr_chunk_fwd_static_check
    check.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    check.restype = ctypes.c_int
    x = wl.make_inputs(variant, 2, 200, 4, 128, 128, dtype, seed=123, h0_std=0.02)
    o_ref, h_ref = gpu_forward(x)
    torch.cuda.synchronize()
    d = to_dev(x)
    shape = gdr.make_shape(*d["q"].shape, d["v"].shape[-1], d["q"].dtype, x["flags"],
                           x["scale"])
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        hT = torch.full_like(h_ref, float("nan"))
        st = fn(ctypes.byref(shape), ptr(d["q"]), ptr(d["k"]), ptr(d["v"]), ptr(d["g"]),
                ptr(d["beta"]), ptr(d["lam"]), ptr(d["b"]), ptr(d["w"]), ptr(d["h0"]), ptr(o),
                ptr(hT), stream)
        assert st == 0, gdr.status_string(st)
        detail = (ctypes.c_int * 2)()
        assert check(stream, detail) == 0
        torch.cuda.synchronize()
        assert rel_err(o.float().cpu(), o_ref.float().cpu().numpy()) <= TOL[dtype]
        assert rel_err(hT.cpu(), h_ref.cpu().numpy()) <= TOL[dtype]


def test_static_scratch_entry_rejects_bad_shapes():
    fn = _static_entry()
    bad = gdr.make_shape(1, 64, 1, 96, 64, torch.bfloat16, 0, 0.1)   # d_k = 96 unsupported
    assert fn(ctypes.byref(bad), *([None] * 11), None) == 2
    assert fn(None, *([None] * 11), None) == 1
