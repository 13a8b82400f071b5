"""kda_recurrent_verify_noalloc against kda_recurrent_verify.

The no-allocation entry point serves callers that cannot hand the library a
workspace (their device memory is planned ahead, or they must not call
cudaMalloc because it can synchronise the device); it keeps its scratch in a
fixed device array inside libkda.  This test calls it through the C ABI twice
in a row -- the second call sees whatever the first left in that shared array
-- and checks both results against the regular entry point, with the parity
tolerances used everywhere else.  It lives in its own file, collected last.
"""
import ctypes

import pytest
import torch

import kda_linear_attention_bounded_gb300 as kda
from kda_linear_attention_bounded_gb300 import inputs
from gpu_helpers import DeviceVerify, check_out, check_state

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    lib = kda.load()
    fn = lib.kda_recurrent_verify_noalloc
    P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    fn.argtypes = [P, P, P, I64, P, I64, P, I64, P, P, F, F, I, I, I, P, I, P, P, I64, P, P]
    fn.restype = I
    return fn


def test_noalloc_verify_matches_workspace_verify_twice():
    inp = inputs.verify_inputs("noalloc", 5, 8, 4, seed=97, pool_slots=7)
    dev = DeviceVerify(inp)
    ref_out, ref_inter = dev.run()          # regular entry point, caller-provided workspace
    torch.cuda.synchronize()
    fn = _noalloc_fn()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        inter = torch.full_like(ref_inter, float("nan"))
        rc = fn(p(dev.q), p(dev.k), p(dev.v), dev.q.stride(0), p(dev.g), dev.g.stride(0), p(dev.beta),
                dev.beta.stride(0), p(dev.A_log), p(dev.dt_bias), inp.lower_bound, inp.scale, inp.B, inp.T, inp.H,
                p(dev.pool), dev.pool.shape[0], p(dev.slots), p(out), out.stride(0), p(inter), stream)
        assert rc == kda.KDA_OK, kda.status_string(rc)
        torch.cuda.synchronize()
        check_out(out, ref_out.float().cpu().numpy(), f"no-alloc call {call} outputs")
        check_state(inter, ref_inter.cpu().numpy(), f"no-alloc call {call} per-step states")
