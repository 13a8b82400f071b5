"""kda_recurrent_verify_noalloc against kda_recurrent_verify.

The no-allocation entry point serves callers that cannot hand the library a
workspace (their device memory is planned ahead, or they must not call
cudaMalloc because it can synchronise the device); it keeps its scratch in a
fixed device array inside libkda.  Both entry points run the same verify
kernel on the same inputs, so their results must agree bit for bit.  The test
calls it through the C ABI twice in a row -- the second call sees whatever the
first left in that shared array -- with one padding row (slot id -1) and one
out-of-range slot id among the requests: both calls must return KDA_OK, write
exactly the rows the regular call writes and leave the skipped requests' rows
as they were.  It lives in its own file, collected last.
"""
import ctypes

import pytest
import torch

import kda_linear_attention_bounded_gb300 as kda
from kda_linear_attention_bounded_gb300 import inputs
from gpu_helpers import DeviceVerify

pytestmark = pytest.mark.gpu

OUT_FILL = 3.0     # value of output rows the calls must not write
STATE_FILL = 7.0   # value of per-step state rows the calls must not write


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
    num_slots = dev.pool.shape[0]
    dev.slots[1] = kda.KDA_PAD_SLOT_ID     # a padding row of a bucketed batch: skipped, no report
    dev.slots[3] = num_slots               # out of range: skipped (the regular call also sets a status bit)
    rows = inp.B * inp.T

    def fresh():
        return (torch.full((rows, inp.H, 128), OUT_FILL, dtype=torch.bfloat16, device="cuda"),
                torch.full((inp.B, inp.T, inp.H, 128, 128), STATE_FILL, dtype=torch.float32, device="cuda"))

    ref_out, ref_inter = fresh()
    dev.run(out=ref_out, intermediate_states=ref_inter)   # regular entry point, caller-provided workspace
    torch.cuda.synchronize()
    for b in (1, 3):
        assert (ref_out[b * inp.T:(b + 1) * inp.T].float() == OUT_FILL).all()
        assert (ref_inter[b] == STATE_FILL).all()

    fn = _noalloc_fn()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out, inter = fresh()
        rc = fn(p(dev.q), p(dev.k), p(dev.v), dev.q.stride(0), p(dev.g), dev.g.stride(0), p(dev.beta),
                dev.beta.stride(0), p(dev.A_log), p(dev.dt_bias), inp.lower_bound, inp.scale, inp.B, inp.T, inp.H,
                p(dev.pool), num_slots, p(dev.slots), p(out), out.stride(0), p(inter), stream)
        assert rc == kda.KDA_OK, kda.status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), f"no-alloc call {call}: outputs differ from the workspace call's"
        assert torch.equal(inter, ref_inter), f"no-alloc call {call}: per-step states differ from the workspace call's"


def test_noalloc_verify_rejects_bad_arguments_before_queuing_work():
    # a call the host checks reject returns its status and leaves the outputs untouched
    inp = inputs.verify_inputs("noalloc_bad", 2, 4, 2, seed=98, pool_slots=3)
    dev = DeviceVerify(inp)
    out = torch.full((inp.B * inp.T, inp.H, 128), OUT_FILL, dtype=torch.bfloat16, device="cuda")
    inter = torch.full((inp.B, inp.T, inp.H, 128, 128), STATE_FILL, dtype=torch.float32, device="cuda")
    fn = _noalloc_fn()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fn(p(dev.q), p(dev.k), p(dev.v), dev.q.stride(0), p(dev.g), dev.g.stride(0), p(dev.beta),
            dev.beta.stride(0), p(dev.A_log), p(dev.dt_bias), -11.0, inp.scale, inp.B, inp.T, inp.H,
            p(dev.pool), dev.pool.shape[0], p(dev.slots), p(out), out.stride(0), p(inter), stream)
    assert rc == kda.KDA_ERR_UNSUPPORTED
    rc = fn(p(dev.q), p(dev.k), p(dev.v), dev.q.stride(0), p(dev.g), dev.g.stride(0), p(dev.beta),
            dev.beta.stride(0), p(dev.A_log), p(dev.dt_bias), inp.lower_bound, inp.scale, inp.B, 65, inp.H,
            p(dev.pool), dev.pool.shape[0], p(dev.slots), p(out), out.stride(0), p(inter), stream)
    assert rc == kda.KDA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (out.float() == OUT_FILL).all() and (inter == STATE_FILL).all()
