"""Parity of kda_recurrent_verify (CUDA, through the C ABI) with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from kda_linear_attention_bounded_gb300 import inputs
import kda_linear_attention_bounded_gb300 as kda
from gpu_helpers import DeviceVerify, check_out, check_state

pytestmark = pytest.mark.gpu


def _parity(inp, head_groups=1):
    dev = DeviceVerify(inp)
    pool_before = dev.pool.clone()
    ws = kda.make_workspace()
    out, inter = dev.run(workspace=ws)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    assert torch.equal(dev.pool, pool_before), "verify must not write the pool"
    H = inp.H
    step = H // head_groups
    for hb in range(0, H, step):
        he = hb + step
        ref_out, ref_steps = oracle.run_verify(inp, heads=(hb, he))
        check_out(out[:, hb:he], ref_out[:, hb:he], f"{inp.name} outputs heads {hb}:{he}")
        check_state(inter[:, :, hb:he], ref_steps[:, :, hb:he], f"{inp.name} per-step states heads {hb}:{he}")


def test_verify_64x8_h16_full():
    _parity(inputs.verify_64x8(), head_groups=4)


@pytest.mark.parametrize("T", [1, 3, 8, 17])
def test_verify_small(T):
    _parity(inputs.verify_inputs("small", 3, T, 2, seed=60 + T, pool_slots=5))


def test_verify_repeated_slots_and_weak_decay():
    inp = inputs.verify_inputs("rep", 4, 8, 2, seed=70, pool_slots=3, g_mean=-8.0)
    inp.slot_ids = np.array([1, 1, 2, 1], np.int32)
    _parity(inp)


def test_verify_bad_slot():
    inp = inputs.verify_inputs("bad", 2, 4, 2, seed=80, pool_slots=3)
    dev = DeviceVerify(inp)
    dev.slots[0] = -1
    ws = kda.make_workspace()
    out = torch.full((8, 2, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    out, inter = dev.run(workspace=ws, out=out)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) & kda.KDA_DEVICE_BAD_SLOT
    assert (out[:4].float() == 3.0).all()
    ref_out, ref_steps = oracle.run_verify(inp)
    check_out(out[4:], ref_out[4:], "good request next to a bad slot")
    check_state(inter[1], ref_steps[1], "good request states")
