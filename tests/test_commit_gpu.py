"""kda_commit_accepted: after verify, the pool slot of request b holds the state
after its last accepted draft token (bit-exact copy of the per-step record, and
within the state tolerance of the fp64 oracle's state after that token)."""
import numpy as np
import pytest
import torch

import oracle
from kda_linear_attention_bounded_gb300 import inputs
import kda_linear_attention_bounded_gb300 as kda
from gpu_helpers import DeviceVerify, check_state, i32_dev

pytestmark = pytest.mark.gpu


def _run(inp, n_acc, heads=None):
    dev = DeviceVerify(inp)
    pool_before = dev.pool.clone()
    ws = kda.make_workspace()
    _, inter = dev.run(workspace=ws)
    n_dev = i32_dev(np.asarray(n_acc))
    kda.commit_accepted(dev.pool, dev.slots, n_dev, inter, workspace=ws)
    torch.cuda.synchronize()
    return dev, pool_before, inter, ws


@pytest.mark.parametrize("T", [1, 8])
def test_commit_small(T):
    inp = inputs.verify_inputs("commit", 6, T, 4, seed=110 + T, pool_slots=9)
    n_acc = np.array([0, 1, T, max(1, T // 2), T, 0], np.int32)
    dev, before, inter, ws = _run(inp, n_acc)
    assert kda.read_device_status(ws) == 0
    _, ref_steps = oracle.run_verify(inp)
    slots = torch.from_numpy(inp.slot_ids).long().cuda()
    for b, n in enumerate(n_acc):
        got = dev.pool[slots[b]]
        if n == 0:
            assert torch.equal(got, before[slots[b]]), f"request {b}: slot changed with no accepted token"
        else:
            assert torch.equal(got, inter[b, n - 1]), f"request {b}: not the state after token {n - 1}"
            check_state(got, ref_steps[b, n - 1], f"request {b} committed state vs oracle")
    others = np.setdiff1d(np.arange(inp.pool.shape[0]), inp.slot_ids)
    idx = torch.from_numpy(others).long().cuda()
    assert torch.equal(dev.pool[idx], before[idx]), "slots of no request changed"


def test_commit_bad_count_and_slot():
    inp = inputs.verify_inputs("commit_bad", 3, 4, 2, seed=120, pool_slots=5)
    dev = DeviceVerify(inp)
    ws = kda.make_workspace()
    _, inter = dev.run(workspace=ws)
    before = dev.pool.clone()
    n_dev = i32_dev(np.array([5, 2, 1], np.int32))      # 5 > T = 4
    dev.slots[2] = 17                                      # out of range
    kda.commit_accepted(dev.pool, dev.slots, n_dev, inter, workspace=ws)
    torch.cuda.synchronize()
    st = kda.read_device_status(ws)
    assert st & kda.KDA_DEVICE_BAD_COUNT and st & kda.KDA_DEVICE_BAD_SLOT
    s0, s1 = int(inp.slot_ids[0]), int(inp.slot_ids[1])
    assert torch.equal(dev.pool[s0], before[s0]), "skipped request must not write its slot"
    assert torch.equal(dev.pool[s1], inter[1, 1]), "valid request next to bad ones is committed"


def test_commit_verify_64x8_full():
    inp = inputs.verify_64x8()
    rng = np.random.default_rng(5)
    n_acc = rng.integers(1, 9, size=inp.B).astype(np.int32)
    dev, before, inter, ws = _run(inp, n_acc)
    assert kda.read_device_status(ws) == 0
    slots = torch.from_numpy(inp.slot_ids).long().cuda()
    n_t = torch.from_numpy(n_acc).long().cuda()
    expect = inter[torch.arange(inp.B, device="cuda"), n_t - 1]
    assert torch.equal(dev.pool[slots], expect)
    _, ref_steps = oracle.run_verify(inp, heads=(0, 2))
    got = dev.pool[slots][:, 0:2].cpu().numpy()
    ref = ref_steps[np.arange(inp.B), n_acc - 1][:, 0:2]
    check_state(got, ref, "committed states (heads 0-1) vs oracle")
