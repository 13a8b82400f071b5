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
        check_out(out[:, hb:he], ref_out[:, hb:he], f"{inp.name} outputs heads {hb}:{he}", segments=inp.T)
        check_state(inter[:, :, hb:he], ref_steps[:, :, hb:he], f"{inp.name} per-step states heads {hb}:{he}")


def test_verify_64x8_h16_full():
    _parity(inputs.verify_64x8(), head_groups=4)


@pytest.mark.parametrize("make", [inputs.verify_64x4, inputs.verify_64x1], ids=["T4", "T1"])
def test_verify_64xT_h16_full(make):
    # the MTP-3 (three drafts plus the bonus token) and plain decode block sizes at the full batch
    _parity(make(), head_groups=2)


@pytest.mark.parametrize("T", [1, 3, 8, 17])
def test_verify_small(T):
    _parity(inputs.verify_inputs("small", 3, T, 2, seed=60 + T, pool_slots=5))


@pytest.mark.parametrize("H", [3, 5, 32])
def test_verify_head_counts_outside_the_bench_shapes(H):
    # odd head counts and a larger one, at a batch below one wave (so value channels are split) and above it
    _parity(inputs.verify_inputs(f"heads_{H}", 2, 5, H, seed=90 + H, pool_slots=4))
    _parity(inputs.verify_inputs(f"heads_{H}_b", 40, 3, H, seed=95 + H, pool_slots=48))


def test_verify_repeated_slots_and_weak_decay():
    inp = inputs.verify_inputs("rep", 4, 8, 2, seed=70, pool_slots=3, g_mean=-8.0)
    inp.slot_ids = np.array([1, 1, 2, 1], np.int32)
    _parity(inp)


def test_verify_bad_slot():
    inp = inputs.verify_inputs("bad", 2, 4, 2, seed=80, pool_slots=3)
    dev = DeviceVerify(inp)
    dev.slots[0] = 3   # == num_slots
    ws = kda.make_workspace()
    out = torch.full((8, 2, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    out, inter = dev.run(workspace=ws, out=out)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) & kda.KDA_DEVICE_BAD_SLOT
    assert (out[:4].float() == 3.0).all()
    ref_out, ref_steps = oracle.run_verify(inp)
    check_out(out[4:], ref_out[4:], "good request next to a bad slot", segments=inp.T)
    check_state(inter[1], ref_steps[1], "good request states")


def test_verify_padding_rows_are_skipped():
    # rows whose slot id is KDA_PAD_SLOT_ID (unused rows of a bucketed batch) are skipped without a status bit,
    # their output and per-step state rows left as they were; the live rows are unaffected by them
    inp = inputs.verify_inputs("pad", 6, 4, 2, seed=85, pool_slots=7)
    pad = [1, 4]
    dev = DeviceVerify(inp)
    for b in pad:
        dev.slots[b] = kda.KDA_PAD_SLOT_ID
    ws = kda.make_workspace()
    out = torch.full((24, 2, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    inter = torch.full((6, 4, 2, 128, 128), 7.0, dtype=torch.float32, device="cuda")
    dev.run(workspace=ws, out=out, intermediate_states=inter)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    ref_out, ref_steps = oracle.run_verify(inp)
    for b in range(6):
        rows = slice(4 * b, 4 * b + 4)
        if b in pad:
            assert (out[rows].float() == 3.0).all() and (inter[b] == 7.0).all(), f"padding row {b} was written"
        else:
            check_out(out[rows], ref_out[rows], f"live request {b}", segments=inp.T)
            check_state(inter[b], ref_steps[b], f"live request {b} states")


@pytest.mark.parametrize("T", [1, 4, 8])
def test_verify_and_commit_replay_from_a_bucket_graph(T):
    # one CUDA graph per (bucket of 8 requests, T): verify + accept/commit captured once on static buffers, then
    # replayed on new token data, head parameters, pool contents and slot ids written into those buffers, with a
    # full bucket and with 5 live requests (3 padding rows).  Each replay equals the direct calls bit for bit.
    H, Bk = 4, 8
    slots_total = 16
    dev = DeviceVerify(inputs.verify_inputs("bucket", Bk, T, H, seed=90 + T, pool_slots=slots_total))
    n_acc = torch.zeros(Bk, dtype=torch.int32, device="cuda")
    ws = kda.make_workspace()
    out = torch.empty((Bk * T, H, 128), dtype=torch.bfloat16, device="cuda")
    inter = torch.empty((Bk, T, H, 128, 128), dtype=torch.float32, device="cuda")

    def step():
        dev.run(workspace=ws, out=out, intermediate_states=inter)
        kda.commit_accepted(dev.pool, dev.slots, n_acc, inter, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for live, seed in ((Bk, 200 + T), (5, 300 + T)):
        new = inputs.verify_inputs("bucket_batch", live, T, H, seed=seed, pool_slots=slots_total)
        fresh = DeviceVerify(new)
        rows = live * T
        for name in ("q", "k", "v", "g", "beta"):
            getattr(dev, name)[:rows].copy_(getattr(fresh, name))
        dev.A_log.copy_(fresh.A_log)
        dev.dt_bias.copy_(fresh.dt_bias)
        dev.pool.copy_(fresh.pool)
        dev.slots.fill_(kda.KDA_PAD_SLOT_ID)
        dev.slots[:live].copy_(fresh.slots)
        acc = np.random.default_rng(seed).integers(0, T + 1, size=live).astype(np.int32)
        n_acc.fill_(T)   # padding rows: any count is ignored
        n_acc[:live].copy_(torch.from_numpy(acc))
        pool_in = fresh.pool.clone()
        graph.replay()
        torch.cuda.synchronize()
        assert kda.read_device_status(ws) == 0

        ref_ws = kda.make_workspace()
        ref_out, ref_inter = fresh.run(workspace=ref_ws)
        kda.commit_accepted(fresh.pool, fresh.slots, torch.from_numpy(acc).cuda(), ref_inter, workspace=ref_ws)
        torch.cuda.synchronize()
        assert kda.read_device_status(ref_ws) == 0
        assert torch.equal(out[:rows], ref_out), f"live={live}: replayed outputs differ from a direct call"
        assert torch.equal(inter[:live], ref_inter), f"live={live}: replayed per-step states differ"
        assert torch.equal(dev.pool, fresh.pool), f"live={live}: pool after the replayed commit differs"
        o_out, o_steps = oracle.run_verify(new)
        check_out(out[:rows], o_out, f"bucket T={T} live={live} outputs", segments=T)
        check_state(inter[:live], o_steps, f"bucket T={T} live={live} per-step states")
        for b in range(live):
            s = int(new.slot_ids[b])
            if acc[b] == 0:
                assert torch.equal(dev.pool[s], pool_in[s])
            else:
                assert torch.equal(dev.pool[s], inter[b, acc[b] - 1])


@pytest.mark.parametrize("T", [3, 4])
def test_small_batches_split_value_channels_bit_identically(T):
    # a batch too small to fill one wave splits each (request, head)'s value channels over 2 or 4 CTAs, and a
    # batch above one wave with T >= 4 over 2 CTAs at three per SM; every column is computed exactly as in the
    # unsplit kernel, so requests verified alone equal the same requests inside a full batch bit for bit (the
    # full batch runs whole items at T = 3 and the three-per-SM split at T = 4)
    full = inputs.verify_inputs("split_full", 64, T, 16, seed=96, pool_slots=256)
    dev = DeviceVerify(full)
    ws = kda.make_workspace()
    out_all, inter_all = dev.run(workspace=ws)
    torch.cuda.synchronize()
    for B in (1, 4, 8):   # 16, 64, 128 (request, head) items: split 4, 4, 2 ways on a 152-SM GPU
        out, inter = kda.recurrent_verify(dev.q[:B * T], dev.k[:B * T], dev.v[:B * T], dev.g[:B * T],
                                          dev.beta[:B * T], dev.A_log, dev.dt_bias, dev.pool, dev.slots[:B], T,
                                          lower_bound=full.lower_bound, scale=full.scale, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out, out_all[:B * T]), f"B={B}: outputs differ from the full batch's"
        assert torch.equal(inter, inter_all[:B]), f"B={B}: per-step states differ from the full batch's"
    assert kda.read_device_status(ws) == 0
    small = inputs.verify_inputs("split_small", 8, 5, 16, seed=97, pool_slots=16)
    _parity(small, head_groups=2)
