"""Parity of the short causal convolutions of q, k, v (CUDA, through the C ABI) with the fp64 oracle: verify
from the slots' windows with per-step window records, the commit of the accepted window, and the spec step."""
import numpy as np
import pytest
import torch

import oracle
from kda_linear_attention_bounded_gb300 import inputs
import kda_linear_attention_bounded_gb300 as kda
from gpu_helpers import DeviceVerify, check_out, check_state, device_conv, i32_dev, widen_bf16

pytestmark = pytest.mark.gpu


def _verify_with_conv(inp, heads=None):
    dev = DeviceVerify(inp)
    conv = device_conv(inp.conv, B=inp.B, T=inp.T)
    pool_before = conv.window_pool.clone()
    ws = kda.make_workspace()
    out, inter = dev.run(workspace=ws, conv=conv)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    assert torch.equal(conv.window_pool, pool_before), "verify must not write the window pool"
    ref_out, ref_steps, ref_win = oracle.run_verify(inp, heads=heads)
    hb, he = heads if heads else (0, inp.H)
    check_out(out[:, hb:he], ref_out[:, hb:he], f"{inp.name} outputs with the convolutions", segments=inp.T)
    check_state(inter[:, :, hb:he], ref_steps[:, :, hb:he], f"{inp.name} per-step states with the convolutions")
    got = widen_bf16(conv.step_windows)
    assert np.array_equal(got[..., hb:he, :], ref_win[..., hb:he, :]), "per-step windows differ from the oracle's"
    return dev, conv, inter, ws


@pytest.mark.parametrize("T,silu", [(1, True), (3, True), (8, True), (5, False)])
def test_verify_with_short_conv_small(T, silu):
    inp = inputs.verify_inputs("conv_small", 3, T, 2, seed=600 + T, pool_slots=5)
    inp.conv = inputs.conv_inputs(2, 5, seed=610 + T, silu=silu)
    _verify_with_conv(inp)


def test_verify_with_short_conv_64x4_h16_full():
    inp = inputs.verify_64x4()
    inp.conv = inputs.conv_inputs(16, 256, seed=620)
    _verify_with_conv(inp, heads=(0, 8))


def test_commit_with_short_conv():
    inp = inputs.verify_inputs("conv_commit", 5, 4, 2, seed=630, pool_slots=7)
    inp.conv = inputs.conv_inputs(2, 7, seed=631)
    dev, conv, inter, ws = _verify_with_conv(inp)
    n_acc = np.array([0, 1, 4, 2, 3], np.int32)
    pool_before, win_before = dev.pool.clone(), conv.window_pool.clone()
    kda.commit_accepted(dev.pool, dev.slots, i32_dev(n_acc), inter, conv=conv, workspace=ws)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    for b, n in enumerate(n_acc):
        s = int(inp.slot_ids[b])
        if n == 0:
            assert torch.equal(conv.window_pool[s], win_before[s]) and torch.equal(dev.pool[s], pool_before[s])
        else:
            assert torch.equal(conv.window_pool[s], conv.step_windows[b, n - 1]), f"request {b}: window not committed"
            assert torch.equal(dev.pool[s], inter[b, n - 1])
    others = np.setdiff1d(np.arange(7), inp.slot_ids)
    idx = torch.from_numpy(others).long().cuda()
    assert torch.equal(conv.window_pool[idx], win_before[idx])


def test_verify_then_commit_then_verify_continues_the_sequence():
    # two verify steps with the accepted window and state committed between them equal one run over the
    # accepted tokens followed by the next block: the window carries the convolution across the steps
    H, T = 2, 4
    first = inputs.verify_inputs("conv_chain", 2, T, H, seed=640, pool_slots=3)
    first.conv = inputs.conv_inputs(H, 3, seed=641)
    dev, conv, inter, ws = _verify_with_conv(first)
    n_acc = np.array([2, 4], np.int32)
    kda.commit_accepted(dev.pool, dev.slots, i32_dev(n_acc), inter, conv=conv, workspace=ws)
    second = inputs.verify_inputs("conv_chain2", 2, T, H, seed=642, pool_slots=3)
    second.slot_ids = first.slot_ids
    second.A_log, second.dt_bias = first.A_log, first.dt_bias
    dev2 = DeviceVerify(second)
    conv2 = kda.ShortConv(conv.weight, conv.window_pool, conv.silu,
                          step_windows=torch.empty_like(conv.step_windows))
    out2, _ = kda.recurrent_verify(dev2.q, dev2.k, dev2.v, dev2.g, dev2.beta, dev.A_log, dev.dt_bias, dev.pool,
                                   dev.slots, T, lower_bound=second.lower_bound, scale=second.scale, conv=conv2,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    # the oracle: per request, the accepted tokens of the first block then the second block, in one run
    for b in range(2):
        n = int(n_acc[b])
        rows1 = slice(b * T, b * T + n)
        rows2 = slice(b * T, b * T + T)
        cat = lambda a1, a2: np.concatenate([a1[rows1], a2[rows2]])
        s = int(first.slot_ids[b])
        ref, _, _, _, _ = oracle.run_conv(
            cat(first.q, second.q), cat(first.k, second.k), cat(first.v, second.v), cat(first.g, second.g),
            cat(first.beta, second.beta), first.A_log, first.dt_bias, first.lower_bound, first.scale,
            np.array([0, n + T], np.int32), first.conv.weight, first.conv.silu,
            win0=oracle.bf16_widen(first.conv.pool[s:s + 1]), S0=first.pool[s:s + 1])
        check_out(out2[b * T:(b + 1) * T], ref[n:], f"request {b}: second block after committing {n} tokens",
                  segments=T)


def test_spec_step_verify_segment_with_short_conv():
    inp = inputs.verify_inputs("conv_step", 4, 3, 2, seed=650, pool_slots=6)
    inp.conv = inputs.conv_inputs(2, 6, seed=651)
    dev = DeviceVerify(inp)
    conv = device_conv(inp.conv, B=inp.B, T=inp.T)
    rows = np.random.default_rng(652).permutation(inp.B * inp.T + 3)[:inp.B * inp.T].astype(np.int32)
    out = torch.zeros((inp.B * inp.T + 3, 2, 128), dtype=torch.bfloat16, device="cuda")
    ws = kda.make_workspace()
    out, _, inter = kda.spec_step(None, None, None, (dev.q, dev.k, dev.v, dev.g, dev.beta), inp.T, dev.A_log,
                                  dev.dt_bias, dev.pool, out, None, i32_dev(rows), spec_slot_ids=dev.slots,
                                  lower_bound=inp.lower_bound, scale=inp.scale, conv=conv, workspace=ws)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    ref_out, ref_steps, ref_win = oracle.run_verify(inp)
    check_out(out[torch.from_numpy(rows).long().cuda()], ref_out, "spec step verify rows with the convolutions",
              segments=inp.T)
    check_state(inter, ref_steps, "spec step per-step states with the convolutions")
    assert np.array_equal(widen_bf16(conv.step_windows), ref_win)


def _prefill_with_conv(inp, heads=None, path=None):
    from gpu_helpers import DevicePrefill
    dev = DevicePrefill(inp)
    conv = device_conv(inp.conv, N=None if inp.final_to_pool else inp.num_seqs)
    ws = dev.workspace()
    out, final = dev.run(workspace=ws, conv=conv, path=path)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    ref_out, ref_S, _, ref_win = oracle.run_prefill(inp, heads=heads)
    hb, he = heads if heads else (0, inp.H)
    check_out(out[:, hb:he], ref_out[:, hb:he], f"{inp.name} outputs with the convolutions", segments=inp.cu_seqlens)
    if inp.final_to_pool:
        slots = torch.from_numpy(inp.slot_ids).long().cuda()
        check_state(dev.pool[slots][:, hb:he], ref_S[:, hb:he], f"{inp.name} final states (pool) with the convolutions")
        got_win = widen_bf16(conv.window_pool[slots])
    else:
        check_state(final[:, hb:he], ref_S[:, hb:he], f"{inp.name} final states (dense)")
        got_win = widen_bf16(conv.window_dense)
    assert np.array_equal(got_win[..., hb:he, :], ref_win[..., hb:he, :]), "final windows differ from the oracle's"
    return dev, conv, out, final


@pytest.mark.parametrize("final_to_pool", [True, False])
def test_prefill_with_short_conv_split_schedule(final_to_pool):
    # KDA_OVERLAP with the convolutions at H = 16: the four longest sequences' state passes run in segments
    # (a segment after the first starts from the scratch state; only the last one writes the final window),
    # the one- and two-token and 64-token sequences beside them on the plain schedule (their windows keep
    # rows of the initial one).  Against the oracle, and bit for bit against the two-kernel path.
    inp = inputs.prefill_inputs("conv_split", [1000, 300, 130, 64, 1, 2, 77], 16, seed=750, pool_slots=9,
                                load_initial=True, final_to_pool=final_to_pool)
    inp.conv = inputs.conv_inputs(16, 9, seed=751)
    dev_s, conv_s, out_s, final_s = _prefill_with_conv(inp, heads=(0, 4), path="overlap")
    dev_t, conv_t, out_t, final_t = _prefill_with_conv(inp, heads=(0, 4), path="two_pass")
    assert torch.equal(out_s, out_t)
    if final_to_pool:
        assert torch.equal(dev_s.pool, dev_t.pool) and torch.equal(conv_s.window_pool, conv_t.window_pool)
    else:
        assert torch.equal(final_s, final_t) and torch.equal(conv_s.window_dense, conv_t.window_dense)


@pytest.mark.parametrize("lb", [-5.0, -8.0])
def test_prefill_with_short_conv_small(lb):
    # full chunks, a one-token and a two-token sequence (their final windows keep rows of the initial one), a
    # zero-length one, a ragged last chunk; both sub-block sizes of the intra-chunk kernel
    inp = inputs.prefill_inputs("conv_prefill", [130, 64, 1, 0, 77, 2], 2, seed=700, pool_slots=8,
                                load_initial=True, final_to_pool=True, lower_bound=lb)
    inp.conv = inputs.conv_inputs(2, 8, seed=701)
    _prefill_with_conv(inp)


def test_prefill_with_short_conv_zero_start_dense_final():
    inp = inputs.prefill_inputs("conv_prefill_dense", [100, 3, 65], 3, seed=710)
    inp.conv = inputs.conv_inputs(3, 4, seed=711, silu=False)
    _prefill_with_conv(inp)


def test_prefill_with_short_conv_2048x8_h16_full():
    inp = inputs.prefill_2048x8()
    inp.final_to_pool = True
    inp.conv = inputs.conv_inputs(16, 64, seed=720)
    _prefill_with_conv(inp, heads=(0, 4))


def test_prefill_then_verify_continue_through_the_window():
    # a prefill that leaves its final state and window in the pool, then a verify block from them, equals one
    # oracle run over both token sets
    H, T = 2, 5
    pre = inputs.prefill_inputs("conv_pv", [77, 130], H, seed=730, pool_slots=4, load_initial=True,
                                final_to_pool=True)
    pre.conv = inputs.conv_inputs(H, 4, seed=731)
    dev, conv, _, _ = _prefill_with_conv(pre)
    ver = inputs.verify_inputs("conv_pv2", 2, T, H, seed=732, pool_slots=4)
    dver = DeviceVerify(ver)
    conv2 = kda.ShortConv(conv.weight, conv.window_pool, conv.silu,
                          step_windows=torch.empty((2, T, 3, 3, H, 128), dtype=torch.bfloat16, device="cuda"))
    ws = kda.make_workspace()
    out, _ = kda.recurrent_verify(dver.q, dver.k, dver.v, dver.g, dver.beta, dev.A_log, dev.dt_bias, dev.pool,
                                  dev.slots, T, lower_bound=pre.lower_bound, scale=pre.scale, conv=conv2,
                                  workspace=ws)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    for b in range(2):
        a, e = int(pre.cu_seqlens[b]), int(pre.cu_seqlens[b + 1])
        cat = lambda x1, x2: np.concatenate([x1[a:e], x2[b * T:(b + 1) * T]])
        s = int(pre.slot_ids[b])
        ref, _, _, _, _ = oracle.run_conv(cat(pre.q, ver.q), cat(pre.k, ver.k), cat(pre.v, ver.v),
                                          cat(pre.g, ver.g), cat(pre.beta, ver.beta), pre.A_log, pre.dt_bias,
                                          pre.lower_bound, pre.scale, np.array([0, e - a + T], np.int32),
                                          pre.conv.weight, pre.conv.silu,
                                          win0=oracle.bf16_widen(pre.conv.pool[s:s + 1]), S0=pre.pool[s:s + 1])
        check_out(out[b * T:(b + 1) * T], ref[e - a:], f"sequence {b}: verify block after its prefill", segments=T)


def test_spec_step_with_short_conv_both_segments():
    from gpu_helpers import DeviceSpecStep
    inp = inputs.spec_step_inputs("conv_step2", [90, 64, 2], 4, 3, 2, seed=740, order="interleaved", extra_rows=2)
    ci = inputs.conv_inputs(2, inp.prefill.pool.shape[0], seed=741)
    inp.prefill.conv = inp.verify.conv = ci
    dev = DeviceSpecStep(inp)
    conv = device_conv(ci, B=inp.verify.B, T=inp.verify.T)
    ws = dev.workspace()
    out, _, inter = dev.run(workspace=ws, conv=conv)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    p_out, p_S, _, p_win = oracle.run_prefill(inp.prefill)
    v_out, v_steps, v_win = oracle.run_verify(inp.verify)
    ns = torch.from_numpy(inp.non_spec_token_indx).long().cuda()
    sp = torch.from_numpy(inp.spec_token_indx).long().cuda()
    check_out(out[ns], p_out, "spec step prefill rows with the convolutions", segments=inp.prefill.cu_seqlens)
    check_out(out[sp], v_out, "spec step verify rows with the convolutions", segments=inp.verify.T)
    check_state(inter, v_steps, "spec step per-step states with the convolutions")
    pslots = torch.from_numpy(inp.prefill.slot_ids).long().cuda()
    check_state(dev.pool[pslots], p_S, "spec step prefill final states")
    assert np.array_equal(widen_bf16(conv.window_pool[pslots]), p_win), "prefill final windows"
    assert np.array_equal(widen_bf16(conv.step_windows), v_win), "verify per-step windows"


def test_prefill_with_short_conv_bad_slot():
    # a slot id outside the pool: that sequence is skipped with the status bit, its chunks read no window, and
    # the other sequence is unaffected
    from gpu_helpers import DevicePrefill
    inp = inputs.prefill_inputs("conv_bad_slot", [70, 90], 2, seed=750, pool_slots=4, load_initial=True,
                                final_to_pool=True)
    inp.conv = inputs.conv_inputs(2, 4, seed=751)
    dev = DevicePrefill(inp)
    dev.slots[1] = 4   # == num_slots
    conv = device_conv(inp.conv)
    ws = dev.workspace()
    out, _ = dev.run(workspace=ws, conv=conv)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) & kda.KDA_DEVICE_BAD_SLOT
    ref_out, ref_S, _, ref_win = oracle.run_prefill(inp)
    check_out(out[:70], ref_out[:70], "the sequence beside a bad slot", segments=[0, 70])
    s0 = int(inp.slot_ids[0])
    check_state(dev.pool[s0], ref_S[0], "its final state")
    assert np.array_equal(widen_bf16(conv.window_pool[s0]), ref_win[0]), "its final window"


def test_spec_step_with_short_conv_and_gated_norm():
    # every option at once: convolutions on both segments, the gated norm on every output row
    from gpu_helpers import DeviceSpecStep, check_norm, device_norm
    inp = inputs.spec_step_inputs("conv_norm_step", [100, 7], 3, 4, 2, seed=760, order="interleaved", extra_rows=1)
    ci = inputs.conv_inputs(2, inp.prefill.pool.shape[0], seed=761)
    inp.prefill.conv = inp.verify.conv = ci
    dev = DeviceSpecStep(inp)
    conv = device_conv(ci, B=inp.verify.B, T=inp.verify.T)
    ni = inputs.norm_inputs(inp.num_out_tokens, 2, seed=762)
    norm = device_norm(ni, 2)
    ws = dev.workspace()
    out, _, inter = dev.run(workspace=ws, conv=conv, norm=norm)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    p_out, p_S, _, p_win = oracle.run_prefill(inp.prefill)
    v_out, v_steps, v_win = oracle.run_verify(inp.verify)
    ns, sp = inp.non_spec_token_indx, inp.spec_token_indx
    y = out.float().cpu().numpy()
    r = norm.rstd.cpu().numpy()
    check_norm(y[ns], r[ns], p_out, ni.gate[ns], ni, "prefill rows, convolutions + norm")
    check_norm(y[sp], r[sp], v_out, ni.gate[sp], ni, "verify rows, convolutions + norm")
    check_state(inter, v_steps, "per-step states, convolutions + norm")
    pslots = torch.from_numpy(inp.prefill.slot_ids).long().cuda()
    check_state(dev.pool[pslots], p_S, "prefill final states, convolutions + norm")
    assert np.array_equal(widen_bf16(conv.window_pool[pslots]), p_win)
    assert np.array_equal(widen_bf16(conv.step_windows), v_win)


def test_prefill_with_short_conv_over_several_launch_groups():
    # 1100 short sequences (two launch groups of <= 1024): each group's first chunks find their slots' windows
    # through the group's sequence offset, and each sequence's final window lands in its own slot
    rng = np.random.default_rng(770)
    lens = [int(x) for x in rng.integers(0, 40, size=1100)]
    inp = inputs.prefill_inputs("conv_many_seqs", lens, 2, seed=771, pool_slots=1100, load_initial=True,
                                final_to_pool=True)
    inp.conv = inputs.conv_inputs(2, 1100, seed=772)
    _prefill_with_conv(inp)
