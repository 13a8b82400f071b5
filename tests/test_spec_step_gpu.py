"""Parity of kda_spec_step (CUDA, through the C ABI): one speculative-decoding step of a layer, the prefill
segment and the verify segment in one call, each output row written at its place in the layer's output.

Checked three ways: against the fp64 oracle run on each segment (prefill and verify of the same layer: one pool,
one set of head parameters), bit for bit against the two plain calls (kda_chunk_prefill, kda_recurrent_verify),
and for the rows that belong to no token (left as they were)."""
import numpy as np
import pytest
import torch

import oracle
from kda_linear_attention_bounded_gb300 import inputs
import kda_linear_attention_bounded_gb300 as kda
from gpu_helpers import DeviceSpecStep, check_out, check_state

pytestmark = pytest.mark.gpu


def _separate_calls(dev):
    """The same step as two plain calls on a copy of the pool (the verify reads no slot the prefill writes, so
    their order does not matter)."""
    inp, pre, ver = dev.inp, dev.pre, dev.ver
    p, v = inp.prefill, inp.verify
    pool = dev.pool.clone()
    ws = kda.make_workspace(nbytes=kda.prefill_workspace_size(p.total_tokens, p.num_seqs, p.H))
    v_out = inter = p_out = final = None
    if v.B:
        v_out, inter = kda.recurrent_verify(ver.q, ver.k, ver.v, ver.g, ver.beta, pre.A_log, pre.dt_bias, pool,
                                            ver.slots, v.T, lower_bound=v.lower_bound, scale=v.scale, workspace=ws)
    if p.num_seqs:
        p_out, final = kda.chunk_prefill(pre.q, pre.k, pre.v, pre.g, pre.beta, pre.A_log, pre.dt_bias, pre.cu,
                                         pre.cu_host, lower_bound=p.lower_bound, scale=p.scale, state_pool=pool,
                                         slot_ids=pre.slots, load_initial=p.load_initial,
                                         final_to_pool=p.final_to_pool, workspace=ws,
                                         path="two_pass")   # the spec step runs the two-kernel path
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    return p_out, final, v_out, inter, pool


def _check_step(inp, heads=None, path=None):
    dev = DeviceSpecStep(inp)
    pool_before = dev.pool.clone()
    ref = _separate_calls(dev)
    ws = dev.workspace()
    out, final, inter = dev.run(workspace=ws, path=path)
    # copies taken by the next kernels on the stream, with no synchronisation in between: the call's work must
    # be complete for them (the verify grid runs beside the state pass and finishes after it)
    seen = (out.clone(), dev.pool.clone(), None if final is None else final.clone())
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    assert torch.equal(seen[0], out) and torch.equal(seen[1], dev.pool), "the stream's next kernel saw unfinished work"
    if final is not None:
        assert torch.equal(seen[2], final), "the stream's next kernel saw unfinished final states"
    p, v = inp.prefill, inp.verify
    ns = torch.from_numpy(inp.non_spec_token_indx).long().cuda()
    sp = torch.from_numpy(inp.spec_token_indx).long().cuda()

    # bit for bit against the plain calls: the step changes only where each row is stored
    p_out, p_final, v_out, v_inter, pool_sep = ref
    if p.total_tokens:
        assert torch.equal(out[ns], p_out), "prefill rows differ from kda_chunk_prefill's output"
    if v.B:
        assert torch.equal(out[sp], v_out), "verify rows differ from kda_recurrent_verify's output"
        assert torch.equal(inter, v_inter), "per-step states differ from kda_recurrent_verify's"
    if p.num_seqs and not p.final_to_pool:
        assert torch.equal(final, p_final), "dense final states differ from kda_chunk_prefill's"
    assert torch.equal(dev.pool, pool_sep), "pool differs from the one the plain calls leave"

    # rows of no token keep their value
    covered = torch.zeros(inp.num_out_tokens, dtype=torch.bool, device="cuda")
    covered[ns] = True
    covered[sp] = True
    assert (out[~covered].float() == DeviceSpecStep.SENTINEL).all(), "a row of no token was written"

    # against the oracle, segment by segment
    hb, he = heads if heads else (0, inp.H)
    if p.num_seqs:
        o_out, o_final, _ = oracle.run_prefill(p, heads=(hb, he))
        if p.total_tokens:
            check_out(out[ns][:, hb:he], o_out[:, hb:he], f"{inp.name} prefill rows heads {hb}:{he}",
                      segments=p.cu_seqlens)
        if p.final_to_pool:
            slots = torch.from_numpy(p.slot_ids).long().cuda()
            check_state(dev.pool[slots][:, hb:he], o_final[:, hb:he], f"{inp.name} final states in the pool")
        else:
            check_state(final[:, hb:he], o_final[:, hb:he], f"{inp.name} dense final states")
    if v.B:
        o_vout, o_steps = oracle.run_verify(v, heads=(hb, he))
        check_out(out[sp][:, hb:he], o_vout[:, hb:he], f"{inp.name} verify rows heads {hb}:{he}", segments=v.T)
        check_state(inter[:, :, hb:he], o_steps[:, :, hb:he], f"{inp.name} per-step states heads {hb}:{he}")
    # slots the prefill does not write back keep their state (the verify only reads the pool)
    written = set(p.slot_ids.tolist()) if (p.num_seqs and p.final_to_pool) else set()
    keep = [s for s in range(inp.prefill.pool.shape[0]) if s not in written]
    idx = torch.tensor(keep, dtype=torch.long, device="cuda")
    assert torch.equal(dev.pool[idx], pool_before[idx]), "a slot the step does not own changed"


@pytest.mark.parametrize("order", ["spec_first", "interleaved"])
def test_spec_step_small(order):
    # ragged prefill lengths (a zero-length sequence included) beside 5 requests x 3 tokens, spare output rows
    _check_step(inputs.spec_step_inputs("step_small", [130, 64, 1, 0, 77], 5, 3, 2, seed=400, order=order,
                                        extra_rows=7))


def test_spec_step_zero_initial_dense_final():
    _check_step(inputs.spec_step_inputs("step_dense", [200, 63], 4, 8, 3, seed=410, order="interleaved",
                                        load_initial=False, final_to_pool=False, extra_rows=3))


def test_spec_step_prefill_only_and_verify_only():
    _check_step(inputs.spec_step_inputs("step_prefill_only", [96, 40], 0, 4, 2, seed=420, order="interleaved",
                                        extra_rows=2))
    _check_step(inputs.spec_step_inputs("step_verify_only", [], 6, 4, 2, seed=421, order="interleaved",
                                        extra_rows=2))


def test_full_and_value_split_state_passes_agree_bit_for_bit():
    # The step stores its prefill rows by index, so its prefill segment runs the state pass that keeps all 128
    # value channels of a (sequence, head) in one CTA; the plain call on these few pairs runs the value-split
    # one (two CTAs, 64 value channels each, untransposed products).  Their products are the same sums in the
    # same order, so outputs and states must agree bit for bit, over 47 chunks of weak decay (lambda ~ -1e-3
    # per step), where any difference would carry.
    _check_step(inputs.spec_step_inputs("step_vs_weak", [3000, 700, 129], 0, 4, 4, seed=430, order="interleaved",
                                        extra_rows=1, g_mean=-8.0))


def test_spec_step_2048x4_64x4_h16_full():
    # the bench workload; the oracle runs on 4 of the 16 heads (the bit-exact checks cover all of them)
    _check_step(inputs.spec_step_2048x4_64x4(), heads=(6, 10))


def test_spec_step_bad_index():
    # an output row index outside [0, num_out_tokens) leaves that row unwritten and sets KDA_DEVICE_BAD_INDEX;
    # every other row is still written
    inp = inputs.spec_step_inputs("step_bad", [70], 2, 4, 2, seed=430, order="interleaved", extra_rows=1)
    dev = DeviceSpecStep(inp)
    dev.ns_idx[3] = -4
    dev.s_idx[5] = inp.num_out_tokens
    ws = dev.workspace()
    out, _, _ = dev.run(workspace=ws)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) & kda.KDA_DEVICE_BAD_INDEX
    o_out, _, _ = oracle.run_prefill(inp.prefill)
    good = np.setdiff1d(np.arange(70), [3])
    rows = torch.from_numpy(inp.non_spec_token_indx[good]).long().cuda()
    check_out(out[rows], o_out[good], "prefill rows beside a bad index")
    o_vout, _ = oracle.run_verify(inp.verify)
    good = np.setdiff1d(np.arange(8), [5])
    rows = torch.from_numpy(inp.spec_token_indx[good]).long().cuda()
    check_out(out[rows], o_vout[good], "verify rows beside a bad index")
    lost = [int(inp.non_spec_token_indx[3]), int(inp.spec_token_indx[5])]
    assert (out[lost].float() == DeviceSpecStep.SENTINEL).all(), "the rows of the bad indices were written"


def test_spec_step_replays_from_a_cuda_graph():
    inp = inputs.spec_step_inputs("step_graph", [150, 64], 8, 4, 2, seed=440, order="interleaved",
                                  load_initial=False, final_to_pool=False)
    dev = DeviceSpecStep(inp)
    ws = dev.workspace()
    out = dev.new_out()
    final = torch.empty((2, 2, 128, 128), dtype=torch.float32, device="cuda")
    inter = torch.empty((8, 4, 2, 128, 128), dtype=torch.float32, device="cuda")
    dev.run(out=out, final_state=final, intermediate_states=inter, workspace=ws)
    torch.cuda.synchronize()
    ref = (out.clone(), final.clone(), inter.clone())
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        dev.run(out=out, final_state=final, intermediate_states=inter, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dev.run(out=out, final_state=final, intermediate_states=inter, workspace=ws)
    out.fill_(DeviceSpecStep.SENTINEL)
    final.zero_()
    inter.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    assert torch.equal(out, ref[0]) and torch.equal(final, ref[1]) and torch.equal(inter, ref[2])


def test_spec_step_with_split_state_passes():
    # the prefill segment on the split schedule (KDA_OVERLAP at H = 16: its four longest sequences' state
    # passes in segments, the other two's beside the last segment, the verify grid behind the last launch):
    # bit for bit the plain calls' results, rows by index
    inp = inputs.spec_step_inputs("split_step", [1200, 700, 64, 3, 130, 1], 6, 4, 16, seed=860,
                                  order="interleaved", extra_rows=3)
    _check_step(inp, heads=(0, 4), path="overlap")
