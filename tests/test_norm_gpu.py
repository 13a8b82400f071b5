"""Parity of the sigmoid-gated RMSNorm fused into the output epilogues (prefill state pass, verify, spec step),
through the C ABI, against the fp64 oracle's norm of the oracle's own outputs; and bit-exactness between the
calls that share the epilogue."""
import numpy as np
import pytest
import torch

import oracle
from kda_linear_attention_bounded_gb300 import inputs
import kda_linear_attention_bounded_gb300 as kda
from gpu_helpers import DevicePrefill, DeviceSpecStep, DeviceVerify, check_norm, check_state, device_norm

pytestmark = pytest.mark.gpu


def _prefill_with_norm(inp, seed, heads=None):
    dev = DevicePrefill(inp)
    ni = inputs.norm_inputs(inp.total_tokens, inp.H, seed=seed)
    norm = device_norm(ni, inp.H)
    ws = dev.workspace()
    plain, _ = dev.run(workspace=ws)
    plain = plain.clone()
    out, final = dev.run(workspace=ws, norm=norm)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    o_ref, f_ref, _ = oracle.run_prefill(inp, heads=heads)
    hb, he = heads if heads else (0, inp.H)
    check_norm(out[:, hb:he], norm.rstd[:, hb:he], o_ref[:, hb:he], ni.gate[:, hb:he], ni,
               f"{inp.name} prefill heads {hb}:{he}", x_gpu=plain[:, hb:he])
    if final is not None:   # the norm leaves the state path alone
        check_state(final[:, hb:he], f_ref[:, hb:he], f"{inp.name} final states beside the norm")


def test_prefill_gated_norm_small():
    # ragged lengths: full chunks, a one-token sequence, a ragged last chunk
    _prefill_with_norm(inputs.prefill_inputs("norm_small", [130, 64, 1, 77], 2, seed=500, pool_slots=6,
                                             load_initial=True), seed=501)


def test_prefill_gated_norm_2048x8_h16_full():
    _prefill_with_norm(inputs.prefill_2048x8(), seed=502)


def test_verify_gated_norm():
    for inp, seed in ((inputs.verify_inputs("norm_verify", 3, 5, 2, seed=510, pool_slots=4), 511),
                      (inputs.verify_64x4(), 512)):
        dev = DeviceVerify(inp)
        ni = inputs.norm_inputs(inp.B * inp.T, inp.H, seed=seed)
        norm = device_norm(ni, inp.H)
        ws = kda.make_workspace()
        plain, _ = dev.run(workspace=ws)
        plain = plain.clone()
        out, inter = dev.run(workspace=ws, norm=norm)
        torch.cuda.synchronize()
        assert kda.read_device_status(ws) == 0
        o_ref, s_ref = oracle.run_verify(inp)
        check_norm(out, norm.rstd, o_ref, ni.gate, ni, f"{inp.name} verify", x_gpu=plain)
        check_state(inter, s_ref, f"{inp.name} per-step states beside the norm")


def test_spec_step_gated_norm_matches_the_plain_calls():
    # the spec step normalises each row with the gate row of its output row; the plain calls given the gate rows
    # gathered into token order store the same bits
    inp = inputs.spec_step_inputs("norm_step", [150, 64, 3], 6, 4, 2, seed=520, order="interleaved", extra_rows=5)
    dev = DeviceSpecStep(inp)
    ni = inputs.norm_inputs(inp.num_out_tokens, inp.H, seed=521)
    norm = device_norm(ni, inp.H)
    ws = dev.workspace()
    pool0 = dev.pool.clone()
    plain, _, _ = dev.run(workspace=ws)
    plain = plain.clone()
    dev.pool.copy_(pool0)
    out, _, inter = dev.run(workspace=ws, norm=norm)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    ns = torch.from_numpy(inp.non_spec_token_indx).long().cuda()
    sp = torch.from_numpy(inp.spec_token_indx).long().cuda()
    # against the oracle, row by row through the index arrays
    p_ref, _, _ = oracle.run_prefill(inp.prefill)
    v_ref, _ = oracle.run_verify(inp.verify)
    check_norm(out[ns], norm.rstd[ns], p_ref, ni.gate[inp.non_spec_token_indx], ni, "spec step prefill rows",
               x_gpu=plain[ns])
    check_norm(out[sp], norm.rstd[sp], v_ref, ni.gate[inp.spec_token_indx], ni, "spec step verify rows",
               x_gpu=plain[sp])
    covered = torch.zeros(inp.num_out_tokens, dtype=torch.bool, device="cuda")
    covered[ns] = True
    covered[sp] = True
    assert (out[~covered].float() == DeviceSpecStep.SENTINEL).all()
    assert torch.isnan(norm.rstd[~covered]).all(), "rstd written for a row of no token"
    # bit for bit against the plain calls with the gate rows in token order (a copy of the pool)
    pre, ver = dev.pre, dev.ver
    pool = torch.from_numpy(inp.prefill.pool).cuda()
    w = norm.weight
    pn = kda.OutputNorm(norm.gate[ns].contiguous(), w, ni.eps,
                        torch.empty((ns.numel(), inp.H), dtype=torch.float32, device="cuda"))
    vn = kda.OutputNorm(norm.gate[sp].contiguous(), w, ni.eps,
                        torch.empty((sp.numel(), inp.H), dtype=torch.float32, device="cuda"))
    ws2 = dev.workspace()
    p, v = inp.prefill, inp.verify
    v_out, v_inter = kda.recurrent_verify(ver.q, ver.k, ver.v, ver.g, ver.beta, pre.A_log, pre.dt_bias, pool,
                                          ver.slots, v.T, lower_bound=v.lower_bound, scale=v.scale, norm=vn,
                                          workspace=ws2)
    p_out, _ = kda.chunk_prefill(pre.q, pre.k, pre.v, pre.g, pre.beta, pre.A_log, pre.dt_bias, pre.cu, pre.cu_host,
                                 lower_bound=p.lower_bound, scale=p.scale, state_pool=pool, slot_ids=pre.slots,
                                 load_initial=p.load_initial, final_to_pool=p.final_to_pool, norm=pn, workspace=ws2,
                                 path="two_pass")   # the spec step runs the two-kernel path
    torch.cuda.synchronize()
    assert kda.read_device_status(ws2) == 0
    assert torch.equal(out[ns], p_out) and torch.equal(norm.rstd[ns], pn.rstd)
    assert torch.equal(out[sp], v_out) and torch.equal(norm.rstd[sp], vn.rstd)
    assert torch.equal(inter, v_inter)
    assert torch.equal(dev.pool, pool)


def test_norm_without_rstd_and_zero_gate():
    # rstd may be omitted; a zero gate halves the normalised row (sigmoid 0 = 1/2)
    inp = inputs.prefill_inputs("norm_zero_gate", [100], 2, seed=530)
    dev = DevicePrefill(inp)
    ni = inputs.norm_inputs(inp.total_tokens, inp.H, seed=531)
    ni.gate[:] = 0
    norm = device_norm(ni, inp.H, with_rstd=False)
    ws = dev.workspace()
    plain, _ = dev.run(workspace=ws)
    plain = plain.clone()
    out, _ = dev.run(workspace=ws, norm=norm)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    o_ref, _, _ = oracle.run_prefill(inp)
    check_norm(out, None, o_ref, ni.gate, ni, "zero gate, no rstd", x_gpu=plain)
