"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
call the library through its binding, and compare against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import kda_linear_attention_bounded_gb300 as kda

# Tolerances of the parity bar (outputs vs the fp64 oracle after the GPU's bf16
# rounding; states in fp32).
OUT_REL_L2 = 1e-2
OUT_MAX_ABS = 3e-2
STATE_REL_L2 = 5e-3


def bf16_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def f32_dev(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def i32_dev(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(device)


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / den) if den > 0 else float(np.linalg.norm(x))


def check_out(out_gpu, out_ref, what):
    x = out_gpu.float().cpu().numpy().astype(np.float64) if torch.is_tensor(out_gpu) else out_gpu
    assert np.isfinite(x).all(), f"{what}: non-finite GPU output"
    r = rel_l2(x, out_ref)
    m = float(np.abs(x - out_ref).max()) if x.size else 0.0
    assert r <= OUT_REL_L2 and m <= OUT_MAX_ABS, f"{what}: rel-L2 {r:.3e} (<= {OUT_REL_L2}), max-abs {m:.3e} (<= {OUT_MAX_ABS})"
    return r, m


def check_state(s_gpu, s_ref, what):
    x = s_gpu.cpu().numpy().astype(np.float64) if torch.is_tensor(s_gpu) else s_gpu
    assert np.isfinite(x).all(), f"{what}: non-finite GPU state"
    r = rel_l2(x, s_ref)
    assert r <= STATE_REL_L2, f"{what}: rel-L2 {r:.3e} (<= {STATE_REL_L2})"
    return r


class DevicePrefill:
    """Device copies of one prefill workload (``inputs.PrefillInputs``)."""

    def __init__(self, inp, device="cuda", token_pad=0):
        self.inp = inp
        H = inp.H
        T = inp.total_tokens

        def tok(bits):
            if token_pad == 0:
                return bf16_dev(bits, device)
            # token stride larger than H*128: embed in a wider row
            buf = torch.zeros((T, H * 128 + token_pad), dtype=torch.bfloat16, device=device)
            buf[:, :H * 128] = bf16_dev(bits, device).reshape(T, H * 128)
            return buf[:, :H * 128].view(T, H, 128)

        self.q, self.k, self.v, self.g = tok(inp.q), tok(inp.k), tok(inp.v), tok(inp.g)
        self.beta = bf16_dev(inp.beta, device)
        self.A_log = f32_dev(inp.A_log, device)
        self.dt_bias = f32_dev(inp.dt_bias, device)
        self.cu = i32_dev(inp.cu_seqlens, device)
        self.cu_host = torch.from_numpy(inp.cu_seqlens.astype(np.int32))
        self.pool = f32_dev(inp.pool, device) if inp.pool is not None else None
        self.slots = i32_dev(inp.slot_ids, device) if inp.slot_ids is not None else None

    def workspace(self, device="cuda"):
        inp = self.inp
        return kda.make_workspace(device, nbytes=kda.prefill_workspace_size(inp.total_tokens, inp.num_seqs, inp.H))

    def run(self, **kw):
        inp = self.inp
        return kda.chunk_prefill(self.q, self.k, self.v, self.g, self.beta, self.A_log, self.dt_bias, self.cu,
                                 self.cu_host, lower_bound=inp.lower_bound, scale=inp.scale,
                                 state_pool=self.pool, slot_ids=self.slots, load_initial=inp.load_initial,
                                 final_to_pool=inp.final_to_pool, **kw)


class DeviceVerify:
    def __init__(self, inp, device="cuda"):
        self.inp = inp
        self.q, self.k, self.v, self.g = (bf16_dev(x, device) for x in (inp.q, inp.k, inp.v, inp.g))
        self.beta = bf16_dev(inp.beta, device)
        self.A_log = f32_dev(inp.A_log, device)
        self.dt_bias = f32_dev(inp.dt_bias, device)
        self.pool = f32_dev(inp.pool, device)
        self.slots = i32_dev(inp.slot_ids, device)

    def run(self, **kw):
        inp = self.inp
        return kda.recurrent_verify(self.q, self.k, self.v, self.g, self.beta, self.A_log, self.dt_bias, self.pool,
                                    self.slots, inp.T, lower_bound=inp.lower_bound, scale=inp.scale, **kw)


class DeviceSpecStep:
    """Device copies of one spec step (``inputs.SpecStepInputs``): both segments read the one pool and the
    one set of head parameters."""

    SENTINEL = 5.0   # value of output rows that belong to no token

    def __init__(self, inp, device="cuda"):
        self.inp = inp
        self.pre = DevicePrefill(inp.prefill, device)
        self.ver = DeviceVerify(inp.verify, device)
        self.pool = self.pre.pool
        self.ver.pool = self.pool
        self.ns_idx = i32_dev(inp.non_spec_token_indx, device)
        self.s_idx = i32_dev(inp.spec_token_indx, device)
        self.device = device

    def workspace(self):
        p = self.inp.prefill
        return kda.make_workspace(self.device, nbytes=kda.prefill_workspace_size(p.total_tokens, p.num_seqs, p.H))

    def new_out(self):
        return torch.full((self.inp.num_out_tokens, self.inp.H, 128), self.SENTINEL, dtype=torch.bfloat16,
                          device=self.device)

    def run(self, out=None, **kw):
        inp, pre, ver = self.inp, self.pre, self.ver
        p, v = inp.prefill, inp.verify
        if out is None:
            out = self.new_out()
        has_pre, has_spec = p.num_seqs > 0, v.B > 0
        return kda.spec_step(
            (pre.q, pre.k, pre.v, pre.g, pre.beta) if has_pre else None, pre.cu, pre.cu_host,
            (ver.q, ver.k, ver.v, ver.g, ver.beta) if has_spec else None, v.T, pre.A_log, pre.dt_bias, self.pool,
            out, self.ns_idx, self.s_idx, prefill_slot_ids=pre.slots, spec_slot_ids=ver.slots,
            load_initial=p.load_initial, final_to_pool=p.final_to_pool, lower_bound=p.lower_bound, scale=p.scale,
            **kw)


def device_norm(ni, H, rows=None, device="cuda", with_rstd=True):
    """An OutputNorm on the device from ``inputs.NormInputs`` (rstd buffer NaN-filled)."""
    gate = bf16_dev(ni.gate, device)
    rows = gate.shape[0] if rows is None else rows
    rstd = torch.full((rows, H), float("nan"), dtype=torch.float32, device=device) if with_rstd else None
    return kda.OutputNorm(gate, f32_dev(ni.weight, device), ni.eps, rstd)


# Normalised outputs y = o rstd w sigmoid(z) are scale-free per row: a row whose attention output is far below
# the typical output scale (strong decay, k^.q^ near 0) keeps the relative error the bf16 products of the chunked
# path leave on it (up to ~1 % measured), and the normalisation turns that into an absolute error of y.  So the
# element-wise bar applies to the norm STAGE -- the GPU's y against the oracle's norm of the GPU's own attention
# output: one bf16 rounding of y plus one of its input, |dy| <= 2^-7 |y| + 1e-5, rstd within 1e-3 -- and the
# end-to-end result (the oracle's norm of the oracle's output) is held to the tensor-wide bars: rel-L2 <= 1e-2
# for y (the output bar) and <= 5e-3 for rstd (the state bar).


def check_norm(y_gpu, rstd_gpu, x_ref, z_bits, ni, what, x_gpu=None):
    """The gated RMSNorm of the GPU against the oracle's: end to end (the oracle's norm of the oracle's output
    rows ``x_ref``) and, given ``x_gpu`` (the GPU's un-normalised output rows from the same call without the
    norm), the norm stage alone (bars above)."""
    import oracle
    w = ni.weight.astype(np.float64)
    y = y_gpu.float().cpu().numpy().astype(np.float64) if torch.is_tensor(y_gpu) else y_gpu
    assert np.isfinite(y).all(), f"{what}: non-finite normalised output"
    y_ref, rstd_ref = oracle.gated_rmsnorm(x_ref, z_bits, w, ni.eps)
    r = rel_l2(y, y_ref)
    assert r <= OUT_REL_L2, f"{what}: normalised outputs rel-L2 {r:.3e} (<= {OUT_REL_L2})"
    rs = None
    if rstd_gpu is not None:
        rs = rstd_gpu.cpu().numpy().astype(np.float64) if torch.is_tensor(rstd_gpu) else rstd_gpu
        assert np.isfinite(rs).all(), f"{what}: rstd not written everywhere"
        rr = rel_l2(rs, rstd_ref)
        assert rr <= STATE_REL_L2, f"{what}: rstd rel-L2 {rr:.3e} (<= {STATE_REL_L2})"
    if x_gpu is not None:
        xg = x_gpu.float().cpu().numpy().astype(np.float64) if torch.is_tensor(x_gpu) else x_gpu
        y_st, rstd_st = oracle.gated_rmsnorm(xg, z_bits, w, ni.eps)
        bad = np.abs(y - y_st) > 2.0 ** -7 * np.abs(y_st) + 1e-5
        assert not bad.any(), f"{what}: norm stage off on {int(bad.sum())} elements (max {float(np.abs(y - y_st).max()):.3e})"
        if rs is not None:
            rel = float(np.abs(rs / rstd_st - 1.0).max())
            assert rel <= 1e-3, f"{what}: norm stage rstd relative error {rel:.3e} (<= 1e-3)"


def device_conv(ci, device="cuda", B=None, T=None, N=None):
    """A ShortConv on the device from ``inputs.ConvInputs`` (a copy of its window pool), with per-step window
    records for B x T verify tokens and/or dense final windows for N sequences (0xFFFF-filled: bf16 NaN)."""
    _, H, d, _ = ci.weight.shape
    steps = dense = None
    if B is not None:
        steps = torch.full((B, T, 3, 3, H, d), -1, dtype=torch.int16, device=device).view(torch.bfloat16)
    if N is not None:
        dense = torch.full((N, 3, 3, H, d), -1, dtype=torch.int16, device=device).view(torch.bfloat16)
    return kda.ShortConv(f32_dev(ci.weight, device), bf16_dev(ci.pool, device), ci.silu, window_dense=dense,
                         step_windows=steps)


def widen_bf16(t):
    """A bf16 CUDA tensor -> fp64 NumPy (exact)."""
    return t.float().cpu().numpy().astype(np.float64)
