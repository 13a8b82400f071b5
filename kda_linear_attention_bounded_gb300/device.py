"""Device copies of the seeded synthetic workloads (``inputs``) and the calls
that run them through the binding.

Marshalling only: host arrays from ``inputs`` are copied to CUDA tensors and
handed to the library's calls; nothing of the method is computed here.  Used by
``bench.py`` and by the GPU tests.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _binding as kda


def bf16_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def f32_dev(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def i32_dev(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(device)


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
