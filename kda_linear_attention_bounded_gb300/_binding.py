"""ctypes binding of libkda (``include/kda.h``), marshalling torch tensors.

Argument marshalling only: every step of the computation runs in libkda's
CUDA kernels.  PyTorch provides device memory and the current stream.  When
the library has not been built this module raises instead of computing
anything another way.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

import torch

from . import build as _build

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_WORKSPACE = 3
KDA_ERR_CUDA = 4
KDA_DEVICE_BAD_SLOT = 1
KDA_DEVICE_TIMEOUT = 2
KDA_DEVICE_BAD_COUNT = 4
KDA_DEVICE_BAD_INDEX = 8
KDA_LOAD_INITIAL = 1
KDA_FINAL_TO_POOL = 2
KDA_TWO_PASS = 4
KDA_FUSED = 8
KDA_OVERLAP = 16
KDA_PAD_SLOT_ID = -1
KDA_CONV_NONE = 0
KDA_CONV_SILU = 1
KDA_SCHEDULE_FUSED = 1
KDA_SCHEDULE_PLAIN = 2
KDA_SCHEDULE_SPLIT = 3

#: exported symbols of include/kda.h
EXPORTS = ("kda_status_string", "kda_workspace_size", "kda_prefill_workspace_size", "kda_workspace_reset",
           "kda_read_device_status", "kda_chunk_prefill", "kda_recurrent_verify", "kda_commit_accepted",
           "kda_recurrent_verify_noalloc", "kda_spec_step", "kda_prefill_schedule")

_lib = None


class TokenTensors(ctypes.Structure):
    """``kda_token_tensors``: q, k, v, g, beta_logits of one set of tokens."""
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("qkv_token_stride", ctypes.c_int64), ("g", ctypes.c_void_p), ("g_token_stride", ctypes.c_int64),
                ("beta_logits", ctypes.c_void_p), ("beta_token_stride", ctypes.c_int64)]


class _OutputNormC(ctypes.Structure):
    """``kda_output_norm``."""
    _fields_ = [("gate", ctypes.c_void_p), ("gate_token_stride", ctypes.c_int64), ("weight", ctypes.c_void_p),
                ("eps", ctypes.c_float), ("rstd", ctypes.c_void_p)]


class OutputNorm:
    """Sigmoid-gated RMSNorm of the output rows (``kda_output_norm``):
    ``y = o * rstd * weight * sigmoid(gate)``, ``rstd = (mean o^2 + eps)^-1/2`` per (row, head).

    gate: CUDA bf16 ``[rows, H, 128]`` (rows as the call's output rows); weight: CUDA fp32 ``[128]``;
    rstd: optional CUDA fp32 ``[rows, H]`` written by the call."""

    def __init__(self, gate, weight, eps=1e-6, rstd=None):
        self.gate, self.weight, self.eps, self.rstd = gate, weight, float(eps), rstd

    def as_c(self, H):
        gs = _token_tensor(self.gate, "norm gate", H)
        w = self.weight
        if w.dtype != torch.float32 or not w.is_cuda or w.numel() != 128 or not w.is_contiguous():
            raise ValueError("norm weight: expected a contiguous CUDA fp32 tensor of 128 entries")
        r = self.rstd
        if r is not None and (r.dtype != torch.float32 or not r.is_cuda or r.dim() != 2 or r.shape[1] != H
                              or not r.is_contiguous()):
            raise ValueError("norm rstd: expected a contiguous CUDA fp32 tensor [rows, H]")
        return _OutputNormC(self.gate.data_ptr(), gs, w.data_ptr(), self.eps, None if r is None else r.data_ptr())


class _ShortConvC(ctypes.Structure):
    """``kda_short_conv``."""
    _fields_ = [("weight", ctypes.c_void_p), ("activation", ctypes.c_int), ("window_pool", ctypes.c_void_p),
                ("window_dense", ctypes.c_void_p), ("step_windows", ctypes.c_void_p)]


class ShortConv:
    """Short causal convolutions of q, k, v (``kda_short_conv``); q, k, v passed to a call are then their raw
    inputs.  weight: CUDA fp32 ``[3, H, 128, 4]``; window_pool: CUDA bf16 ``[slots, 3, 3, H, 128]``;
    window_dense: prefill, ``[num_seqs, 3, 3, H, 128]`` final windows with dense final states; step_windows:
    verify / commit, ``[B, T, 3, 3, H, 128]``."""

    def __init__(self, weight, window_pool, silu=True, window_dense=None, step_windows=None):
        self.weight, self.window_pool, self.silu = weight, window_pool, bool(silu)
        self.window_dense, self.step_windows = window_dense, step_windows

    def as_c(self):
        w = self.weight
        if w.dtype != torch.float32 or not w.is_cuda or w.dim() != 4 or w.shape[2:] != (128, 4) or not w.is_contiguous():
            raise ValueError("conv weight: expected a contiguous CUDA fp32 tensor [3, H, 128, 4]")
        for name in ("window_pool", "window_dense", "step_windows"):
            t = getattr(self, name)
            if t is not None and (t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous()):
                raise ValueError(f"conv {name}: expected a contiguous CUDA bf16 tensor")
        return _ShortConvC(w.data_ptr(), KDA_CONV_SILU if self.silu else KDA_CONV_NONE,
                           *(None if t is None else t.data_ptr()
                             for t in (self.window_pool, self.window_dense, self.step_windows)))


def _conv_arg(conv):
    return None if conv is None else ctypes.byref(conv.as_c())


def _norm_arg(norm, H):
    return None if norm is None else ctypes.byref(norm.as_c(H))


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load():
    """Load libkda; raise if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libkda is not built ({path} missing): run __graft_entry__.build() "
                           "or `python -m kda_linear_attention_bounded_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.kda_status_string.argtypes = [I]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_workspace_size.argtypes = []
    lib.kda_workspace_size.restype = SZ
    lib.kda_prefill_workspace_size.argtypes = [I64, I, I]
    lib.kda_prefill_workspace_size.restype = SZ
    lib.kda_workspace_reset.argtypes = [P, SZ, P]
    lib.kda_workspace_reset.restype = I
    lib.kda_read_device_status.argtypes = [P, SZ, ctypes.POINTER(ctypes.c_uint32), P]
    lib.kda_read_device_status.restype = I
    NP = ctypes.POINTER(_OutputNormC)
    CP = ctypes.POINTER(_ShortConvC)
    lib.kda_chunk_prefill.argtypes = [P, P, P, I64, P, I64, P, I64, P, P, F, F, P, P, I, I, P, I, P, I, P,
                                      I64, NP, CP, P, P, SZ, P]
    lib.kda_chunk_prefill.restype = I
    lib.kda_recurrent_verify.argtypes = [P, P, P, I64, P, I64, P, I64, P, P, F, F, I, I, I, P, I, P, P, I64,
                                         NP, CP, P, P, SZ, P]
    lib.kda_recurrent_verify.restype = I
    lib.kda_commit_accepted.argtypes = [P, I, P, P, P, CP, I, I, I, P, SZ, P]
    lib.kda_commit_accepted.restype = I
    TT = ctypes.POINTER(TokenTensors)
    lib.kda_spec_step.argtypes = [TT, P, P, I, P, I, P, TT, I, I, P, P, P, P, F, F, I, P, I, P, I64, I64, NP, CP, P,
                                  P, P, SZ, P]
    lib.kda_spec_step.restype = I
    lib.kda_prefill_schedule.argtypes = [P, I, I, I, F, I, SZ, I, P]
    lib.kda_prefill_schedule.restype = I
    _lib = lib
    return lib


def prefill_schedule(cu_seqlens_host, H, *, lower_bound=-5.0, path=None, conv=False, workspace_bytes=None,
                     sms=0):
    """``kda_prefill_schedule``: the schedule ``chunk_prefill`` takes for these sequence lengths (host only, no
    GPU needed).  Returns ``{"kind": "fused" | "plain" | "split", "value_split": bool, "segments": int,
    "split_sequences": int}``."""
    lib = load()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens_host, dtype=np.int32))
    N = cu.size - 1
    if workspace_bytes is None:
        workspace_bytes = prefill_workspace_size(int(cu[-1]), N, H)
    flags = {None: 0, "two_pass": KDA_TWO_PASS, "fused": KDA_FUSED, "overlap": KDA_OVERLAP}[path]
    info = (ctypes.c_int * 4)()
    rc = lib.kda_prefill_schedule(cu.ctypes.data, N, int(H), flags, float(lower_bound), 1 if conv else 0,
                                  int(workspace_bytes), int(sms), info)
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill_schedule")
    kind = {KDA_SCHEDULE_FUSED: "fused", KDA_SCHEDULE_PLAIN: "plain", KDA_SCHEDULE_SPLIT: "split"}[info[0]]
    return {"kind": kind, "value_split": bool(info[1]), "segments": int(info[2]), "split_sequences": int(info[3])}


def status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def workspace_size() -> int:
    return int(load().kda_workspace_size())


def prefill_workspace_size(total_tokens: int, num_seqs: int, H: int) -> int:
    """Bytes of workspace ``chunk_prefill`` needs (status word + one block per chunk and head)."""
    return int(load().kda_prefill_workspace_size(int(total_tokens), int(num_seqs), int(H)))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_ptr(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def make_workspace(device=None, stream=None, nbytes=None) -> torch.Tensor:
    """Allocate (through torch) and clear a workspace for the calls: at least
    ``workspace_size()`` bytes, or ``nbytes`` if larger (a prefill needs
    ``prefill_workspace_size(...)``)."""
    n = max(workspace_size(), int(nbytes or 0))
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    rc = load().kda_workspace_reset(_ptr(ws), ws.numel(), _stream_ptr(stream, ws.device))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_workspace_reset")
    return ws


def read_device_status(workspace: torch.Tensor, stream=None) -> int:
    val = ctypes.c_uint32(0)
    rc = load().kda_read_device_status(_ptr(workspace), workspace.numel(), ctypes.byref(val),
                                       _stream_ptr(stream, workspace.device))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_read_device_status")
    return int(val.value)


def _token_tensor(x, name, H):
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 3:
        raise ValueError(f"{name}: expected a CUDA bf16 tensor [tokens, H, 128]")
    sh, st = x.shape, x.stride()
    if sh[1] != H or sh[2] != 128 or st[2] != 1 or st[1] != 128:
        raise ValueError(f"{name}: expected [tokens, {H}, 128] with contiguous heads")
    return st[0]


def _beta_stride(b, H):
    if b.dtype != torch.bfloat16 or not b.is_cuda or b.dim() != 2:
        raise ValueError("beta_logits: expected a CUDA bf16 tensor [tokens, H]")
    st = b.stride()
    if b.shape[1] != H or st[1] != 1:
        raise ValueError("beta_logits: expected a CUDA bf16 tensor [tokens, H]")
    return st[0]


def chunk_prefill(q, k, v, g, beta_logits, A_log, dt_bias, cu_seqlens, cu_seqlens_host, *,
                  lower_bound=-5.0, scale=None, state_pool=None, slot_ids=None, load_initial=False,
                  final_to_pool=False, out=None, final_state=None, norm=None, conv=None, workspace=None,
                  stream=None, path=None):
    """``kda_chunk_prefill``.  Returns ``(out, final_state)`` (final_state is None
    when the final states go to the pool).  ``norm``: an :class:`OutputNorm` applied to the output rows.
    ``path``: None (the library picks), ``"two_pass"`` (``KDA_TWO_PASS``), ``"fused"`` (``KDA_FUSED``) or
    ``"overlap"`` (``KDA_OVERLAP``)."""
    lib = load()
    H = q.shape[1]
    qs = _token_tensor(q, "q", H)
    if _token_tensor(k, "k", H) != qs or _token_tensor(v, "v", H) != qs:
        raise ValueError("q, k and v must share one token stride")
    gs = _token_tensor(g, "g", H)
    bs = _beta_stride(beta_logits, H)
    cu_host = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
    if cu_host.is_cuda:
        raise ValueError("cu_seqlens_host must be in host memory")
    N = cu_host.numel() - 1
    T_total = q.shape[0]
    dev = q.device
    if out is None:
        out = torch.empty((T_total, H, 128), dtype=torch.bfloat16, device=dev)
    os_ = _token_tensor(out, "out", H)
    if not final_to_pool and final_state is None:
        final_state = torch.empty((N, H, 128, 128), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = make_workspace(dev, stream, prefill_workspace_size(T_total, N, H))
    flags = (KDA_LOAD_INITIAL if load_initial else 0) | (KDA_FINAL_TO_POOL if final_to_pool else 0) | \
        {None: 0, "two_pass": KDA_TWO_PASS, "fused": KDA_FUSED, "overlap": KDA_OVERLAP}[path]
    if scale is None:
        scale = 1.0 / math.sqrt(128.0)
    rc = lib.kda_chunk_prefill(
        _ptr(q), _ptr(k), _ptr(v), qs, _ptr(g), gs, _ptr(beta_logits), bs, _ptr(A_log), _ptr(dt_bias),
        float(lower_bound), float(scale), _ptr(cu_seqlens), cu_host.data_ptr(), N, H,
        _ptr(state_pool), 0 if state_pool is None else state_pool.shape[0], _ptr(slot_ids), flags,
        _ptr(out), os_, _norm_arg(norm, H), _conv_arg(conv), _ptr(None if final_to_pool else final_state),
        _ptr(workspace), workspace.numel(), _stream_ptr(stream, dev))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_prefill")
    return out, (None if final_to_pool else final_state)


def recurrent_verify(q, k, v, g, beta_logits, A_log, dt_bias, state_pool, slot_ids, T, *,
                     lower_bound=-5.0, scale=None, out=None, intermediate_states=None, norm=None, conv=None,
                     workspace=None, stream=None):
    """``kda_recurrent_verify``.  Returns ``(out, intermediate_states)``.  ``norm``: an :class:`OutputNorm`
    applied to the output rows."""
    lib = load()
    H = q.shape[1]
    qs = _token_tensor(q, "q", H)
    if _token_tensor(k, "k", H) != qs or _token_tensor(v, "v", H) != qs:
        raise ValueError("q, k and v must share one token stride")
    gs = _token_tensor(g, "g", H)
    bs = _beta_stride(beta_logits, H)
    B = slot_ids.numel()
    dev = q.device
    if out is None:
        out = torch.empty((B * T, H, 128), dtype=torch.bfloat16, device=dev)
    os_ = _token_tensor(out, "out", H)
    if intermediate_states is None:
        intermediate_states = torch.empty((B, T, H, 128, 128), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = make_workspace(dev, stream)
    if scale is None:
        scale = 1.0 / math.sqrt(128.0)
    rc = lib.kda_recurrent_verify(
        _ptr(q), _ptr(k), _ptr(v), qs, _ptr(g), gs, _ptr(beta_logits), bs, _ptr(A_log), _ptr(dt_bias),
        float(lower_bound), float(scale), B, int(T), H, _ptr(state_pool), state_pool.shape[0], _ptr(slot_ids),
        _ptr(out), os_, _norm_arg(norm, H), _conv_arg(conv), _ptr(intermediate_states), _ptr(workspace),
        workspace.numel(), _stream_ptr(stream, dev))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_recurrent_verify")
    return out, intermediate_states


def commit_accepted(state_pool, slot_ids, num_accepted, intermediate_states, *, conv=None, workspace=None,
                    stream=None):
    """``kda_commit_accepted``: pool[slot_ids[b]] = intermediate_states[b, num_accepted[b] - 1] (and, with
    ``conv``, conv.window_pool[slot_ids[b]] = conv.step_windows[b, num_accepted[b] - 1])."""
    lib = load()
    B, T, H = intermediate_states.shape[:3]
    dev = state_pool.device
    for name, t, dt in (("slot_ids", slot_ids, torch.int32), ("num_accepted", num_accepted, torch.int32)):
        if t.dtype != dt or not t.is_cuda or t.numel() != B:
            raise ValueError(f"{name}: expected a CUDA int32 tensor of {B} entries")
    if workspace is None:
        workspace = make_workspace(dev, stream)
    rc = lib.kda_commit_accepted(_ptr(state_pool), state_pool.shape[0], _ptr(slot_ids), _ptr(num_accepted),
                                 _ptr(intermediate_states), _conv_arg(conv), B, T, H, _ptr(workspace),
                                 workspace.numel(),
                                 _stream_ptr(stream, dev))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_commit_accepted")
    return state_pool


def _token_struct(tensors, H):
    """(q, k, v, g, beta_logits) -> (TokenTensors, tokens)."""
    q, k, v, g, beta = tensors
    qs = _token_tensor(q, "q", H)
    if _token_tensor(k, "k", H) != qs or _token_tensor(v, "v", H) != qs:
        raise ValueError("q, k and v must share one token stride")
    if k.shape[0] != q.shape[0] or v.shape[0] != q.shape[0] or g.shape[0] != q.shape[0] or beta.shape[0] != q.shape[0]:
        raise ValueError("q, k, v, g and beta_logits must have the same number of tokens")
    tt = TokenTensors(q.data_ptr(), k.data_ptr(), v.data_ptr(), qs, g.data_ptr(), _token_tensor(g, "g", H),
                      beta.data_ptr(), _beta_stride(beta, H))
    return tt, q.shape[0]


def spec_step(prefill, cu_seqlens, cu_seqlens_host, spec, T, A_log, dt_bias, state_pool, core_attn_out,
              non_spec_token_indx, spec_token_indx, *, prefill_slot_ids=None, spec_slot_ids=None,
              load_initial=False, final_to_pool=False, final_state=None, intermediate_states=None,
              lower_bound=-5.0, scale=None, norm=None, conv=None, workspace=None, stream=None, path=None):
    """``kda_spec_step``: the prefill segment and the verify segment of one speculative-decoding step, their
    outputs written into ``core_attn_out`` rows ``non_spec_token_indx`` / ``spec_token_indx``.
    ``path``: the prefill segment's path, as in :func:`chunk_prefill`.

    ``prefill`` and ``spec`` are ``(q, k, v, g, beta_logits)`` tuples (or None for an absent segment);
    ``norm``: an :class:`OutputNorm` over the rows of ``core_attn_out``.
    Returns ``(core_attn_out, final_state, intermediate_states)``."""
    lib = load()
    H = core_attn_out.shape[1]
    os_ = _token_tensor(core_attn_out, "core_attn_out", H)
    dev = core_attn_out.device
    pre = spc = None
    N = B = Tp = 0
    cu_host = None
    if prefill is not None:
        pre, Tp = _token_struct(prefill, H)
        cu_host = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
        if cu_host.is_cuda:
            raise ValueError("cu_seqlens_host must be in host memory")
        N = cu_host.numel() - 1
        if not final_to_pool and final_state is None:
            final_state = torch.empty((N, H, 128, 128), dtype=torch.float32, device=dev)
    if spec is not None:
        spc, Bt = _token_struct(spec, H)
        if Bt % T:
            raise ValueError("spec segment: tokens must be a multiple of T")
        B = Bt // T
        if intermediate_states is None:
            intermediate_states = torch.empty((B, T, H, 128, 128), dtype=torch.float32, device=dev)
    for name, idx, n in (("non_spec_token_indx", non_spec_token_indx, Tp), ("spec_token_indx", spec_token_indx, B * T)):
        if n and (idx is None or idx.dtype != torch.int32 or not idx.is_cuda or idx.numel() != n or not idx.is_contiguous()):
            raise ValueError(f"{name}: expected a contiguous CUDA int32 tensor of {n} entries")
    if workspace is None:
        workspace = make_workspace(dev, stream, prefill_workspace_size(Tp, N, H))
    flags = (KDA_LOAD_INITIAL if load_initial else 0) | (KDA_FINAL_TO_POOL if final_to_pool else 0) | \
        {None: 0, "two_pass": KDA_TWO_PASS, "fused": KDA_FUSED, "overlap": KDA_OVERLAP}[path]
    if scale is None:
        scale = 1.0 / math.sqrt(128.0)
    rc = lib.kda_spec_step(
        None if pre is None else ctypes.byref(pre), _ptr(cu_seqlens),
        None if cu_host is None else cu_host.data_ptr(), N, _ptr(prefill_slot_ids), flags,
        _ptr(None if final_to_pool else final_state), None if spc is None else ctypes.byref(spc), B, int(T),
        _ptr(spec_slot_ids), _ptr(intermediate_states), _ptr(A_log), _ptr(dt_bias), float(lower_bound),
        float(scale), H, _ptr(state_pool), 0 if state_pool is None else state_pool.shape[0], _ptr(core_attn_out),
        os_, core_attn_out.shape[0], _norm_arg(norm, H), _conv_arg(conv), _ptr(non_spec_token_indx),
        _ptr(spec_token_indx),
        _ptr(workspace),
        workspace.numel(), _stream_ptr(stream, dev))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_spec_step")
    return core_attn_out, (None if final_to_pool else final_state), intermediate_states
