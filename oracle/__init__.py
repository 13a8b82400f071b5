"""fp64 CPU oracle for the KDA bounded-gate recurrence -- test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA path: the
arithmetic lives in ``kda_oracle.c`` (plain C, double precision, token by
token), built with gcc into ``oracle/_build`` and called through ctypes.  The
code here only marshals NumPy arrays.

bf16 tensors are passed as their uint16 bit patterns and widened exactly
inside the C code.  Pins: ``tests/test_oracle_pins.py`` (worked example,
closed forms, invariants, brute force) and ``tests/test_oracle_mutants.py``
(planted mistakes that the pins must catch).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")

#: the l2-norm epsilon the pages leave open (adopted reading)
L2NORM_EPS = 1e-6


def build(force: bool = False, src: str = SOURCE, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE double semantics)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", tmp, src, "-lm"],
                       check=True)
        os.replace(tmp, out)
    return out


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def bf16_widen(bits):
    """bf16 bit patterns -> fp64 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """ctypes front end of one build of ``kda_oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P, I, Dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.kda_oracle_run.argtypes = [P, P, P, P, P, P, P, Dbl, Dbl, Dbl, P, I, I, I, I, I, I, P, P, P, P, I]
        lib.kda_oracle_run.restype = I
        lib.kda_oracle_run_conv.argtypes = [P, P, P, P, P, P, P, Dbl, Dbl, Dbl, P, I, I, I, I, I, I, P, P, P, P, I,
                                            P, I, I, P, P, P]
        lib.kda_oracle_run_conv.restype = I
        lib.kda_oracle_conv_step.argtypes = [P, P, P, I, I, I, P]
        lib.kda_oracle_conv_step.restype = None
        lib.kda_oracle_core.argtypes = [P, P, P, P, P, I, I, I, Dbl, P, P, P]
        lib.kda_oracle_core.restype = I
        lib.kda_oracle_gate.argtypes = [P, P, Dbl, Dbl, I, P]
        lib.kda_oracle_gate.restype = None
        lib.kda_oracle_l2norm.argtypes = [P, I, Dbl, P]
        lib.kda_oracle_l2norm.restype = None
        lib.kda_oracle_gated_rmsnorm.argtypes = [P, P, P, Dbl, I, I, P, P]
        lib.kda_oracle_gated_rmsnorm.restype = None
        self.lib = lib

    def run(self, q, k, v, g, beta_logits, A_log, dt_bias, lower_bound, scale, cu_seqlens, *,
            S0=None, heads=None, record_steps=False, want_final=True, nthreads=None,
            eps=L2NORM_EPS):
        """Run the recurrence over a packed varlen batch.

        q, k, g: uint16 bf16 bits ``[T, H, dk]``; v: ``[T, H, dv]``; beta_logits: ``[T, H]``;
        A_log: ``[H]``; dt_bias: ``[H, dk]``; cu_seqlens: ``[N+1]``;
        S0: ``[N, H, dk, dv]`` (any float dtype, widened to fp64) or None for zero.
        heads: ``(begin, end)`` computes a subset of heads (the others stay NaN).

        Returns ``out [T, H, dv]``, ``S_final [N, H, dk, dv]`` (or None) and
        ``steps [T, H, dk, dv]`` (state after each token, or None), all fp64.
        """
        q, k, v, g = (_c(x, np.uint16) for x in (q, k, v, g))
        beta_logits = _c(beta_logits, np.uint16)
        A_log = _c(A_log, np.float32)
        dt_bias = _c(dt_bias, np.float32)
        cu = _c(cu_seqlens, np.int32)
        T, H, dk = q.shape
        dv = v.shape[2]
        N = cu.shape[0] - 1
        hb, he = (0, H) if heads is None else heads
        S0d = None if S0 is None else _c(S0, np.float64)
        out = np.full((T, H, dv), np.nan)
        S_final = np.full((N, H, dk, dv), np.nan) if want_final else None
        steps = np.full((T, H, dk, dv), np.nan) if record_steps else None
        rc = self.lib.kda_oracle_run(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(A_log), _ptr(dt_bias),
            float(lower_bound), float(scale), float(eps), _ptr(cu), N, H, dk, dv, hb, he,
            _ptr(S0d), _ptr(out), _ptr(S_final), _ptr(steps), int(nthreads or default_threads()))
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (rc={rc})")
        return out, S_final, steps

    def run_conv(self, q, k, v, g, beta_logits, A_log, dt_bias, lower_bound, scale, cu_seqlens, conv_w, silu, *,
                 win0=None, S0=None, heads=None, record_steps=False, record_windows=False, want_final=True,
                 nthreads=None, eps=L2NORM_EPS):
        """:meth:`run` with q, k and v first passed through their short causal convolutions.

        conv_w: ``[3 (q, k, v), H, d, W]`` (tap W-1 on the current input); silu: apply SiLU after each
        convolution; win0: ``[N, 3, W-1, H, d]`` initial windows (raw inputs, oldest first) or None for zero.
        Returns ``out``, ``S_final``, ``steps`` as :meth:`run`, then ``win_final [N, 3, W-1, H, d]`` (or None)
        and ``win_steps [T, 3, W-1, H, d]`` (the window after each token, or None), all fp64."""
        q, k, v, g = (_c(x, np.uint16) for x in (q, k, v, g))
        beta_logits = _c(beta_logits, np.uint16)
        A_log = _c(A_log, np.float32)
        dt_bias = _c(dt_bias, np.float32)
        cu = _c(cu_seqlens, np.int32)
        T, H, dk = q.shape
        dv = v.shape[2]
        N = cu.shape[0] - 1
        w = _c(conv_w, np.float64)
        W = w.shape[-1]
        if w.shape != (3, H, dk, W) or dk != dv:
            raise ValueError("conv_w must be [3, H, d, W] with dk == dv == d")
        hb, he = (0, H) if heads is None else heads
        S0d = None if S0 is None else _c(S0, np.float64)
        w0 = None if win0 is None else _c(win0, np.float64)
        out = np.full((T, H, dv), np.nan)
        S_final = np.full((N, H, dk, dv), np.nan) if want_final else None
        steps = np.full((T, H, dk, dv), np.nan) if record_steps else None
        wf = np.full((N, 3, W - 1, H, dk), np.nan) if want_final else None
        ws = np.full((T, 3, W - 1, H, dk), np.nan) if record_windows else None
        rc = self.lib.kda_oracle_run_conv(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(A_log), _ptr(dt_bias),
            float(lower_bound), float(scale), float(eps), _ptr(cu), N, H, dk, dv, hb, he,
            _ptr(S0d), _ptr(out), _ptr(S_final), _ptr(steps), int(nthreads or default_threads()),
            _ptr(w), W, 1 if silu else 0, _ptr(w0), _ptr(wf), _ptr(ws))
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (rc={rc})")
        return out, S_final, steps, wf, ws

    def conv_step(self, win, x, w, silu):
        """One step of one short convolution row: returns ``(y, new window)``; win ``[W-1, d]``, x ``[d]``,
        w ``[d, W]``."""
        win = _c(win, np.float64).copy()
        x = _c(x, np.float64)
        w = _c(w, np.float64)
        d, W = w.shape
        y = np.empty(d)
        self.lib.kda_oracle_conv_step(_ptr(win), _ptr(x), _ptr(w), W, d, 1 if silu else 0, _ptr(y))
        return y, win

    def run_prefill(self, inp, **kw):
        """Oracle for a prefill workload object (the ``inputs`` module's ``PrefillInputs``)."""
        S0 = inp.initial_states() if inp.load_initial else None
        if inp.conv is not None:   # returns the final windows too
            c = inp.conv
            win0 = bf16_widen(c.pool[inp.slot_ids]) if inp.load_initial else None
            out, S, steps, wf, _ = self.run_conv(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.A_log, inp.dt_bias,
                                                 inp.lower_bound, inp.scale, inp.cu_seqlens, c.weight, c.silu,
                                                 win0=win0, S0=S0, **kw)
            return out, S, steps, wf
        return self.run(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.A_log, inp.dt_bias,
                        inp.lower_bound, inp.scale, inp.cu_seqlens, S0=S0, **kw)

    def run_verify(self, inp, **kw):
        """Oracle for a verify workload: ``B`` sequences of ``T`` tokens seeded from the pool.

        Returns ``out [B*T, H, dv]`` and ``steps [B, T, H, dk, dv]`` (state after
        each draft token)."""
        cu = (np.arange(inp.B + 1) * inp.T).astype(np.int32)
        S0 = inp.pool[inp.slot_ids]
        if inp.conv is not None:   # returns the per-step windows too: [B, T, 3, W-1, H, d]
            c = inp.conv
            out, _, steps, _, ws = self.run_conv(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.A_log, inp.dt_bias,
                                                 inp.lower_bound, inp.scale, cu, c.weight, c.silu,
                                                 win0=bf16_widen(c.pool[inp.slot_ids]), S0=S0, record_steps=True,
                                                 record_windows=True, want_final=False, **kw)
            return (out, steps.reshape(inp.B, inp.T, inp.H, steps.shape[-2], steps.shape[-1]),
                    ws.reshape(inp.B, inp.T, *ws.shape[1:]))
        out, _, steps = self.run(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.A_log, inp.dt_bias,
                                 inp.lower_bound, inp.scale, cu, S0=S0, record_steps=True,
                                 want_final=False, **kw)
        return out, steps.reshape(inp.B, inp.T, inp.H, steps.shape[-2], steps.shape[-1])

    def core(self, qh, kh, v, lam, beta, scale, S0=None):
        """Recurrence on one (sequence, head) with normalised q/k, log-decay and beta given.

        qh, kh: ``[T, dk]``; v: ``[T, dv]``; lam: ``[T, dk]``; beta: ``[T]``.
        Returns ``out [T, dv]``, final ``S [dk, dv]`` and ``steps [T, dk, dv]``.
        """
        qh, kh, v, lam = (_c(x, np.float64) for x in (qh, kh, v, lam))
        beta = _c(beta, np.float64)
        T, dk = qh.shape
        dv = v.shape[1]
        S = np.zeros((dk, dv)) if S0 is None else _c(S0, np.float64).copy()
        out = np.empty((T, dv))
        steps = np.empty((T, dk, dv))
        rc = self.lib.kda_oracle_core(_ptr(qh), _ptr(kh), _ptr(v), _ptr(lam), _ptr(beta), T, dk, dv,
                                      float(scale), _ptr(S), _ptr(out), _ptr(steps))
        if rc != 0:
            raise ValueError("oracle core rejected the arguments")
        return out, S, steps

    def gate(self, g, dt_bias, A_log, lower_bound):
        """Per-channel log-decay of one (token, head)."""
        g = _c(g, np.float64)
        dtb = _c(dt_bias, np.float64)
        lam = np.empty_like(g)
        self.lib.kda_oracle_gate(_ptr(g), _ptr(dtb), float(A_log), float(lower_bound), g.shape[0], _ptr(lam))
        return lam

    def l2norm(self, x, eps=L2NORM_EPS):
        x = _c(x, np.float64)
        out = np.empty_like(x)
        self.lib.kda_oracle_l2norm(_ptr(x), x.shape[0], float(eps), _ptr(out))
        return out

    def gated_rmsnorm(self, x, z, w, eps):
        """Sigmoid-gated RMSNorm over the last axis: ``x`` rows (any float, widened to fp64), ``z`` the bf16
        gate bits of the same shape, ``w`` the weight of the last axis.  Returns ``y`` (fp64, shape of x)
        and ``rstd`` (fp64, x's shape without the last axis)."""
        x = _c(x, np.float64)
        z = _c(z, np.uint16)
        w = _c(w, np.float64)
        if z.shape != x.shape or w.shape != (x.shape[-1],):
            raise ValueError("gated_rmsnorm: z must match x and w the last axis")
        d = x.shape[-1]
        rows = x.size // d if d else 0
        y = np.empty_like(x)
        rstd = np.empty(x.shape[:-1])
        self.lib.kda_oracle_gated_rmsnorm(_ptr(x), _ptr(z), _ptr(w), float(eps), rows, d, _ptr(y), _ptr(rstd))
        return y, rstd


_default = None


def get() -> Oracle:
    """The oracle built from ``kda_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def run(*a, **kw):
    return get().run(*a, **kw)


def run_prefill(inp, **kw):
    return get().run_prefill(inp, **kw)


def run_verify(inp, **kw):
    return get().run_verify(inp, **kw)


def core(*a, **kw):
    return get().core(*a, **kw)


def gate(*a, **kw):
    return get().gate(*a, **kw)


def l2norm(*a, **kw):
    return get().l2norm(*a, **kw)


def gated_rmsnorm(*a, **kw):
    return get().gated_rmsnorm(*a, **kw)


def run_conv(*a, **kw):
    return get().run_conv(*a, **kw)


def conv_step(*a, **kw):
    return get().conv_step(*a, **kw)
