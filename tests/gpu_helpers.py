"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
call the library through its binding, and compare against the oracle."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import kda_linear_attention_bounded_gb300 as kda
from kda_linear_attention_bounded_gb300.device import (  # noqa: F401  (re-exported for the tests)
    DevicePrefill, DeviceSpecStep, DeviceVerify, bf16_dev, f32_dev, i32_dev)

# Tolerances of the parity bar (outputs vs the fp64 oracle after the GPU's bf16
# rounding; states in fp32).
OUT_REL_L2 = 1e-2
OUT_MAX_ABS = 3e-2
STATE_REL_L2 = 5e-3


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / den) if den > 0 else float(np.linalg.norm(x))


# The bar for the worst single (sequence or request, head) pair: twice the tensor-wide bar.  A tensor-wide
# figure alone hides one bad pair among many (one pair at 10x the bar moves the tensor-wide rel-L2 of 128 pairs
# by under 1x); the factor 2 leaves room for the spread of a pair's error around the tensor-wide value.
PAIR_FACTOR = 2.0
PAIR_FLOOR = 0.5   # an output pair's reference norm counts as at least half that of as many typical rows

# Where each check appends its figures (one JSON line per check), when set: the margins table is built from it.
_LOG = os.environ.get("KDA_PARITY_LOG")


def _log(kind, what, **fig):
    if _LOG:
        with open(_LOG, "a") as f:
            f.write(json.dumps({"kind": kind, "what": what, **fig}) + "\n")


def _pair_rel(err2, ref2):
    """Per-pair rel-L2 from per-pair sums of squared errors and of squared reference values; a pair whose
    reference is zero reports its absolute error norm."""
    err2 = np.asarray(err2, dtype=np.float64)
    ref2 = np.asarray(ref2, dtype=np.float64)
    out = np.sqrt(err2)
    nz = ref2 > 0
    out[nz] = np.sqrt(err2[nz] / ref2[nz])
    return out


def _token_segments(rows, segments):
    """[start, end) row ranges of the pairs' sequences: ``segments`` is a cu_seqlens array (prefill rows in token
    order), an int T (verify: consecutive blocks of T rows), or None (all rows one segment)."""
    if segments is None:
        return [(0, rows)]
    if isinstance(segments, (int, np.integer)):
        T = int(segments)
        return [(b * T, (b + 1) * T) for b in range(rows // T)]
    cu = np.asarray(segments, dtype=np.int64)
    return [(int(a), int(b)) for a, b in zip(cu[:-1], cu[1:]) if b > a]


ROW_BINS = ((0.0, 0.05), (0.05, 0.2), (0.2, 0.5), (0.5, 2.0), (2.0, float("inf")))


def row_error_bins(x, ref):
    """Relative error of every (row, head) output vector, binned by its reference norm over the median norm:
    [(bin, rows, mean, max)].  Informational: a row far below the typical output norm keeps the absolute error
    of the bf16 products around it, so its relative error grows."""
    if x.ndim != 3 or not x.size:
        return []
    nrm = np.linalg.norm(ref, axis=2).ravel()
    err = np.linalg.norm(x - ref, axis=2).ravel()
    live = nrm > 0
    if not live.any():
        return []
    rel = err[live] / nrm[live]
    scaled = nrm[live] / np.median(nrm[live])
    out = []
    for lo, hi in ROW_BINS:
        m = (scaled >= lo) & (scaled < hi)
        if m.any():
            out.append([lo, hi, int(m.sum()), float(rel[m].mean()), float(rel[m].max())])
    return out


def check_out(out_gpu, out_ref, what, segments=None):
    """Outputs ``[rows, H, d]`` against the oracle: tensor-wide rel-L2 and max-abs, and the rel-L2 of every
    (segment, head) pair (``segments`` as in ``_token_segments``), the worst within ``PAIR_FACTOR`` x the bar.
    A pair's error is taken relative to the larger of its reference norm and half the norm that as many rows of
    the tensor's mean squared row norm would have: the output of a sequence of a few tokens can be far smaller
    than a typical row (its Q+ S and P U terms nearly cancel), and the bf16 products' absolute error around it
    then makes its own relative error meaningless."""
    x = out_gpu.float().cpu().numpy().astype(np.float64) if torch.is_tensor(out_gpu) else np.asarray(out_gpu, np.float64)
    ref = np.asarray(out_ref, dtype=np.float64)
    assert np.isfinite(x).all(), f"{what}: non-finite GPU output"
    r = rel_l2(x, ref)
    m = float(np.abs(x - ref).max()) if x.size else 0.0
    worst = (0.0, None)
    if x.size and x.ndim == 3:
        d2 = ((x - ref) ** 2).sum(axis=2)      # [rows, H]
        r2 = (ref ** 2).sum(axis=2)
        row_sq = float(r2.mean())              # mean squared norm of one (row, head) output vector
        for (a, b) in _token_segments(x.shape[0], segments):
            pr = _pair_rel(d2[a:b].sum(axis=0), np.maximum(r2[a:b].sum(axis=0), PAIR_FLOOR ** 2 * (b - a) * row_sq))
            h = int(np.argmax(pr))
            if pr[h] > worst[0]:
                worst = (float(pr[h]), (a, b, h))
    _log("out", what, rel_l2=r, max_abs=m, worst_pair=worst[0], worst_at=worst[1], rows=row_error_bins(x, ref))
    assert r <= OUT_REL_L2 and m <= OUT_MAX_ABS, (
        f"{what}: rel-L2 {r:.3e} (<= {OUT_REL_L2}), max-abs {m:.3e} (<= {OUT_MAX_ABS}); "
        f"worst (rows, head) {worst[1]}: {worst[0]:.3e}")
    assert worst[0] <= PAIR_FACTOR * OUT_REL_L2, (
        f"{what}: worst (rows, head) pair {worst[1]} rel-L2 {worst[0]:.3e} (<= {PAIR_FACTOR * OUT_REL_L2}); "
        f"tensor-wide {r:.3e}")
    return r, m


def check_state(s_gpu, s_ref, what):
    """States against the oracle: tensor-wide rel-L2 and the rel-L2 of every (sequence or request, head) pair,
    the worst within ``PAIR_FACTOR`` x the bar.  Shapes: ``[N, H, d, d]`` (final states; pair (n, h)),
    ``[B, T, H, d, d]`` (per-step states; pair (b, h) over its T steps), ``[H, d, d]`` or ``[d, d]``."""
    x = s_gpu.cpu().numpy().astype(np.float64) if torch.is_tensor(s_gpu) else np.asarray(s_gpu, np.float64)
    ref = np.asarray(s_ref, dtype=np.float64)
    assert np.isfinite(x).all(), f"{what}: non-finite GPU state"
    r = rel_l2(x, ref)
    d2, r2 = (x - ref) ** 2, ref ** 2
    axes = {5: (1, 3, 4), 4: (2, 3), 3: (1, 2), 2: (0, 1)}.get(x.ndim)
    worst, at = 0.0, None
    if axes is not None and x.size:
        pr = _pair_rel(d2.sum(axis=axes), r2.sum(axis=axes))
        idx = np.unravel_index(int(np.argmax(pr)), pr.shape) if pr.ndim else ()
        worst, at = float(np.max(pr)), tuple(int(i) for i in idx)
    _log("state", what, rel_l2=r, worst_pair=worst, worst_at=at)
    assert r <= STATE_REL_L2, f"{what}: rel-L2 {r:.3e} (<= {STATE_REL_L2}); worst pair {at}: {worst:.3e}"
    assert worst <= PAIR_FACTOR * STATE_REL_L2, (
        f"{what}: worst pair {at} rel-L2 {worst:.3e} (<= {PAIR_FACTOR * STATE_REL_L2}); tensor-wide {r:.3e}")
    return r


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
