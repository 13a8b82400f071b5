"""Pins of the fp64 oracle against facts the definition fixes.

Each ``pin_*`` function takes an :class:`oracle.Oracle` and raises
``AssertionError`` when the oracle disagrees with something that does not
depend on the oracle itself: a hand-derived worked example, closed forms,
invariants of the recurrence, special cases that reduce to a library routine,
and an independent (matrix-product / chunked) formulation.  The set is chosen
so that a plausible slip anywhere in the oracle (a dropped term, a wrong sign,
a transposed index, a swapped operand, a misplaced bias) fails at least one of
them; ``test_oracle_mutants.py`` plants such slips and checks exactly that.

Definition being pinned (vLLM PR #55737 "Use FlashKDA for KDA chunked
prefill", PR summary: bounded gate, in-kernel q/k l2norm, raw beta logits):
  lambda = lower_bound * sigmoid(exp(A_log) (g + dt_bias)),  alpha = exp(lambda)
  S_t = (I - beta k^ k^T) Diag(alpha) S_{t-1} + beta k^ v^T,  o_t = scale S_t^T q^
"""
from __future__ import annotations

import math
import os

import numpy as np
from scipy.special import expit

from kda_linear_attention_bounded_gb300.inputs import f32_to_bf16_bits, bf16_bits_to_f32
import chunk_algebra

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_example_d2.txt")


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    ref = max(1.0, float(np.max(np.abs(b)))) if b.size else 1.0
    assert err <= tol * ref, f"{what}: max |diff| {err:.3e} > {tol:.1e} (scale {ref:.3e})"


def _rand_unit(rng, T, d):
    x = rng.standard_normal((T, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


# --------------------------------------------------------------------------
# worked example (hand-derived, tests/golden/worked_example_d2.txt)
# --------------------------------------------------------------------------

def load_golden(path=GOLDEN):
    params, tokens, outs, final = {}, [], {}, None
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "param":
                params[tok[1]] = float(tok[2])
            elif tok[0] == "token":
                tokens.append([float(x) for x in tok[2:]])
            elif tok[0] == "out":
                outs[int(tok[1])] = [float(x) for x in tok[2:]]
            elif tok[0] == "final":
                final = [float(x) for x in tok[1:]]
    return params, np.array(tokens), outs, np.array(final)


def pin_worked_example(O):
    p, toks, outs, final = load_golden()
    T = toks.shape[0]
    d = 2
    q = f32_to_bf16_bits(toks[:, 0:2].astype(np.float32)).reshape(T, 1, d)
    k = f32_to_bf16_bits(toks[:, 2:4].astype(np.float32)).reshape(T, 1, d)
    v = f32_to_bf16_bits(toks[:, 4:6].astype(np.float32)).reshape(T, 1, d)
    g = f32_to_bf16_bits(toks[:, 6:8].astype(np.float32)).reshape(T, 1, d)
    beta = f32_to_bf16_bits(toks[:, 8:9].astype(np.float32)).reshape(T, 1)
    A_log = np.full(1, p["A_log"], np.float32)
    dtb = np.full((1, d), p["dt_bias"], np.float32)
    cu = np.array([0, T], np.int32)
    out, S, _ = O.run(q, k, v, g, beta, A_log, dtb, p["lower_bound"], p["scale"], cu, eps=p["eps"])
    for t, o in outs.items():
        _close(out[t, 0], o, 1e-12, f"worked example output t={t}")
    _close(S[0, 0].reshape(-1), final, 1e-12, "worked example final state")


# --------------------------------------------------------------------------
# gate and normalisation special cases
# --------------------------------------------------------------------------

def pin_gate_special_cases(O):
    rng = np.random.default_rng(7)
    d = 16
    dtb = rng.standard_normal(d) * 0.1
    lb = -5.0
    # g + dt_bias = 0  =>  lambda = lb / 2 exactly, for any A_log
    for A_log in (0.0, 1.3, math.log(16.0)):
        _close(O.gate(-dtb, dtb, A_log, lb), np.full(d, lb / 2), 1e-15, "gate at g+dt_bias=0")
    # general values against scipy's logistic function
    g = rng.standard_normal(d)
    for A_log in (0.0, 0.7, math.log(11.0)):
        ref = lb * expit(math.exp(A_log) * (g + dtb))
        _close(O.gate(g, dtb, A_log, lb), ref, 1e-14, "gate vs scipy expit")
    # saturation: large positive argument -> lb, large negative -> 0
    _close(O.gate(np.full(d, 60.0), np.zeros(d), 0.0, lb), np.full(d, lb), 1e-15, "gate saturates to lb")
    _close(O.gate(np.full(d, -60.0), np.zeros(d), 0.0, lb), np.zeros(d), 1e-20, "gate saturates to 0")


def pin_l2norm(O):
    rng = np.random.default_rng(8)
    x = rng.standard_normal(128) * 3.0
    y = O.l2norm(x, eps=0.0)
    _close(np.linalg.norm(y), 1.0, 1e-15, "l2norm gives a unit vector")
    _close(y * np.linalg.norm(x), x, 1e-14, "l2norm keeps the direction")
    _close(O.l2norm(np.zeros(8), eps=1e-6), np.zeros(8), 0.0, "l2norm of zero is zero")


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def _full_path_single(O, T, d, seed, S0_std=0.0, lb=-5.0, scale=None, A_log=None):
    rng = np.random.default_rng(seed)
    f = lambda *s: f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32))
    q, k, v, g = f(T, 1, d), f(T, 1, d), f(T, 1, d), f(T, 1, d)
    beta = f(T, 1)
    A_log = np.array([math.log(3.0) if A_log is None else A_log], np.float32)
    dtb = (rng.standard_normal((1, d)) * 0.1).astype(np.float32)
    S0 = (rng.standard_normal((1, 1, d, d)) * S0_std) if S0_std else None
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    return dict(q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dtb=dtb, S0=S0, lb=lb, scale=scale,
                cu=np.array([0, T], np.int32))


def _widen(x):
    return bf16_bits_to_f32(x).astype(np.float64)


def pin_single_token_closed_form(O):
    """T = 1: S_1 = (I - beta k^ k^T) Diag(alpha) S0 + beta k^ v^T,  o = scale S_1^T q^.

    With S0 = 0 this is o = scale * beta * (k^ . q^) * v."""
    d = 128
    for S0_std in (0.0, 0.05):
        c = _full_path_single(O, 1, d, seed=11 + int(S0_std * 100), S0_std=S0_std)
        out, S, _ = O.run(c["q"], c["k"], c["v"], c["g"], c["beta"], c["A_log"], c["dtb"], c["lb"],
                          c["scale"], c["cu"], S0=c["S0"], eps=0.0)
        q, k, v, g = (_widen(c[n])[0, 0] for n in ("q", "k", "v", "g"))
        qh, kh = q / np.linalg.norm(q), k / np.linalg.norm(k)
        beta = expit(_widen(c["beta"])[0, 0])
        alpha = np.exp(c["lb"] * expit(math.exp(float(c["A_log"][0])) * (g + c["dtb"][0].astype(np.float64))))
        S0 = np.zeros((d, d)) if c["S0"] is None else c["S0"][0, 0]
        M = (np.eye(d) - beta * np.outer(kh, kh)) @ np.diag(alpha)
        S1 = M @ S0 + beta * np.outer(kh, v)
        _close(S[0, 0], S1, 1e-12, "T=1 state, product form")
        _close(out[0, 0], c["scale"] * S1.T @ qh, 1e-12, "T=1 output")
        if c["S0"] is None:
            _close(out[0, 0], c["scale"] * beta * float(kh @ qh) * v, 1e-12, "T=1 output, zero state")


def pin_product_form(O):
    """Several tokens: the oracle equals the matrix-product statement of the
    recurrence, evaluated with explicit dk x dk transition matrices."""
    d, T = 8, 23
    rng = np.random.default_rng(12)
    qh, kh = _rand_unit(rng, T, d), _rand_unit(rng, T, d)
    v = rng.standard_normal((T, d))
    lam = -rng.uniform(0.0, 2.0, (T, d))
    beta = rng.uniform(0.0, 1.0, T)
    S0 = rng.standard_normal((d, d))
    out, S, steps = O.core(qh, kh, v, lam, beta, 0.37, S0=S0)
    Sref = S0.copy()
    for t in range(T):
        M = (np.eye(d) - beta[t] * np.outer(kh[t], kh[t])) @ np.diag(np.exp(lam[t]))
        Sref = M @ Sref + beta[t] * np.outer(kh[t], v[t])
        _close(steps[t], Sref, 1e-12, f"product form state t={t}")
        _close(out[t], 0.37 * Sref.T @ qh[t], 1e-12, f"product form output t={t}")
    _close(S, Sref, 1e-12, "product form final state")


def pin_zero_beta_is_pure_decay(O):
    """beta = 0: S_T = Diag(prod_t alpha_t) S0 and o_t = scale (Diag(prod_{s<=t} alpha_s) S0)^T q^_t."""
    d, T = 16, 9
    rng = np.random.default_rng(13)
    qh, kh = _rand_unit(rng, T, d), _rand_unit(rng, T, d)
    v = rng.standard_normal((T, d))
    lam = -rng.uniform(0.0, 1.5, (T, d))
    S0 = rng.standard_normal((d, d))
    out, S, _ = O.core(qh, kh, v, lam, np.zeros(T), 0.5, S0=S0)
    cum = np.cumsum(lam, axis=0)
    for t in range(T):
        _close(out[t], 0.5 * (np.exp(cum[t])[:, None] * S0).T @ qh[t], 1e-12, f"pure decay output t={t}")
    _close(S, np.exp(cum[-1])[:, None] * S0, 1e-12, "pure decay final state")
    # through the full path: beta logit -inf gives beta = 0 exactly
    c = _full_path_single(O, 5, d, seed=14, S0_std=0.1)
    beta = np.full((5, 1), 0xFF80, np.uint16)  # bf16 -inf
    out2, S2, _ = O.run(c["q"], c["k"], c["v"], c["g"], beta, c["A_log"], c["dtb"], c["lb"], c["scale"],
                        c["cu"], S0=c["S0"], eps=0.0)
    g = _widen(c["g"])[:, 0]
    lam = c["lb"] * expit(math.exp(float(c["A_log"][0])) * (g + c["dtb"][0].astype(np.float64)))
    _close(S2[0, 0], np.exp(lam.sum(0))[:, None] * c["S0"][0, 0], 1e-12, "beta logit -inf: pure decay")


def pin_orthonormal_retrieval(O):
    """alpha = 1, beta = 1, orthonormal keys: S_T = sum_i k_i v_i^T, S_T^T k_i = v_i;
    writing an existing key again replaces its value (delta rule)."""
    d = 32
    rng = np.random.default_rng(15)
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    keys = Qm.T[:20]
    vals = rng.standard_normal((20, d))
    lam = np.zeros((20, d))
    _, S, _ = O.core(keys, keys, vals, lam, np.ones(20), 1.0)
    _close(S, keys.T @ vals, 1e-12, "orthonormal keys: S = sum k v^T")
    for i in range(20):
        _close(S.T @ keys[i], vals[i], 1e-12, f"retrieval of key {i}")
    # overwrite key 3 with a new value
    newv = rng.standard_normal((1, d))
    out, S2, _ = O.core(keys[3:4], keys[3:4], newv, np.zeros((1, d)), np.ones(1), 1.0, S0=S)
    _close(S2.T @ keys[3], newv[0], 1e-12, "delta rule overwrites a stored key")
    _close(out[0], newv[0], 1e-12, "querying with the written key returns its new value")
    for i in (0, 5, 19):
        _close(S2.T @ keys[i], vals[i], 1e-12, f"other keys untouched ({i})")


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def pin_split_with_carry(O):
    """run(T1) -> S -> run(T2 from S) equals run(T1 + T2)."""
    d, T = 32, 41
    c = _full_path_single(O, T, d, seed=16, S0_std=0.05)
    whole, Sw, _ = O.run(c["q"], c["k"], c["v"], c["g"], c["beta"], c["A_log"], c["dtb"], c["lb"],
                         c["scale"], c["cu"], S0=c["S0"])
    for cut in (1, 17, 40):
        sl1, sl2 = slice(0, cut), slice(cut, T)
        o1, S1, _ = O.run(c["q"][sl1], c["k"][sl1], c["v"][sl1], c["g"][sl1], c["beta"][sl1], c["A_log"],
                          c["dtb"], c["lb"], c["scale"], np.array([0, cut], np.int32), S0=c["S0"])
        o2, S2, _ = O.run(c["q"][sl2], c["k"][sl2], c["v"][sl2], c["g"][sl2], c["beta"][sl2], c["A_log"],
                          c["dtb"], c["lb"], c["scale"], np.array([0, T - cut], np.int32), S0=S1)
        _close(np.concatenate([o1, o2]), whole, 1e-13, f"split at {cut}: outputs")
        _close(S2, Sw, 1e-13, f"split at {cut}: final state")


def pin_varlen_packing(O):
    """Packing sequences with cu_seqlens equals running each one separately;
    a zero-length sequence returns its initial state."""
    d, H = 16, 3
    rng = np.random.default_rng(17)
    lens = [5, 0, 13, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    f = lambda *s: f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32))
    q, k, v, g, beta = f(T, H, d), f(T, H, d), f(T, H, d), f(T, H, d), f(T, H)
    A_log = np.log(rng.uniform(1, 16, H)).astype(np.float32)
    dtb = (rng.standard_normal((H, d)) * 0.1).astype(np.float32)
    S0 = rng.standard_normal((len(lens), H, d, d)) * 0.1
    out, S, _ = O.run(q, k, v, g, beta, A_log, dtb, -5.0, 0.25, cu, S0=S0)
    for n, L in enumerate(lens):
        sl = slice(cu[n], cu[n + 1])
        o1, S1, _ = O.run(q[sl], k[sl], v[sl], g[sl], beta[sl], A_log, dtb, -5.0, 0.25,
                          np.array([0, L], np.int32), S0=S0[n:n + 1])
        _close(out[sl], o1, 0.0, f"packed vs separate, sequence {n}: outputs")
        _close(S[n], S1[0], 0.0, f"packed vs separate, sequence {n}: state")
    _close(S[1], S0[1], 0.0, "zero-length sequence keeps its initial state")


def pin_linearity(O):
    """For fixed q, k, decay and beta, (out, S_T) is linear in (V, S0)."""
    d, T = 12, 15
    rng = np.random.default_rng(18)
    qh, kh = _rand_unit(rng, T, d), _rand_unit(rng, T, d)
    lam = -rng.uniform(0, 3, (T, d))
    beta = rng.uniform(0, 1, T)
    V1, V2 = rng.standard_normal((2, T, d))
    S1, S2 = rng.standard_normal((2, d, d))
    a, b = 0.75, -1.5
    o1, F1, _ = O.core(qh, kh, V1, lam, beta, 0.3, S0=S1)
    o2, F2, _ = O.core(qh, kh, V2, lam, beta, 0.3, S0=S2)
    o3, F3, _ = O.core(qh, kh, a * V1 + b * V2, lam, beta, 0.3, S0=a * S1 + b * S2)
    _close(o3, a * o1 + b * o2, 1e-12, "linearity: outputs")
    _close(F3, a * F1 + b * F2, 1e-12, "linearity: state")


def pin_qk_scale_invariance(O):
    """Scaling q and k by a power of two (exact in bf16) leaves the result unchanged."""
    d, T = 32, 11
    c = _full_path_single(O, T, d, seed=19, S0_std=0.05)
    base, Sb, _ = O.run(c["q"], c["k"], c["v"], c["g"], c["beta"], c["A_log"], c["dtb"], c["lb"], c["scale"],
                        c["cu"], S0=c["S0"], eps=0.0)
    q4 = f32_to_bf16_bits(bf16_bits_to_f32(c["q"]) * 4)
    k8 = f32_to_bf16_bits(bf16_bits_to_f32(c["k"]) * 0.125)
    sc, Ss, _ = O.run(q4, k8, c["v"], c["g"], c["beta"], c["A_log"], c["dtb"], c["lb"], c["scale"],
                      c["cu"], S0=c["S0"], eps=0.0)
    _close(sc, base, 1e-13, "q/k scale invariance: outputs")
    _close(Ss, Sb, 1e-13, "q/k scale invariance: state")


def pin_contraction_bound(O):
    """||S_t||_F <= ||S_{t-1}||_F + beta_t ||v_t||  (||I - beta k^k^T||_2 <= 1, alpha <= 1)."""
    d, T = 24, 60
    rng = np.random.default_rng(20)
    qh, kh = _rand_unit(rng, T, d), _rand_unit(rng, T, d)
    v = rng.standard_normal((T, d))
    lam = -rng.uniform(0, 0.2, (T, d))
    beta = rng.uniform(0, 1, T)
    S0 = rng.standard_normal((d, d))
    _, _, steps = O.core(qh, kh, v, lam, beta, 1.0, S0=S0)
    prev = np.linalg.norm(S0)
    for t in range(T):
        cur = np.linalg.norm(steps[t])
        assert cur <= prev + beta[t] * np.linalg.norm(v[t]) + 1e-12, f"contraction bound violated at t={t}"
        prev = cur


def pin_chunked_equals_sequential(O):
    """The chunk-parallel algebra (exact ratios, chunk 1/4/16/64) and the
    kernel's anchored 16- and 32-row sub-block factorisations (chunk 64) reproduce
    the token-by-token oracle, for weak and strong decay."""
    rng = np.random.default_rng(21)
    for d, T, lam_hi in ((8, 150, 0.05), (8, 200, 5.0), (128, 130, 5.0), (128, 97, 0.02)):
        qh, kh = _rand_unit(rng, T, d), _rand_unit(rng, T, d)
        v = rng.standard_normal((T, d))
        lam = -rng.uniform(0, lam_hi, (T, d))
        beta = rng.uniform(0, 1, T)
        S0 = rng.standard_normal((d, d)) * 0.1
        ref, Sref, _ = O.core(qh, kh, v, lam, beta, 0.2, S0=S0)
        for C in (1, 4, 16, 64):
            o, S = chunk_algebra.chunked_exact(qh, kh, v, lam, beta, 0.2, S0, C)
            _close(o, ref, 1e-10, f"chunked (C={C}, d={d}) outputs")
            _close(S, Sref, 1e-10, f"chunked (C={C}, d={d}) state")
        for sub in (16, 32):   # the kernel's two sub-block sizes
            o, S, worst = chunk_algebra.chunked_anchored(qh, kh, v, lam, beta, 0.2, S0, 64, sub)
            _close(o, ref, 1e-10, f"anchored chunk (d={d}, {sub}-row blocks) outputs")
            _close(S, Sref, 1e-10, f"anchored chunk (d={d}, {sub}-row blocks) state")
            assert worst <= sub // 2 * lam_hi + 1e-9


# --------------------------------------------------------------------------
# sigmoid-gated RMSNorm of the output rows
# --------------------------------------------------------------------------

def pin_gated_rmsnorm(O):
    """Closed forms of y = x rstd w sigmoid(z), rstd = (mean x^2 + eps)^(-1/2): a constant row (the mean, not the
    sum, of squares; eps under the root; the gate after the norm, varying along the row; a sigmoid of it; the
    weight per channel), the zero gate (sigmoid 0 = 1/2 exactly) and the scale invariance it leaves."""
    d = 128
    rng = np.random.default_rng(31)
    z = f32_to_bf16_bits(rng.standard_normal(d).astype(np.float32) * 2.0)
    zd = bf16_bits_to_f32(z).astype(np.float64)
    w = rng.uniform(0.5, 1.5, d)
    for c, eps in ((3.0, 1e-6), (-0.25, 1e-5), (1e-3, 1e-6)):
        y, rstd = O.gated_rmsnorm(np.full(d, c), z, w, eps)
        inv = 1.0 / math.sqrt(c * c + eps)
        _close(rstd * 1e-3, inv * 1e-3, 1e-14, f"rstd of a constant row {c}")
        _close(y, c * inv * w * expit(zd), 1e-14, f"gated norm of a constant row {c}")
    x = rng.standard_normal((5, d)) * rng.uniform(0.1, 10.0, (5, 1))
    zero = np.zeros((5, d), np.uint16)   # bf16 +0.0
    y, rstd = O.gated_rmsnorm(x, zero, np.ones(d), 0.0)
    _close((y ** 2).mean(axis=1), np.full(5, 0.25), 1e-13, "zero gate, eps 0: mean of y^2 is 1/4")
    _close(y * 2.0 / rstd[:, None], x, 1e-12, "zero gate: y = x rstd / 2")
    y2, _ = O.gated_rmsnorm(x * 7.5, zero, np.ones(d), 0.0)
    _close(y2, y, 1e-13, "scale invariance with eps 0")
    ms = (x ** 2).mean(axis=1)
    y3, _ = O.gated_rmsnorm(x, zero, np.ones(d), 0.3)
    _close((y3 ** 2).mean(axis=1), 0.25 * ms / (ms + 0.3), 1e-13, "eps under the root: mean y^2 = ms / (ms + eps) / 4")


# --------------------------------------------------------------------------
# short causal convolutions of q, k, v
# --------------------------------------------------------------------------

def pin_short_conv_step(O):
    """One channel row of the short convolution: the impulse response reads the taps in order (tap W-1 on the
    current input), a random signal matches numpy's convolve with the reversed taps, SiLU is z sigmoid(z), and
    the window ends holding the last W-1 inputs (oldest first)."""
    rng = np.random.default_rng(41)
    d, W, T = 6, 4, 23
    # impulse at t = 0 from a zero window: y_t = w[:, Wi-1-t], for the kernels' width and others
    for Wi in (1, 2, 3, 4, 5):
        wi = rng.standard_normal((d, Wi))
        win = np.zeros((Wi - 1, d))
        for t in range(Wi + 2):
            x = np.ones(d) if t == 0 else np.zeros(d)
            y, win = O.conv_step(win, x, wi, False)
            _close(y, wi[:, Wi - 1 - t] if t < Wi else np.zeros(d), 1e-15, f"W = {Wi}: impulse response at t = {t}")
    w = rng.standard_normal((d, W))
    # a random signal, zero window: numpy convolve with reversed taps; SiLU on top
    xs = rng.standard_normal((T, d))
    for silu in (False, True):
        win = np.zeros((W - 1, d))
        ys = []
        for t in range(T):
            y, win = O.conv_step(win, xs[t], w, silu)
            ys.append(y)
        ref = np.stack([np.convolve(xs[:, c], w[c, ::-1])[:T] for c in range(d)], axis=1)
        if silu:
            ref = ref * expit(ref)
        _close(np.array(ys), ref, 1e-13, f"random signal vs numpy convolve (silu={silu})")
        _close(win, xs[T - (W - 1):], 0.0, "the window holds the last W-1 inputs, oldest first")
    # a carried window continues the signal: the first W-1 outputs see it
    win0 = rng.standard_normal((W - 1, d))
    y0, _ = O.conv_step(win0, xs[0], w, False)
    _close(y0, (w[:, :W - 1] * win0.T).sum(axis=1) + w[:, W - 1] * xs[0], 1e-14, "first output uses the window")


def pin_short_conv_in_the_path(O):
    """The convolutions feed the recurrence: identity taps without SiLU reproduce the plain run; general taps
    equal an independent numpy convolution of each of q, k, v fed to the core (so q's convolution reaches q,
    k's k, v's v); running in two pieces with the final window carried equals one run."""
    rng = np.random.default_rng(42)
    d, H, T, W = 16, 2, 29, 4
    f = lambda *sh: f32_to_bf16_bits(rng.standard_normal(sh).astype(np.float32))
    q, k, v, g, beta = f(T, H, d), f(T, H, d), f(T, H, d), f(T, H, d), f(T, H)
    A_log = np.log(rng.uniform(1, 4, H)).astype(np.float32)
    dtb = (rng.standard_normal((H, d)) * 0.1).astype(np.float32)
    cu = np.array([0, T], np.int32)
    lb, scale = -2.0, 0.3
    ident = np.zeros((3, H, d, W))
    ident[..., W - 1] = 1.0
    out_id, S_id, _, _, _ = O.run_conv(q, k, v, g, beta, A_log, dtb, lb, scale, cu, ident, False)
    out_pl, S_pl, _ = O.run(q, k, v, g, beta, A_log, dtb, lb, scale, cu)
    _close(out_id, out_pl, 1e-14, "identity taps: outputs of the plain run")
    _close(S_id, S_pl, 1e-14, "identity taps: final state of the plain run")
    w = rng.standard_normal((3, H, d, W)) * 0.6
    win0 = rng.standard_normal((1, 3, W - 1, H, d))
    out, S, _, wf, _ = O.run_conv(q, k, v, g, beta, A_log, dtb, lb, scale, cu, w, True, win0=win0)
    for h in range(H):
        conv = []
        for m, x in enumerate((q, k, v)):
            xs = np.concatenate([win0[0, m, :, h, :], _widen(x[:, h, :])])   # window rows, then the inputs
            z = np.stack([np.convolve(xs[:, c], w[m, h, c, ::-1])[W - 1:W - 1 + T] for c in range(d)], axis=1)
            conv.append(z * expit(z))
        qh = conv[0] / np.sqrt((conv[0] ** 2).sum(axis=1, keepdims=True) + oracle_eps())
        kh = conv[1] / np.sqrt((conv[1] ** 2).sum(axis=1, keepdims=True) + oracle_eps())
        lam = lb * expit(math.exp(A_log[h]) * (_widen(g[:, h, :]) + dtb[h]))
        bt = expit(_widen(beta[:, h]))
        o_ref, S_ref, _ = O.core(qh, kh, conv[2], lam, bt, scale)
        _close(out[:, h], o_ref, 1e-12, f"head {h}: conv'd q/k/v fed to the core")
        _close(S[0, h], S_ref, 1e-12, f"head {h}: final state")
        for m, x in enumerate((q, k, v)):
            _close(wf[0, m, :, h], _widen(x[T - (W - 1):, h, :]), 0.0, f"head {h}: final window of input {m}")
    cut = 11
    o1, S1, _, w1, _ = O.run_conv(q[:cut], k[:cut], v[:cut], g[:cut], beta[:cut], A_log, dtb, lb, scale,
                                  np.array([0, cut], np.int32), w, True, win0=win0)
    o2, S2, _, w2, _ = O.run_conv(q[cut:], k[cut:], v[cut:], g[cut:], beta[cut:], A_log, dtb, lb, scale,
                                  np.array([0, T - cut], np.int32), w, True, win0=w1, S0=S1)
    _close(np.concatenate([o1, o2]), out, 1e-13, "split with the window carried: outputs")
    _close(S2, S, 1e-13, "split with the window carried: final state")
    _close(w2, wf, 0.0, "split with the window carried: final window")


def oracle_eps():
    import oracle
    return oracle.L2NORM_EPS


ALL_PINS = [
    pin_worked_example,
    pin_gate_special_cases,
    pin_l2norm,
    pin_single_token_closed_form,
    pin_product_form,
    pin_zero_beta_is_pure_decay,
    pin_orthonormal_retrieval,
    pin_split_with_carry,
    pin_varlen_packing,
    pin_linearity,
    pin_qk_scale_invariance,
    pin_contraction_bound,
    pin_chunked_equals_sequential,
    pin_gated_rmsnorm,
    pin_short_conv_step,
    pin_short_conv_in_the_path,
]
