"""fp64 NumPy statement of the chunked (chunk-parallel) form of the recurrence.

Test helper only.  It restates, for one (sequence, head), the chunk algebra
that the CUDA prefill kernel evaluates, so the tests can pin it against the
token-by-token oracle on small inputs:

Within a chunk of rows r = 0..C-1 starting from state S (dk x dv), with
b_r = sum_{j<=r} lambda_j (per key channel) and Gamma_r = exp(b_r):

  A[r,i] = beta_r * sum_c k_rc k_ic exp(b_rc - b_ic)            (i < r)
  P[r,i] =          sum_c q_rc k_ic exp(b_rc - b_ic)            (i <= r)
  T      = (I + A)^-1 Diag(beta)
  W = T (K o Gamma),  U^ = T V,  U = U^ - W S
  O = scale * ((Q o Gamma) S + P U)
  S' = Diag(Gamma_last) S + (K o exp(b_last - b))^T U

(derivation: unroll S_r = Diag(alpha_r) S_{r-1} + k_r u_r^T over the chunk;
the corrections u_r then satisfy (I + A) U = Diag(beta)(V - (K o Gamma) S)).

``chunked_anchored`` evaluates A and P the way the kernel does, through
16-row sub-blocks whose exponentials never leave the fp32 range.
"""
from __future__ import annotations

import numpy as np

SUB = 16


def _chunks(T, C):
    for c0 in range(0, T, C):
        yield c0, min(c0 + C, T)


def chunked_exact(qh, kh, v, lam, beta, scale, S0, C):
    """Chunked evaluation with exact exp(b_r - b_i) ratios (fp64)."""
    T, dk = qh.shape
    dv = v.shape[1]
    S = np.array(S0, dtype=np.float64, copy=True)
    out = np.zeros((T, dv))
    for c0, c1 in _chunks(T, C):
        n = c1 - c0
        Q, K, V, L, bt = qh[c0:c1], kh[c0:c1], v[c0:c1], lam[c0:c1], beta[c0:c1]
        b = np.cumsum(L, axis=0)
        r = np.arange(n)
        lower = r[:, None] >= r[None, :]
        strict = r[:, None] > r[None, :]
        diff = np.where(lower[:, :, None], b[:, None, :] - b[None, :, :], -np.inf)
        ratio = np.exp(diff)
        A = bt[:, None] * np.einsum("rc,ic,ric->ri", K, K, ratio) * strict
        P = np.einsum("rc,ic,ric->ri", Q, K, ratio) * lower
        Tm = np.linalg.solve(np.eye(n) + A, np.diag(bt))
        gam = np.exp(b)
        W = Tm @ (K * gam)
        U = Tm @ V - W @ S
        out[c0:c1] = scale * ((Q * gam) @ S + P @ U)
        S = np.exp(b[-1])[:, None] * S + (K * np.exp(b[-1] - b)).T @ U
    return out, S


def anchored_factors(b, sub=SUB):
    """Sub-block factorisation of exp(b_r - b_i) for one chunk of C = sub*nb rows.

    Rows are grouped in blocks R of `sub` rows (16, or 32 for the kernel's
    lower_bound >= -5 variant).  With m_R = b at the block's middle row
    (sub/2 - 1) and a_R = b at its last row:
      same block:       exp(b_r - b_i) = E_r * Einv_i,  E = exp(b - m_R(r)),  Einv = exp(m_R - b)
      block I < R:      exp(b_r - b_i) = (E_r * c[R,I]) * Gp_i,
                        c[R,I] = exp(m_R - a_I) <= 1,  Gp_i = exp(a_I - b_i) <= 1
    Returns the factors and the largest exponent magnitude that had to be
    represented (must stay below ~87 for fp32).
    """
    n, dk = b.shape
    assert n % sub == 0
    nb = n // sub
    m = b[sub // 2 - 1::sub]          # [nb, dk]  middle row of each block
    a = b[sub - 1::sub]               # [nb, dk]  last row of each block
    blk = np.arange(n) // sub
    e_exp = b - m[blk]
    einv_exp = m[blk] - b
    gp_exp = a[blk] - b
    c_exp = m[:, None, :] - a[None, :, :]  # [R, I, dk]
    worst = max(np.abs(e_exp).max(), np.abs(einv_exp).max())
    E, Einv, Gp = np.exp(e_exp), np.exp(einv_exp), np.exp(gp_exp)
    Rr, Ii = np.meshgrid(np.arange(nb), np.arange(nb), indexing="ij")
    c = np.where((Rr > Ii)[:, :, None], np.exp(np.minimum(c_exp, 0.0)), 0.0)
    assert (gp_exp <= 1e-12).all()
    return dict(E=E, Einv=Einv, Gp=Gp, c=c, m=m, a=a, worst_exponent=worst)


def chunked_anchored(qh, kh, v, lam, beta, scale, S0, C=64, sub=SUB):
    """Chunked evaluation with A, P built from the anchored sub-block factors.

    Each chunk is padded to C rows with q = k = v = 0, lambda = 0, beta = 0
    (padding rows change neither the state nor the decay).
    """
    assert C % sub == 0
    T, dk = qh.shape
    dv = v.shape[1]
    S = np.array(S0, dtype=np.float64, copy=True)
    out = np.zeros((T, dv))
    worst = 0.0
    for c0, c1 in _chunks(T, C):
        n = c1 - c0
        pad = C - n
        Q = np.pad(qh[c0:c1], ((0, pad), (0, 0)))
        K = np.pad(kh[c0:c1], ((0, pad), (0, 0)))
        V = np.pad(v[c0:c1], ((0, pad), (0, 0)))
        L = np.pad(lam[c0:c1], ((0, pad), (0, 0)))
        bt = np.pad(beta[c0:c1], (0, pad))
        b = np.cumsum(L, axis=0)
        f = anchored_factors(b, sub)
        worst = max(worst, f["worst_exponent"])
        FK, FQ = K * f["E"], Q * f["E"]
        G, Gp = K * f["Einv"], K * f["Gp"]
        A = np.zeros((C, C))
        P = np.zeros((C, C))
        nb = C // sub
        for R in range(nb):
            rs = slice(R * sub, (R + 1) * sub)
            for I in range(R + 1):
                cs = slice(I * sub, (I + 1) * sub)
                if I == R:
                    A[rs, cs] = FK[rs] @ G[cs].T
                    P[rs, cs] = FQ[rs] @ G[cs].T
                else:
                    cRI = f["c"][R, I]
                    A[rs, cs] = (FK[rs] * cRI) @ Gp[cs].T
                    P[rs, cs] = (FQ[rs] * cRI) @ Gp[cs].T
        r = np.arange(C)
        A = bt[:, None] * A * (r[:, None] > r[None, :])
        P = P * (r[:, None] >= r[None, :])
        Tm = np.linalg.solve(np.eye(C) + A, np.diag(bt))
        blk = r // sub
        em = np.exp(f["m"])[blk]                 # exp(m_R(r))
        Kplus = FK * em                           # k o exp(b)
        Qplus = FQ * em
        Kprime = G * np.exp(b[-1] - f["m"])[blk]  # k o exp(b_last - b)
        W = Tm @ Kplus
        U = Tm @ V - W @ S
        o = scale * (Qplus @ S + P @ U)
        out[c0:c1] = o[:n]
        S = np.exp(b[-1])[:, None] * S + Kprime.T @ U
    return out, S, worst
