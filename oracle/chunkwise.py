"""Chunked reformulation of the gated delta rule, numpy fp64.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  This is *a check of* the
token-loop oracle and the source of per-stage intermediates for kernel-level
parity; it is not the oracle itself.  It is written straight from the algebra
below with library primitives (matmul, triangular solve) and no blocking,
fusion or reordering beyond it.

Why a chunked form exists at all: the pages explain that chunk/tile-parallel
linear attention splits the work into an intra-tile causal part and an
inter-tile recurrent state, and that the intra-tile part needs the reciprocal
of the cumulative decay Gamma ("What a Trillion-Parameter MoE Model Reveals
About the Next Stage of LLM Scaling", section 3.1; "Architecture Evolution and
Training Engineering for Trillion-Scale Sparse Multimodal Models", sections
3.1-3.2, where Gamma = exp(cumsum(log-decay)) and every causal tile is one
dense GEMM scaled by inv_gamma).  With the lower-bounded decay the reciprocal
1/gamma_r <= a_min^{-C} stays finite, so the diagonal tile is computed with the
same dense products as the others.

Notation for one chunk of C rows r = 1..C (rows of Q, K [C, dk] and V [C, dv]):

    lambda_r = log alpha_r,  b_r = sum_{s<=r} lambda_s,  gamma_r = exp(b_r),
    gamma_C  = gamma of the last row,
    K_hat = diag(1/gamma) K,   Q_hat = diag(gamma) Q,   K_til = diag(gamma_C/gamma) K,
    A     = strict_lower( diag(beta*gamma) K K_hat^T )
    T     = (I + A)^{-1}
    U     = T diag(beta) V,         Wk = T diag(beta*gamma) K
    W     = U - Wk M_n                                   (M_n = S^T at chunk start)
    O     = Q_hat M_n + lower_incl(Q_hat K_hat^T) W
    M_{n+1} = gamma_C M_n + K_til^T W

Derivation (exact, no approximation): with w_r = v_r - alpha_r M_{r-1}^T k_r the
token step is M_r = alpha_r M_{r-1} + beta_r k_r w_r^T.  Unrolling inside the
chunk gives M_r = gamma_r M_n + sum_{s<=r} (gamma_r/gamma_s) beta_s k_s w_s^T;
substituting into w_r and scaling row r by beta_r gives (I + A) W = diag(beta) V
- diag(beta*gamma) K M_n with W_r = beta_r w_r, i.e. W = U - Wk M_n; o_r =
M_r^T q_r then gives O, and r = C gives M_{n+1}.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def alpha(g, a_min):
    """Lower-bounded decay alpha = a_min + (1 - a_min) sigmoid(g) (fp64)."""
    g = np.asarray(g, np.float64)
    return a_min + (1.0 - a_min) / (1.0 + np.exp(-g))


def log_alpha(g, bound, decay="affine"):
    """log alpha per token: the log of the linear-domain form above, or the pages'
    log-domain form log alpha = g_min sigmoid(g) (decay "log", bound = g_min)."""
    g = np.asarray(g, np.float64)
    if decay == "log":
        return bound / (1.0 + np.exp(-g))
    return np.log(alpha(g, bound))


def chunk_decay(g, a_min, C, decay="affine"):
    """Chunk-local cumulative log-decay for one head: returns (b, gamma, inv_gamma)
    over all T rows, each restarting at every chunk boundary (row 0 of a chunk
    has b = log alpha of that row)."""
    lam = log_alpha(g, a_min, decay)
    T = lam.shape[0]
    b = np.empty(T, np.float64)
    for n0 in range(0, T, C):
        b[n0:n0 + C] = np.cumsum(lam[n0:n0 + C])
    gam = np.exp(b)
    return b, gam, 1.0 / gam


def head(q, k, v, g, beta, a_min, M0=None, C=64, keep=False, decay="affine"):
    """Chunked forward for one head.  q,k [T,dk], v [T,dv], g,beta [T], M0 [dk,dv]
    or None.  Returns (out [T,dv], M_final [dk,dv], intermediates or None).

    With ``keep`` the per-chunk intermediates are returned as a dict of lists:
    gamma, A, T, U, Wk, W, M (state at each chunk start), P (the masked decayed
    scores).  The last chunk may be shorter than C (ragged tail): it is the same
    algebra on fewer rows.
    """
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    g, beta = np.asarray(g, np.float64), np.asarray(beta, np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    M = np.zeros((dk, dv)) if M0 is None else np.array(M0, np.float64)
    _, gam_all, _ = chunk_decay(g, a_min, C, decay)
    out = np.empty((T, dv))
    inter = {n: [] for n in ("gamma", "A", "T", "U", "Wk", "W", "M", "P")} if keep else None
    for n0 in range(0, T, C):
        sl = slice(n0, min(n0 + C, T))
        K, Q, V, bt, gam = k[sl], q[sl], v[sl], beta[sl], gam_all[sl]
        c = K.shape[0]
        gC = gam[-1]
        K_hat = K / gam[:, None]
        Q_hat = Q * gam[:, None]
        K_til = K * (gC / gam)[:, None]
        A = np.tril((bt * gam)[:, None] * (K @ K_hat.T), -1)
        Tm = solve_triangular(np.eye(c) + A, np.eye(c), lower=True, unit_diagonal=True)
        U = Tm @ (bt[:, None] * V)
        Wk = Tm @ ((bt * gam)[:, None] * K)
        W = U - Wk @ M
        P = np.tril(Q_hat @ K_hat.T)
        out[sl] = Q_hat @ M + P @ W
        if keep:
            for name, val in (("gamma", gam), ("A", A), ("T", Tm), ("U", U),
                              ("Wk", Wk), ("W", W), ("M", M.copy()), ("P", P)):
                inter[name].append(val)
        M = gC * M + K_til.T @ W
    return out, M, inter


def fwd(q, k, v, g, beta, a_min, init_state=None, C=64, decay="affine"):
    """Chunked forward over [B,H,T,...] arrays (fp64 results)."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    out = np.empty((B, H, T, dv))
    fin = np.empty((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            M0 = None if init_state is None else np.asarray(init_state[b, h], np.float64)
            out[b, h], fin[b, h], _ = head(q[b, h], k[b, h], v[b, h], g[b, h], beta[b, h],
                                           a_min, M0, C, decay=decay)
    return out, fin
