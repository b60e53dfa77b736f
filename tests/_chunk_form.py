"""A second, chunkwise formulation of the KDA recurrence, in fp64 numpy.

Used only by the tests: it pins the token-by-token oracle from a different derivation (the
WY/UT chunk algebra) and documents the chunk algebra the tensor-core prefill follows.

Within a chunk of C tokens starting from state S0, with per-channel cumulative
log-retention gam_r = sum_{s<=r} g_s (so Gamma_r = exp(gam_r)):

  A[r, s] = beta_r * sum_i k_ri k_si exp(gam_ri - gam_si)      (s < r)
  P[r, s] = sum_i q_ri k_si exp(gam_ri - gam_si)                (s <= r)
  T       = (I + A)^-1
  u       = T diag(beta) (V - (K * Gamma) S0)                   (the corrected writes)
  O       = (Q * Gamma) S0 + P u
  S_C     = Diag(Gamma_C) S0 + (K * Gamma_C / Gamma)^T u

which equals the token recurrence of the pages exactly in exact arithmetic.
"""
import numpy as np


def l2n(x, eps):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


def chunked_head(q, k, v, g, beta, S0, C, *, g_min=-5.0, l2_eps=1e-6, qk_l2norm=True,
                 scale=1.0):
    """One head, one sequence: q, k [T, dk]; v [T, dv]; g [T, dk]; beta [T]; S0 [dk, dv]."""
    T = q.shape[0]
    if qk_l2norm:
        q = l2n(q, l2_eps)
        k = l2n(k, l2_eps)
    g = np.maximum(g, g_min)
    S = S0.astype(np.float64).copy()
    out = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        sl = slice(c0, min(T, c0 + C))
        qc, kc, vc, gc, bc = q[sl], k[sl], v[sl], g[sl], beta[sl]
        n = qc.shape[0]
        gam = np.cumsum(gc, axis=0)
        diff = gam[:, None, :] - gam[None, :, :]          # [r, s, i] = gam_r - gam_s
        low = np.tril(np.ones((n, n), dtype=bool), -1)
        incl = np.tril(np.ones((n, n), dtype=bool), 0)
        decay = np.exp(np.where(incl[:, :, None], diff, 0.0))
        A = np.where(low, bc[:, None] * np.einsum("ri,si,rsi->rs", kc, kc, decay), 0.0)
        P = np.where(incl, np.einsum("ri,si,rsi->rs", qc, kc, decay), 0.0)
        Tm = np.linalg.inv(np.eye(n) + A)
        G = np.exp(gam)
        u = Tm @ (bc[:, None] * (vc - (kc * G) @ S))
        out[sl] = scale * ((qc * G) @ S + P @ u)
        S = G[-1][:, None] * S + (kc * np.exp(gam[-1] - gam)).T @ u
    return out, S
