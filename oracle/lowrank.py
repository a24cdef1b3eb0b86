"""LowRank ``exp_sum`` per-sample scale on a dense sum layer, float64.

pyjuice LowRank API doc (intro formulas): per sample b, with A_b [M,k] and
B_b [k,N], the scale and the effective parameters are

    g_b[i,j]     = exp( sum_r A_b[i,r] B_b[r,j] )                 ("exp_sum" form)
    Z_b[i]       = sum_j theta[i,j] g_b[i,j]
    theta_b[i,j] = theta[i,j] g_b[i,j] / Z_b[i]

and the layer is the dense sum layer with theta_b in place of theta:
    out[i,b] = log sum_j theta_b[i,j] exp(x[j,b]).

Tensor layout (same doc, Tensor layout): A [B,M,k], B [B,k,N] float32.

Backward (same doc, Training) for node flows f [M,B]; with
p_ij = theta_b[i,j] exp(x_j - out_i) and q_ij = theta_b[i,j]:
    D_b      = f_i (p - q)              d(sum f out)/d(A_b B_b)
    dA_b     = D_b B_b^T,   dB_b = A_b^T D_b
    e[j,b]   = sum_i f_i p_ij           element flows
    F+[i,j]  = sum_b f_i p_ij           parameter flows
    W[i,j]   = sum_b f_b[i] g_b[i,j] / Z_b[i]   the parameter-free Z-correction
                                         statistic; F-[i,j] = theta[i,j] W[i,j]

Per the doc's Note, the plain fallback materialises the per-sample [M,N] scale
in chunks of samples; this oracle does one sample at a time. The shift by the
row maximum of A_b B_b and by the column maximum of x cancels exactly and only
keeps the float64 exponentials in range.
"""
from __future__ import annotations

import numpy as np


def _per_sample(theta, A, Bm, x, b):
    S = A[b] @ Bm[b]                          # [M,N] log-scale
    s = S.max(axis=1, keepdims=True)
    g = np.exp(S - s)                         # g_b / exp(s_i)
    tg = theta * g
    Z = tg.sum(axis=1)                        # Z_b / exp(s_i)
    m = x[:, b].max()
    u = np.exp(x[:, b] - m)
    num = tg @ u
    with np.errstate(divide="ignore"):
        out = m + np.log(num) - np.log(Z)
        logZ = np.log(Z) + s[:, 0]
    return S, g, Z, u, m, out, logZ


def lowrank_exp_sum_fwd(theta, A, Bm, x):
    """Returns out [M,B] and logZ [B,M] (log Z_b[i], what a backward pass reuses)."""
    theta = np.asarray(theta, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    Bm = np.asarray(Bm, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    M, N = theta.shape
    B = x.shape[1]
    out = np.empty((M, B))
    logZ = np.empty((B, M))
    for b in range(B):
        _, _, _, _, _, o, lz = _per_sample(theta, A, Bm, x, b)
        out[:, b] = o
        logZ[b] = lz
    return out, logZ


def lowrank_exp_sum_bwd(theta, A, Bm, x, f):
    """Returns dA [B,M,K], dB [B,K,N], e [N,B], Fplus [M,N], W [M,N] (and out, logZ),
    plus absdA = |f| (p + q) |B_b|^T and absdB = |A_b|^T |f| (p + q): the sums of the
    absolute terms behind each gradient entry before any cancellation (D = f (p - q)
    cancels within each entry and D's rows sum to zero), the scale against which the
    error of a rounded evaluation is measured."""
    theta = np.asarray(theta, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    Bm = np.asarray(Bm, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    f = np.asarray(f, dtype=np.float64)
    M, N = theta.shape
    B = x.shape[1]
    K = A.shape[2]
    dA = np.empty((B, M, K))
    dB = np.empty((B, K, N))
    e = np.empty((N, B))
    Fplus = np.zeros((M, N))
    Wst = np.zeros((M, N))
    absdA = np.empty((B, M, K))
    absdB = np.empty((B, K, N))
    out = np.empty((M, B))
    logZ = np.empty((B, M))
    for b in range(B):
        S, g, Z, u, m, o, lz = _per_sample(theta, A, Bm, x, b)
        out[:, b] = o
        logZ[b] = lz
        q = theta * g / Z[:, None]                         # theta_b
        p = q * np.exp(x[:, b][None, :] - o[:, None])      # theta_b exp(x_j - out_i)
        fb = f[:, b][:, None]
        D = fb * (p - q)
        dA[b] = D @ Bm[b].T
        dB[b] = A[b].T @ D
        Dmag = np.abs(fb) * (p + q)
        absdA[b] = Dmag @ np.abs(Bm[b]).T
        absdB[b] = np.abs(A[b]).T @ Dmag
        e[:, b] = (fb * p).sum(axis=0)
        Fplus += fb * p
        Wst += fb * g / Z[:, None]
    return dict(dA=dA, dB=dB, e=e, Fplus=Fplus, W=Wst, out=out, logZ=logZ, absdA=absdA, absdB=absdB)
