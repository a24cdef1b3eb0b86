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


# ----------------------------------------------------------------- "sum_exp" form
# pyjuice LowRank API doc (intro formulas): the second form of the scale,
#     g_b[i,j] = sum_r exp(A_b[i,r]) exp(B_b[r,j])          ("sum_exp": a mixture of
# k rank-one scales), with Z_b and theta_b as above. The layer, its flows and the
# Z-correction statistic are the same functions of theta_b and g_b as for "exp_sum";
# only the chain rule into the factors differs: with D = f (p - q) as above,
#     d(sum f out)/d g_b[i,j] = D[i,j] / g_b[i,j]
#     dA_b[i,r] = exp(A_b[i,r]) sum_j (D / g)[i,j] exp(B_b[r,j])
#     dB_b[r,j] = exp(B_b[r,j]) sum_i exp(A_b[i,r]) (D / g)[i,j].
# Each row of A_b is shifted by its maximum and each row of B_b by its maximum before the
# exponentials (the shift of a row of A scales g's row and cancels in theta_b; the shift
# of a row r of B is folded into column r of A), so float64 holds every term.


def _per_sample_sum_exp(theta, A, Bm, x, b):
    beta = Bm[b].max(axis=1)                                 # [K]
    c = np.exp(Bm[b] - beta[:, None])                        # exp(B) / exp(beta_r)
    Ab = A[b] + beta[None, :]
    alpha = Ab.max(axis=1)                                   # [M]
    a = np.exp(Ab - alpha[:, None])                          # exp(A) exp(beta) / exp(alpha_i)
    g = a @ c                                                # g_b / exp(alpha_i)
    tg = theta * g
    Z = tg.sum(axis=1)
    m = x[:, b].max()
    u = np.exp(x[:, b] - m)
    num = tg @ u
    with np.errstate(divide="ignore"):
        out = m + np.log(num) - np.log(Z)
        logZ = np.log(Z) + alpha
    return a, c, g, Z, u, out, logZ


def lowrank_sum_exp_fwd(theta, A, Bm, x):
    """Returns out [M,B] and logZ [B,M] of the "sum_exp" form."""
    theta, A, Bm, x = (np.asarray(v, dtype=np.float64) for v in (theta, A, Bm, x))
    M, N = theta.shape
    B = x.shape[1]
    out = np.empty((M, B))
    logZ = np.empty((B, M))
    for b in range(B):
        _, _, _, _, _, o, lz = _per_sample_sum_exp(theta, A, Bm, x, b)
        out[:, b] = o
        logZ[b] = lz
    return out, logZ


def lowrank_sum_exp_bwd(theta, A, Bm, x, f):
    """Returns dA [B,M,K], dB [B,K,N], e [N,B], Fplus [M,N], W [M,N], out, logZ of the
    "sum_exp" form, and absdA, absdB: the sums of the absolute terms behind each gradient
    entry before cancellation (as for "exp_sum")."""
    theta, A, Bm, x, f = (np.asarray(v, dtype=np.float64) for v in (theta, A, Bm, x, f))
    M, N = theta.shape
    B = x.shape[1]
    K = A.shape[2]
    dA = np.empty((B, M, K))
    dB = np.empty((B, K, N))
    absdA = np.empty((B, M, K))
    absdB = np.empty((B, K, N))
    e = np.empty((N, B))
    Fplus = np.zeros((M, N))
    Wst = np.zeros((M, N))
    out = np.empty((M, B))
    logZ = np.empty((B, M))
    for b in range(B):
        a, c, g, Z, u, o, lz = _per_sample_sum_exp(theta, A, Bm, x, b)
        out[:, b] = o
        logZ[b] = lz
        q = theta * g / Z[:, None]
        p = q * np.exp(x[:, b][None, :] - o[:, None])
        fb = f[:, b][:, None]
        D = fb * (p - q)
        with np.errstate(divide="ignore", invalid="ignore"):
            R = np.where(g > 0, D / np.where(g > 0, g, 1.0), 0.0)        # d/dg (up to exp(alpha_i))
            Rabs = np.where(g > 0, np.abs(fb) * (p + q) / np.where(g > 0, g, 1.0), 0.0)
        # the exp(alpha_i) of g's row cancels against the same factor of a_ir c_rj
        dA[b] = a * (R @ c.T)
        dB[b] = c * (a.T @ R)
        absdA[b] = a * (Rabs @ c.T)
        absdB[b] = c * (a.T @ Rabs)
        e[:, b] = (fb * p).sum(axis=0)
        Fplus += fb * p
        Wst += fb * g / Z[:, None]
    return dict(dA=dA, dB=dB, e=e, Fplus=Fplus, W=Wst, out=out, logZ=logZ, absdA=absdA, absdB=absdB)
