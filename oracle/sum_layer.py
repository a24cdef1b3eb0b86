"""Dense log-space sum layer: forward and EM flows, float64.

pyjuice PR #62, Summary 2: a dense layer exponentiates its children, multiplies
by the parameters and takes the log. With m_b the per-sample maximum over the
group's children (the per-group column maximum the Tests section checks):

    out[i,b] = m_b + log sum_j theta[i,j] * exp(x[j,b] - m_b)

pyjuice PR #62, Summary 3 names the two backward contractions (element flows and
parameter flows). For node flows f[i,b]:

    e[j,b] = sum_i theta[i,j] * f[i,b] * exp(x[j,b] - out[i,b])
    F[i,j] = theta[i,j] * sum_b f[i,b] * exp(x[j,b] - out[i,b])

Layout: theta [G,M,N]; x [R,B] rows of child log-values; group g's children are
rows g*child_stride .. g*child_stride+N-1 of x (child_stride = 0 with G = 1 is the
shared-children layout, child_stride >= N the evenly strided groups of Summary 2,
second bullet). out and f are [G,M,B]; e is shaped like x; F like theta.

Readings where the pages are silent:
* a column whose children are all -inf has m_b = -inf and out = -inf, with zero flows;
* a zero sum gives out = -inf; a node with out = -inf passes no flow.
"""
from __future__ import annotations

import numpy as np


def _group_rows(g: int, child_stride: int, N: int) -> slice:
    return slice(g * child_stride, g * child_stride + N)


def column_max(xs: np.ndarray) -> np.ndarray:
    """m_b = max_j x[j,b]; -inf for an all -inf column (or no children)."""
    if xs.shape[0] == 0:
        return np.full(xs.shape[1], -np.inf)
    return xs.max(axis=0)


def _shifted_exp(xs: np.ndarray, m: np.ndarray) -> np.ndarray:
    """exp(x - m_b), with exp(-inf - (-inf)) read as 0."""
    mf = np.where(np.isfinite(m), m, 0.0)
    with np.errstate(invalid="ignore", over="ignore"):
        u = np.exp(xs - mf[None, :])
    u[:, ~np.isfinite(m)] = 0.0
    return u


def _safe_log(a: np.ndarray) -> np.ndarray:
    with np.errstate(divide="ignore"):
        return np.log(a)


def sum_layer_fwd(theta, x, child_stride: int = 0) -> np.ndarray:
    """out[g,i,b] = m_{g,b} + log sum_j theta[g,i,j] exp(x[g*cs+j,b] - m_{g,b})."""
    theta = np.asarray(theta, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    G, M, N = theta.shape
    B = x.shape[1]
    out = np.empty((G, M, B))
    for g in range(G):
        xs = x[_group_rows(g, child_stride, N)]
        m = column_max(xs)
        u = _shifted_exp(xs, m)
        acc = theta[g] @ u
        mf = np.where(np.isfinite(m), m, 0.0)
        o = mf[None, :] + _safe_log(acc)
        o[:, ~np.isfinite(m)] = -np.inf
        out[g] = o
    return out


def sum_layer_bwd(theta, x, child_stride: int, out, f):
    """Element flows e (shaped like x; rows outside every group are 0) and
    parameter flows F [G,M,N].

    Computed through the exact factorisation
        exp(x[j,b] - out[i,b]) = exp(x[j,b] - m_b) * exp(m_b - out[i,b]),
    which turns both contractions into matrix products. ``sum_layer_bwd_literal``
    is the unfactored triple loop it is tested against.
    """
    theta = np.asarray(theta, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    out = np.asarray(out, dtype=np.float64)
    f = np.asarray(f, dtype=np.float64)
    G, M, N = theta.shape
    e = np.zeros_like(x)
    F = np.zeros_like(theta)
    for g in range(G):
        rows = _group_rows(g, child_stride, N)
        xs = x[rows]
        m = column_max(xs)
        u = _shifted_exp(xs, m)                       # exp(x - m_b)
        mf = np.where(np.isfinite(m), m, 0.0)
        with np.errstate(over="ignore", invalid="ignore"):
            r = np.exp(mf[None, :] - out[g])           # exp(m_b - out)
        w = np.where(np.isfinite(out[g]), f[g] * r, 0.0)
        e[rows] += u * (theta[g].T @ w)
        F[g] = theta[g] * (w @ u.T)
    return e, F


def sum_layer_bwd_literal(theta, x, child_stride: int, out, f):
    """Literal loops over (g, i, j, b) of the two flow definitions; tiny shapes only."""
    theta = np.asarray(theta, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    G, M, N = theta.shape
    B = x.shape[1]
    e = np.zeros_like(x)
    F = np.zeros_like(theta)
    for g in range(G):
        for i in range(M):
            for j in range(N):
                r = g * child_stride + j
                acc = 0.0
                for b in range(B):
                    if not np.isfinite(out[g, i, b]):
                        continue
                    t = f[g, i, b] * np.exp(x[r, b] - out[g, i, b])
                    e[r, b] += theta[g, i, j] * t
                    acc += t
                F[g, i, j] = theta[g, i, j] * acc
    return e, F
