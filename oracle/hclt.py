"""HCLT circuit as a tree of per-edge sum layers, float64.

pyjuice PR #62 times a whole HCLT circuit (Results table: 1024 latents, 768
variables, 512 categories) and runs its layers as batched GEMMs over evenly
strided child groups (Summary 2, second bullet). The pages do not define the
circuit; the plain reading used here is a latent tree over the variables:

    n_v(z) = E_v[z, x_v] * prod_{c : parent[c] = v} s_c(z)      (product layer)
    s_c(z) = sum_{z'} W_c[z, z'] n_c(z')                         (sum layer per edge)
    LL     = log sum_z pi[z] n_0(z)                              (root sum layer)

with variable 0 the root, parent[i] in [0, i) for i > 0, one H x H sum layer per
tree edge (W is not tied across edges). In log space every sum layer is
``sum_layer_fwd`` / ``sum_layer_bwd``. Flows as for the HMM: root flow 1 per
sample, product nodes pass their flow unchanged to every child, so
dW_c = parameter flows of edge c, dE_v[z, k] = sum of the flows reaching n_v(z)
over the samples with x_v = k, dpi = the root's parameter flows.

Processing nodes in decreasing index order visits every child before its parent,
because parent[i] < i.
"""
from __future__ import annotations

import numpy as np

from .sum_layer import sum_layer_fwd, sum_layer_bwd


def _log(a):
    with np.errstate(divide="ignore"):
        return np.log(a)


def children_lists(parent):
    n = len(parent)
    ch = [[] for _ in range(n)]
    for c in range(1, n):
        ch[int(parent[c])].append(c)
    return ch


def hclt_forward(parent, data, pi, W, E):
    """Returns ll [B], y (log n_v [H,B] per node), s (log s_c [H,B] per edge child c)."""
    parent = np.asarray(parent)
    data = np.asarray(data)
    pi = np.asarray(pi, dtype=np.float64)
    n = len(parent)
    B = data.shape[0]
    ch = children_lists(parent)
    y = [None] * n
    s = [None] * n
    for v in range(n - 1, -1, -1):
        acc = _log(np.asarray(E[v], dtype=np.float64))[:, data[:, v]]
        for c in ch[v]:
            acc = acc + s[c]
        y[v] = acc
        if v > 0:
            s[v] = sum_layer_fwd(np.asarray(W[v], dtype=np.float64)[None], y[v])[0]
    ll = sum_layer_fwd(pi[None, None, :], y[0])[0, 0]
    return ll, y, s


def hclt_fwd_bwd(parent, data, pi, W, E):
    """Returns ll [B], dpi [H], dW [n,H,H] (dW[0] = 0), dE [n,H,C]."""
    parent = np.asarray(parent)
    data = np.asarray(data)
    pi = np.asarray(pi, dtype=np.float64)
    n = len(parent)
    B = data.shape[0]
    H = pi.shape[0]
    C = np.asarray(E[0]).shape[1]
    ll, y, s = hclt_forward(parent, data, pi, W, E)
    e0, Fpi = sum_layer_bwd(pi[None, None, :], y[0], 0, ll[None, None, :], np.ones((1, 1, B)))
    dpi = Fpi[0, 0]
    flow = [None] * n
    flow[0] = e0
    dW = np.zeros((n, H, H))
    dE = np.zeros((n, H, C))
    for c in range(1, n):            # parent[c] < c: the parent's flow is final
        v = int(parent[c])
        e, F = sum_layer_bwd(np.asarray(W[c], dtype=np.float64)[None], y[c], 0, s[c][None],
                             flow[v][None])
        dW[c] = F[0]
        flow[c] = e
    for v in range(n):
        for b in range(B):
            dE[v][:, data[b, v]] += flow[v][:, b]
    return ll, dpi, dW, dE


def hclt_ll(parent, data, pi, W, E):
    return hclt_forward(parent, data, pi, W, E)[0]
