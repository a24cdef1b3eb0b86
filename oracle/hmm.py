"""HMM circuit as a chain of shared-children sum layers, float64.

pyjuice PR #62 times whole HMM circuits (Results table: 4096 latents x 32
positions; 1024 x 64) and says their sum layers share their children, so the
children are exponentiated once for all blocks (Summary 2, first bullet). The
pages do not spell out the circuit; the plain reading used here is the standard
HMM  P(x_1..x_T) = sum_z pi(z_1) prod_t E(z_t, x_t) prod_t A(z_t, z_{t+1}),
built as a probabilistic circuit from the last position back:

    P_T(k) = E[k, x_T]                                  (input layer)
    S_t(k) = sum_l A[k,l] P_{t+1}(l)                    (sum layer, M = N = H,
                                                         shared children, tied over t)
    P_t(k) = E[k, x_t] * S_t(k)                         (product layer)
    LL     = log sum_k pi[k] P_1(k)                     (root sum layer)

Everything is held in log space and every sum layer is ``sum_layer_fwd`` /
``sum_layer_bwd``. The root flow is 1 per sample; a product node passes its flow
unchanged to its children, so the flows are the posterior expected counts:

    dpi[k]   = flow of the root's parameter pi[k]
    dA[k,l]  = sum over the T-1 tied layers of their parameter flows
    dE[k,v]  = sum over (t, b) with x_{t,b} = v of the flow reaching P_t(k)

Emission and initial flows are not listed on the pages; they are what an EM
step needs and are included for that reason.
"""
from __future__ import annotations

import numpy as np

from .sum_layer import sum_layer_fwd, sum_layer_bwd


def _log(a):
    with np.errstate(divide="ignore"):
        return np.log(a)


def hmm_forward_chain(pi, A, E, tokens):
    """Log-values of every node: returns (ll [B], xs list of log P_t [H,B], ss list
    of log S_t [H,B] for t = 0..T-2 (zero-based))."""
    pi = np.asarray(pi, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    E = np.asarray(E, dtype=np.float64)
    tokens = np.asarray(tokens)
    B, T = tokens.shape
    logE = _log(E)
    xs = [None] * T
    ss = [None] * (T - 1)
    xs[T - 1] = logE[:, tokens[:, T - 1]]
    for t in range(T - 2, -1, -1):
        ss[t] = sum_layer_fwd(A[None], xs[t + 1])[0]
        xs[t] = logE[:, tokens[:, t]] + ss[t]
    ll = sum_layer_fwd(pi[None, None, :], xs[0])[0, 0]
    return ll, xs, ss


def hmm_fwd_bwd(pi, A, E, tokens):
    """Returns ll [B], dpi [H], dA [H,H], dE [H,V] (flows summed over the batch)."""
    pi = np.asarray(pi, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    E = np.asarray(E, dtype=np.float64)
    tokens = np.asarray(tokens)
    B, T = tokens.shape
    H, V = E.shape
    ll, xs, ss = hmm_forward_chain(pi, A, E, tokens)

    # root sum layer: theta = pi as one node over the H children P_1
    e0, Fpi = sum_layer_bwd(pi[None, None, :], xs[0], 0, ll[None, None, :], np.ones((1, 1, B)))
    dpi = Fpi[0, 0]
    flows = [None] * T
    flows[0] = e0
    dA = np.zeros((H, H))
    for t in range(T - 1):
        # the product node P_t passes its flow to its sum-node child S_t
        e, F = sum_layer_bwd(A[None], xs[t + 1], 0, ss[t][None], flows[t][None])
        dA += F[0]
        flows[t + 1] = e
    dE = np.zeros((H, V))
    for t in range(T):
        for b in range(B):
            dE[:, tokens[b, t]] += flows[t][:, b]
    return ll, dpi, dA, dE


def hmm_ll(pi, A, E, tokens):
    return hmm_forward_chain(pi, A, E, tokens)[0]
