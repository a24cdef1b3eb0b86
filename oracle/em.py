"""EM M-step of the sum layers' parameters, float64.

Test infrastructure: only tests/, ``__graft_entry__.smoke()`` and bench.py's oracle legs
use this module; the library never does.

pyjuice LowRank API doc (Training): with the denominator statistic W kept
(apply_z_correction), the M-step is the conditional update

    theta <- normalize(theta * F+ / F-),   F-[i,j] = theta[i,j] * W[i,j],

i.e. normalize(F+ / W) wherever theta > 0; with apply_z_correction off it is the plain
normalize(F+). ``normalize`` divides each node's parameters by their sum over the node's
children (the rows here), as the parameters themselves are normalized (same doc, intro:
"normalized over the children of node i"). For the plain sum layers of the HMM and the
HCLT the M-step is normalize(F) of the parameter flows: with flows that are posterior
expected counts this is the Baum-Welch update of an HMM.

Readings where the pages are silent:
  * a pair with W = 0 (no denominator flow reached it; then F+ = 0 as well) contributes 0
    to the ratio;
  * a node whose ratio sums to 0 (no flow reached the node at all) keeps its parameters.
"""
from __future__ import annotations

import numpy as np


def normalize(R: np.ndarray, theta_prev: np.ndarray) -> np.ndarray:
    """Rows of R (any leading group axes) divided by their sums; rows summing to 0 (or
    to a non-finite value) keep theta_prev's row."""
    R = np.asarray(R, dtype=np.float64)
    prev = np.asarray(theta_prev, dtype=np.float64)
    s = R.sum(axis=-1, keepdims=True)
    ok = np.isfinite(s) & (s > 0)
    with np.errstate(divide="ignore", invalid="ignore"):
        out = R / np.where(ok, s, 1.0)
    return np.where(ok, out, prev)


def em_plain(F: np.ndarray, theta_prev: np.ndarray) -> np.ndarray:
    """theta <- normalize(F)."""
    return normalize(F, theta_prev)


def em_conditional(Fplus: np.ndarray, W: np.ndarray, theta_prev: np.ndarray) -> np.ndarray:
    """theta <- normalize(theta * F+ / (theta * W)) = normalize(F+ / W), 0 where W = 0."""
    Fplus = np.asarray(Fplus, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(W > 0, Fplus / np.where(W > 0, W, 1.0), 0.0)
    return normalize(ratio, theta_prev)


def hmm_em_step(pi, A, E, tokens):
    """One Baum-Welch step of the HMM circuit: the flows dpi, dA, dE of the oracle's
    forward-backward (posterior expected counts) normalized per node."""
    from oracle.hmm import hmm_fwd_bwd

    _, dpi, dA, dE = hmm_fwd_bwd(pi, A, E, tokens)
    return (em_plain(dpi[None, :], np.asarray(pi, np.float64)[None, :])[0], em_plain(dA, A), em_plain(dE, E))
