"""HMM circuit whose transition layers carry the LowRank "exp_sum" scale, float64.

Test infrastructure: only tests/, ``__graft_entry__.smoke()`` and bench.py's oracle legs
use this module; the library never does.

The HMM circuit is the one of oracle/hmm.py (built from the last position back; the
transition sum layers S_t = A P_{t+1} are tied copies of one node vector). pyjuice LowRank
API doc (intro formulas, Tensor layout; Parameters: tie_external off by default, "one
[pair of tensors] per copy") puts the per-sample scale on every copy: the layer of
position t (t = 0 .. T-2) uses its own factors FA[t] [B,H,K], FB[t] [B,K,H],

    A_b^(t)[k,l] = A[k,l] exp((FA[t][b] FB[t][b])[k,l]) / Z_b^(t)[k],

so S_t(k) = sum_l A_b^(t)[k,l] P_{t+1}(l) per sample. The flows of the tied parameters A
are the sums over the copies of the layers' F+ and W (same doc, Training); the factor
gradients are per copy. Every layer is ``lowrank_exp_sum_fwd`` / ``_bwd``.
"""
from __future__ import annotations

import numpy as np

from .lowrank import lowrank_exp_sum_bwd, lowrank_exp_sum_fwd


def _log(a):
    with np.errstate(divide="ignore"):
        return np.log(a)


def hmm_lowrank_forward(pi, A, E, tokens, FA, FB):
    """Returns ll [B], logP [T][H,B] (log P_t) and the layers' logZ [T-1][B,H]."""
    pi, A, E = (np.asarray(v, dtype=np.float64) for v in (pi, A, E))
    tokens = np.asarray(tokens)
    B, T = tokens.shape
    H = A.shape[0]
    logE = _log(E)
    logP = [None] * T
    logZ = [None] * (T - 1)
    logP[T - 1] = logE[:, tokens[:, T - 1]]
    for t in range(T - 2, -1, -1):
        out, lz = lowrank_exp_sum_fwd(A, FA[t], FB[t], logP[t + 1])
        logZ[t] = lz
        logP[t] = out + logE[:, tokens[:, t]]
    z = _log(pi)[:, None] + logP[0]
    m = z.max(axis=0)
    with np.errstate(invalid="ignore"):
        ll = m + np.log(np.exp(z - m).sum(axis=0))
    return ll, logP, logZ


def hmm_lowrank_fwd_bwd(pi, A, E, tokens, FA, FB):
    """Returns dict(ll, dpi, dA = sum_t F+_t, W = sum_t W_t, dE, dFA [T-1,B,H,K],
    dFB [T-1,B,K,H], absdFA, absdFB): the root flow is 1 per sample, so the factor
    gradients are those of sum_b LL_b; absdF* are the layers' sums of absolute terms
    before cancellation (lowrank_exp_sum_bwd's absdA, absdB)."""
    pi = np.asarray(pi, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    tokens = np.asarray(tokens)
    B, T = tokens.shape
    H, V = np.asarray(E).shape
    ll, logP, _ = hmm_lowrank_forward(pi, A, E, tokens, FA, FB)
    with np.errstate(invalid="ignore"):
        f = np.exp(_log(pi)[:, None] + logP[0] - ll[None, :])   # flows of P_0 (= posterior of z_0)
    f = np.where(np.isfinite(ll)[None, :], f, 0.0)
    dpi = f.sum(axis=1)
    dE = np.zeros((H, V))
    dA = np.zeros((H, H))
    W = np.zeros((H, H))
    K = np.asarray(FA).shape[-1]
    dFA = np.zeros((T - 1, B, H, K))
    dFB = np.zeros((T - 1, B, K, H))
    absdFA = np.zeros_like(dFA)
    absdFB = np.zeros_like(dFB)
    for t in range(T):
        np.add.at(dE.T, tokens[:, t], f.T)                        # dE[:, x_{t,b}] += f[:, b]
        if t == T - 1:
            break
        r = lowrank_exp_sum_bwd(A, FA[t], FB[t], logP[t + 1], f)  # the flow of S_t is P_t's
        dA += r["Fplus"]
        W += r["W"]
        dFA[t] = r["dA"]
        dFB[t] = r["dB"]
        absdFA[t] = r["absdA"]
        absdFB[t] = r["absdB"]
        f = r["e"]                                                # the flows of P_{t+1}
    return dict(ll=ll, dpi=dpi, dA=dA, W=W, dE=dE, dFA=dFA, dFB=dFB, absdFA=absdFA, absdFB=absdFB)
