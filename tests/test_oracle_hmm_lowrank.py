"""Pins of the HMM-with-LowRank-transitions oracle (oracle/hmm_lowrank.py): zero factors
against the plain HMM oracle, the log-likelihood against a sum over every hidden path
with each sample's own transition matrices, finite differences of sum_b LL against the
factor gradients, and the flow totals (posterior expected counts)."""
import itertools

import numpy as np

from oracle.hmm import hmm_fwd_bwd
from oracle.hmm_lowrank import hmm_lowrank_forward, hmm_lowrank_fwd_bwd
from workloads import hmm_inputs


def _case(H=4, T=4, V=3, B=3, K=2, spread=1.0, seed=20):
    d = hmm_inputs(H, T, V, B, seed=seed)
    rng = np.random.default_rng(seed + 1)
    s = np.sqrt(spread / np.sqrt(K))
    FA = s * rng.standard_normal((T - 1, B, H, K))
    FB = s * rng.standard_normal((T - 1, B, K, H))
    return d, FA, FB


def test_zero_factors_are_the_plain_hmm():
    d, FA, FB = _case(H=5, T=5, V=4, B=4)
    FA[:] = 0.0
    r = hmm_lowrank_fwd_bwd(d["pi"], d["A"], d["E"], d["tokens"], FA, FB)
    # theta_b = A g / Z normalizes A's rows over the children: the plain HMM with the
    # float32 A's rows normalized in float64
    A = d["A"].astype(np.float64)
    An = A / A.sum(1, keepdims=True)
    ll, dpi, dA, dE = hmm_fwd_bwd(d["pi"], An, d["E"], d["tokens"])  # F+: flows of the effective A
    np.testing.assert_allclose(r["ll"], ll, rtol=1e-12)
    np.testing.assert_allclose(r["dpi"], dpi, rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(r["dA"], dA, rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(r["dE"], dE, rtol=1e-10, atol=1e-14)


def test_log_likelihood_by_enumerating_paths():
    d, FA, FB = _case()
    pi, A, E = (d[k].astype(np.float64) for k in ("pi", "A", "E"))
    ll, _, _ = hmm_lowrank_forward(pi, A, E, d["tokens"], FA, FB)
    B, T = d["tokens"].shape
    H = A.shape[0]
    for b in range(B):
        x = d["tokens"][b]
        At = []
        for t in range(T - 1):
            g = A * np.exp(FA[t, b] @ FB[t, b])
            At.append(g / g.sum(1, keepdims=True))              # A_b^(t), rows normalized
        p = 0.0
        for z in itertools.product(range(H), repeat=T):
            w = pi[z[0]] * np.prod([E[z[t], x[t]] for t in range(T)])
            w *= np.prod([At[t][z[t], z[t + 1]] for t in range(T - 1)])
            p += w
        assert abs(ll[b] - np.log(p)) <= 1e-12 * max(1.0, abs(np.log(p)))


def test_finite_differences_of_the_factor_gradients():
    d, FA, FB = _case(seed=21)
    r = hmm_lowrank_fwd_bwd(d["pi"], d["A"], d["E"], d["tokens"], FA, FB)
    obj = lambda fa, fb: float(hmm_lowrank_forward(d["pi"], d["A"], d["E"], d["tokens"], fa, fb)[0].sum())
    h = 1e-6
    rng = np.random.default_rng(3)
    for _ in range(6):
        t, b, k, q = rng.integers(3), rng.integers(3), rng.integers(4), rng.integers(2)
        p, m = FA.copy(), FA.copy()
        p[t, b, k, q] += h
        m[t, b, k, q] -= h
        assert abs((obj(p, FB) - obj(m, FB)) / (2 * h) - r["dFA"][t, b, k, q]) <= 1e-7
        p, m = FB.copy(), FB.copy()
        p[t, b, q, k] += h
        m[t, b, q, k] -= h
        assert abs((obj(FA, p) - obj(FA, m)) / (2 * h) - r["dFB"][t, b, q, k]) <= 1e-7


def test_flow_totals():
    d, FA, FB = _case(H=6, T=5, V=4, B=7, spread=2.0, seed=22)
    r = hmm_lowrank_fwd_bwd(d["pi"], d["A"], d["E"], d["tokens"], FA, FB)
    B, T = d["tokens"].shape
    np.testing.assert_allclose(r["dpi"].sum(), B, rtol=1e-12)
    np.testing.assert_allclose(r["dA"].sum(), B * (T - 1), rtol=1e-12)
    np.testing.assert_allclose((d["A"] * r["W"]).sum(), B * (T - 1), rtol=1e-12)
    np.testing.assert_allclose(r["dE"].sum(0), np.bincount(d["tokens"].ravel(), minlength=4), rtol=1e-12)
