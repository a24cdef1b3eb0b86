"""Pins of the float64 EM M-step oracle (oracle/em.py) to facts other than itself:
the closed form of normalize on scaled stochastic rows, the readings for empty rows,
Baum-Welch against expected counts enumerated over every hidden path of a tiny HMM, the
monotone log-likelihood of repeated Baum-Welch steps, the monotone objective of the
LowRank conditional step (a minorize-maximize step of a row-scale-invariant objective),
and its reduction to the plain step when the scale is 1."""
import itertools

import numpy as np
import pytest

from oracle.em import em_conditional, em_plain, hmm_em_step, normalize
from oracle.hmm import hmm_ll
from oracle.lowrank import lowrank_exp_sum_bwd, lowrank_exp_sum_fwd
from oracle.sum_layer import sum_layer_bwd, sum_layer_fwd
from workloads import hmm_inputs



def test_normalize_scaled_stochastic_rows():
    rng = np.random.default_rng(0)
    P = rng.random((3, 5, 7))
    P /= P.sum(-1, keepdims=True)
    s = rng.random((3, 5, 1)) * 10 + 0.1
    out = normalize(s * P, np.zeros_like(P))
    np.testing.assert_allclose(out, P, rtol=1e-14, atol=0)
    np.testing.assert_allclose(out.sum(-1), 1.0, rtol=1e-14)


def test_readings_empty_rows_and_zero_denominators():
    prev = np.array([[0.5, 0.5, 0.0], [0.2, 0.3, 0.5]])
    F = np.array([[0.0, 0.0, 0.0], [1.0, 2.0, 1.0]])
    out = em_plain(F, prev)
    np.testing.assert_array_equal(out[0], prev[0])          # no flow: keeps its parameters
    np.testing.assert_allclose(out[1], [0.25, 0.5, 0.25])
    W = np.array([[0.0, 1.0, 2.0], [2.0, 0.0, 1.0]])
    Fp = np.array([[0.0, 1.0, 1.0], [2.0, 0.0, 3.0]])
    out = em_conditional(Fp, W, prev)
    np.testing.assert_allclose(out[0], [0.0, 2 / 3, 1 / 3])  # F+/W = (0, 1, 1/2)
    np.testing.assert_allclose(out[1], [0.25, 0.0, 0.75])    # F+/W = (1, 0, 3)


def _path_counts(pi, A, E, tokens):
    """Posterior expected counts by enumerating every hidden path (tiny H, T)."""
    pi, A, E = (np.asarray(a, np.float64) for a in (pi, A, E))
    H, V = E.shape
    cpi, cA, cE = np.zeros(H), np.zeros((H, H)), np.zeros((H, V))
    for x in tokens:
        T = len(x)
        paths = list(itertools.product(range(H), repeat=T))
        w = np.array([pi[z[0]] * np.prod([E[z[t], x[t]] for t in range(T)])
                      * np.prod([A[z[t], z[t + 1]] for t in range(T - 1)]) for z in paths])
        w /= w.sum()
        for z, wz in zip(paths, w):
            cpi[z[0]] += wz
            for t in range(T - 1):
                cA[z[t], z[t + 1]] += wz
            for t in range(T):
                cE[z[t], x[t]] += wz
    return cpi, cA, cE


def test_baum_welch_matches_enumerated_counts():
    d = hmm_inputs(3, 4, 3, 5, seed=11)
    cpi, cA, cE = _path_counts(d["pi"], d["A"], d["E"], d["tokens"])
    npi, nA, nE = hmm_em_step(d["pi"], d["A"], d["E"], d["tokens"])
    np.testing.assert_allclose(npi, cpi / cpi.sum(), rtol=1e-10)
    np.testing.assert_allclose(nA, cA / cA.sum(1, keepdims=True), rtol=1e-10)
    np.testing.assert_allclose(nE, cE / cE.sum(1, keepdims=True), rtol=1e-10)


def test_baum_welch_log_likelihood_never_decreases():
    d = hmm_inputs(5, 6, 4, 12, seed=12)
    pi, A, E = d["pi"], d["A"], d["E"]
    prev = hmm_ll(pi, A, E, d["tokens"]).sum()
    for _ in range(6):
        pi, A, E = hmm_em_step(pi, A, E, d["tokens"])
        ll = hmm_ll(pi, A, E, d["tokens"]).sum()
        assert ll >= prev - 1e-9
        prev = ll


def _lowrank_case(seed, M=6, N=9, K=3, B=5, spread=1.0):
    rng = np.random.default_rng(seed)
    theta = rng.random((M, N)) + 0.05
    theta /= theta.sum(1, keepdims=True)
    A = rng.normal(0, spread, (B, M, K)) / np.sqrt(K)
    Bm = rng.normal(0, spread, (B, K, N))
    x = rng.normal(0, 2, (N, B))
    f = rng.random((M, B)) + 0.1
    return theta, A, Bm, x, f


def test_lowrank_conditional_step_increases_flow_weighted_objective():
    # sum_b sum_i f_b[i] out_b[i] does not change when a row of theta is scaled, and the
    # conditional update maximises a minorizer of it (log Z <= log Z0 + Z / Z0 - 1)
    theta, A, Bm, x, f = _lowrank_case(3)
    obj = lambda th: float((f * lowrank_exp_sum_fwd(th, A, Bm, x)[0]).sum())
    prev = obj(theta)
    for _ in range(8):
        r = lowrank_exp_sum_bwd(theta, A, Bm, x, f)
        theta = em_conditional(r["Fplus"], r["W"], theta)
        cur = obj(theta)
        assert cur >= prev - 1e-10
        prev = cur
    # and the plain normalize(F+) of the same statistics is a different update
    r = lowrank_exp_sum_bwd(theta, A, Bm, x, f)
    assert np.abs(em_plain(r["Fplus"], theta) - em_conditional(r["Fplus"], r["W"], theta)).max() > 1e-6


def test_lowrank_conditional_with_unit_scale_is_the_plain_step():
    theta, A, Bm, x, f = _lowrank_case(4)
    A[:] = 0.0
    r = lowrank_exp_sum_bwd(theta, A, Bm, x, f)
    out = sum_layer_fwd(theta[None], x, 0)
    _, F = sum_layer_bwd(theta[None], x, 0, out, f[None])
    np.testing.assert_allclose(em_conditional(r["Fplus"], r["W"], theta), em_plain(F[0], theta), rtol=1e-12)
