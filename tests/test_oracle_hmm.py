"""Pins of the HMM-circuit oracle: brute force over hidden paths, normalisation over
all sequences, the textbook forward recursion, Baum-Welch posteriors, flow
invariants, finite differences, a closed form and a hand-worked example."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle.hmm import hmm_fwd_bwd, hmm_ll
from workloads import hmm_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(H, T, V, B, seed):
    d = hmm_inputs(H, T, V, B, seed)
    return (d["pi"].astype(np.float64), d["A"].astype(np.float64), d["E"].astype(np.float64),
            d["tokens"])


def _brute(pi, A, E, tokens):
    """Enumerate every hidden path: LL and posterior expected counts."""
    H, V = E.shape
    B, T = tokens.shape
    ll = np.empty(B)
    dpi = np.zeros(H)
    dA = np.zeros((H, H))
    dE = np.zeros((H, V))
    for b in range(B):
        x = tokens[b]
        paths = list(itertools.product(range(H), repeat=T))
        w = np.empty(len(paths))
        for n, z in enumerate(paths):
            p = pi[z[0]] * E[z[0], x[0]]
            for t in range(1, T):
                p *= A[z[t - 1], z[t]] * E[z[t], x[t]]
            w[n] = p
        P = w.sum()
        ll[b] = np.log(P)
        for n, z in enumerate(paths):
            q = w[n] / P
            dpi[z[0]] += q
            for t in range(T):
                dE[z[t], x[t]] += q
            for t in range(T - 1):
                dA[z[t], z[t + 1]] += q
    return ll, dpi, dA, dE


@pytest.mark.parametrize("H,T,V,B,seed", [(3, 5, 4, 3, 20), (2, 8, 3, 2, 21)])
def test_brute_force_paths(H, T, V, B, seed):
    pi, A, E, tok = _inputs(H, T, V, B, seed)
    ll, dpi, dA, dE = hmm_fwd_bwd(pi, A, E, tok)
    bll, bpi, bA, bE = _brute(pi, A, E, tok)
    np.testing.assert_allclose(ll, bll, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dpi, bpi, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dA, bA, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dE, bE, rtol=1e-10, atol=1e-13)


def test_probabilities_sum_to_one_over_all_sequences():
    H, T, V = 3, 4, 4
    pi, A, E, _ = _inputs(H, T, V, 1, seed=22)
    # renormalise in float64: the float32 cast leaves rows ~1e-8 off 1
    pi, A, E = pi / pi.sum(), A / A.sum(-1, keepdims=True), E / E.sum(-1, keepdims=True)
    seqs = np.array(list(itertools.product(range(V), repeat=T)), dtype=np.int32)   # 256
    ll = hmm_ll(pi, A, E, seqs)
    assert abs(np.exp(ll).sum() - 1.0) < 1e-12


def test_textbook_forward_recursion():
    # alpha_1 = pi * E[:, x1]; alpha_{t+1} = (alpha_t @ A) * E[:, x_{t+1}]; LL = log sum alpha_T
    pi, A, E, tok = _inputs(16, 12, 8, 5, seed=23)
    ll = hmm_ll(pi, A, E, tok)
    for b in range(tok.shape[0]):
        x = tok[b]
        a = pi * E[:, x[0]]
        c = 0.0
        for t in range(1, len(x)):
            s = a.sum()
            c += np.log(s)
            a = ((a / s) @ A) * E[:, x[t]]
        ref = c + np.log(a.sum())
        assert abs(ll[b] - ref) < 1e-11


def test_baum_welch_posteriors():
    # scaled forward-backward (Rabiner): gamma and xi give dpi, dA, dE
    pi, A, E, tok = _inputs(10, 9, 6, 4, seed=24)
    _, dpi, dA, dE = hmm_fwd_bwd(pi, A, E, tok)
    H, V = E.shape
    rpi, rA, rE = np.zeros(H), np.zeros((H, H)), np.zeros((H, V))
    for b in range(tok.shape[0]):
        x = tok[b]
        T = len(x)
        al = np.zeros((T, H))
        c = np.zeros(T)
        al[0] = pi * E[:, x[0]]
        c[0] = al[0].sum()
        al[0] /= c[0]
        for t in range(1, T):
            al[t] = (al[t - 1] @ A) * E[:, x[t]]
            c[t] = al[t].sum()
            al[t] /= c[t]
        be = np.ones((T, H))
        for t in range(T - 2, -1, -1):
            be[t] = (A @ (E[:, x[t + 1]] * be[t + 1])) / c[t + 1]
        gam = al * be
        rpi += gam[0]
        for t in range(T):
            rE[:, x[t]] += gam[t]
        for t in range(T - 1):
            rA += al[t][:, None] * A * (E[:, x[t + 1]] * be[t + 1])[None, :] / c[t + 1]
    np.testing.assert_allclose(dpi, rpi, rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(dA, rA, rtol=1e-9, atol=1e-14)
    np.testing.assert_allclose(dE, rE, rtol=1e-10, atol=1e-14)


def test_flow_invariants():
    pi, A, E, tok = _inputs(32, 8, 16, 16, seed=1)       # the tiny HMM workload's shape
    _, dpi, dA, dE = hmm_fwd_bwd(pi, A, E, tok)
    B, T = tok.shape
    assert abs(dpi.sum() - B) < 1e-9
    assert abs(dA.sum() - B * (T - 1)) < 1e-8
    assert abs(dE.sum() - B * T) < 1e-8
    # each emission column's flow mass = number of occurrences of that token
    counts = np.bincount(tok.ravel(), minlength=E.shape[1])
    np.testing.assert_allclose(dE.sum(axis=0), counts, atol=1e-9)


def test_flows_are_gradients_finite_differences():
    # dpi, dA, dE = d(sum_b LL)/d(log param)  (parameters unnormalised)
    pi, A, E, tok = _inputs(4, 5, 3, 3, seed=25)
    _, dpi, dA, dE = hmm_fwd_bwd(pi, A, E, tok)
    eps = 1e-6

    def obj(p, a, e):
        return float(hmm_ll(p, a, e, tok).sum())

    for k in range(4):
        pp, pm = pi.copy(), pi.copy()
        pp[k] *= np.exp(eps)
        pm[k] *= np.exp(-eps)
        assert abs((obj(pp, A, E) - obj(pm, A, E)) / (2 * eps) - dpi[k]) < 1e-8
    for (k, l) in [(0, 0), (1, 3), (3, 2)]:
        ap, am = A.copy(), A.copy()
        ap[k, l] *= np.exp(eps)
        am[k, l] *= np.exp(-eps)
        assert abs((obj(pi, ap, E) - obj(pi, am, E)) / (2 * eps) - dA[k, l]) < 1e-8
    for (k, v) in [(0, 0), (2, 1), (3, 2)]:
        ep, em = E.copy(), E.copy()
        ep[k, v] *= np.exp(eps)
        em[k, v] *= np.exp(-eps)
        assert abs((obj(pi, A, ep) - obj(pi, A, em)) / (2 * eps) - dE[k, v]) < 1e-8


def test_uniform_emissions_closed_form():
    # E = 1/V  =>  LL = -T log V for every pi and A
    H, T, V, B = 64, 16, 1024, 4
    pi, A, _, tok = _inputs(H, T, V, B, seed=26)
    pi, A = pi / pi.sum(), A / A.sum(-1, keepdims=True)      # exact rows in float64
    E = np.full((H, V), 1.0 / V)
    ll = hmm_ll(pi, A, E, tok)
    np.testing.assert_allclose(ll, -T * np.log(V), rtol=0, atol=1e-10)


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "hmm_2state_hand.json")) as fh:
        g = json.load(fh)
    ll, dpi, dA, dE = hmm_fwd_bwd(np.array(g["pi"]), np.array(g["A"]), np.array(g["E"]),
                                  np.array(g["tokens"], dtype=np.int32))
    num, den = g["P_fraction"]
    assert abs(ll[0] - np.log(num / den)) < 1e-14
    np.testing.assert_allclose(dpi, np.array(g["posterior_z1"]), rtol=1e-13)
