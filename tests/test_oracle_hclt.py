"""Pins of the HCLT-circuit oracle: brute force over latent assignments,
normalisation over all data, the chain tree = HMM cross-check, a closed form,
flow invariants and finite differences."""
import itertools

import numpy as np

from oracle.hclt import hclt_fwd_bwd, hclt_ll
from oracle.hmm import hmm_fwd_bwd
from workloads import hclt_inputs, hclt_parents, hmm_inputs


def _inputs(n, H, C, B, seed, parent=None):
    d = hclt_inputs(n, H, C, B, seed, parent=parent)
    return (d["parent"], d["data"], d["pi"].astype(np.float64), d["W"].astype(np.float64),
            d["E"].astype(np.float64))


def _brute(parent, data, pi, W, E):
    n = len(parent)
    H = len(pi)
    B = data.shape[0]
    C = E.shape[2]
    ll = np.empty(B)
    dpi = np.zeros(H)
    dW = np.zeros((n, H, H))
    dE = np.zeros((n, H, C))
    assigns = list(itertools.product(range(H), repeat=n))
    for b in range(B):
        x = data[b]
        w = np.empty(len(assigns))
        for a, z in enumerate(assigns):
            p = pi[z[0]]
            for v in range(n):
                p *= E[v, z[v], x[v]]
                if v > 0:
                    p *= W[v, z[parent[v]], z[v]]
            w[a] = p
        P = w.sum()
        ll[b] = np.log(P)
        for a, z in enumerate(assigns):
            q = w[a] / P
            dpi[z[0]] += q
            for v in range(n):
                dE[v, z[v], x[v]] += q
                if v > 0:
                    dW[v, z[parent[v]], z[v]] += q
    return ll, dpi, dW, dE


def test_brute_force_assignments():
    parent, data, pi, W, E = _inputs(5, 2, 3, 3, seed=30)
    ll, dpi, dW, dE = hclt_fwd_bwd(parent, data, pi, W, E)
    bll, bpi, bW, bE = _brute(parent, data, pi, W, E)
    np.testing.assert_allclose(ll, bll, atol=1e-12)
    np.testing.assert_allclose(dpi, bpi, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dW[1:], bW[1:], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dE, bE, rtol=1e-10, atol=1e-13)


def test_star_and_branching_trees_brute_force():
    for parent in (np.array([-1, 0, 0, 0, 0], np.int32), np.array([-1, 0, 1, 1, 0], np.int32)):
        p, data, pi, W, E = _inputs(5, 3, 2, 2, seed=31, parent=parent)
        ll, dpi, dW, dE = hclt_fwd_bwd(p, data, pi, W, E)
        bll, bpi, bW, bE = _brute(p, data, pi, W, E)
        np.testing.assert_allclose(ll, bll, atol=1e-12)
        np.testing.assert_allclose(dW[1:], bW[1:], rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(dE, bE, rtol=1e-10, atol=1e-13)


def test_probabilities_sum_to_one_over_all_data():
    parent, _, pi, W, E = _inputs(4, 3, 3, 1, seed=32)
    # renormalise in float64: the float32 cast leaves rows ~1e-8 off 1
    pi, W, E = pi / pi.sum(), W / W.sum(-1, keepdims=True), E / E.sum(-1, keepdims=True)
    data = np.array(list(itertools.product(range(3), repeat=4)), dtype=np.int32)   # 81
    ll = hclt_ll(parent, data, pi, W, E)
    assert abs(np.exp(ll).sum() - 1.0) < 1e-12


def test_chain_tree_equals_hmm():
    H, T, V, B = 6, 7, 5, 4
    d = hmm_inputs(H, T, V, B, seed=33)
    pi, A, E = (d[k].astype(np.float64) for k in ("pi", "A", "E"))
    parent = np.arange(-1, T - 1, dtype=np.int32)
    W = np.broadcast_to(A, (T, H, H)).copy()
    Ev = np.broadcast_to(E, (T, H, V)).copy()
    ll, dpi, dW, dE = hclt_fwd_bwd(parent, d["tokens"], pi, W, Ev)
    hll, hpi, hA, hE = hmm_fwd_bwd(pi, A, E, d["tokens"])
    np.testing.assert_allclose(ll, hll, atol=1e-12)
    np.testing.assert_allclose(dpi, hpi, rtol=1e-11)
    np.testing.assert_allclose(dW[1:].sum(0), hA, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(dE.sum(0), hE, rtol=1e-11, atol=1e-14)


def test_uniform_emissions_closed_form():
    n, H, C, B = 40, 8, 16, 3
    parent, data, pi, W, _ = _inputs(n, H, C, B, seed=34)
    pi, W = pi / pi.sum(), W / W.sum(-1, keepdims=True)      # exact rows in float64
    E = np.full((n, H, C), 1.0 / C)
    ll = hclt_ll(parent, data, pi, W, E)
    np.testing.assert_allclose(ll, -n * np.log(C), atol=1e-10)


def test_flow_invariants():
    n, H, C, B = 30, 6, 5, 7
    parent, data, pi, W, E = _inputs(n, H, C, B, seed=35)
    _, dpi, dW, dE = hclt_fwd_bwd(parent, data, pi, W, E)
    assert abs(dpi.sum() - B) < 1e-10
    np.testing.assert_allclose(dW[1:].sum(axis=(1, 2)), B, atol=1e-10)
    np.testing.assert_allclose(dE.sum(axis=(1, 2)), B, atol=1e-10)
    # the flow into a child's latents equals the flow into the parent's latents
    np.testing.assert_allclose(dW[1:].sum(axis=2), dE[parent[1:]].sum(axis=2), atol=1e-10)


def test_flows_are_gradients_finite_differences():
    parent, data, pi, W, E = _inputs(6, 3, 4, 2, seed=36)
    _, dpi, dW, dE = hclt_fwd_bwd(parent, data, pi, W, E)
    eps = 1e-6

    def obj(p, w, e):
        return float(hclt_ll(parent, data, p, w, e).sum())

    for (c, z, y) in [(1, 0, 0), (3, 2, 1), (5, 1, 2)]:
        wp, wm = W.copy(), W.copy()
        wp[c, z, y] *= np.exp(eps)
        wm[c, z, y] *= np.exp(-eps)
        assert abs((obj(pi, wp, E) - obj(pi, wm, E)) / (2 * eps) - dW[c, z, y]) < 1e-8
    for (v, z, k) in [(0, 0, 1), (4, 2, 3)]:
        ep, em = E.copy(), E.copy()
        ep[v, z, k] *= np.exp(eps)
        em[v, z, k] *= np.exp(-eps)
        assert abs((obj(pi, W, ep) - obj(pi, W, em)) / (2 * eps) - dE[v, z, k]) < 1e-8


def test_parent_recipe():
    p = hclt_parents(768, seed=5)
    assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, 768))
