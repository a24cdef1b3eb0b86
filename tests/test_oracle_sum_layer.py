"""Pins of the float64 sum-layer oracle against closed forms, invariants, special
cases and finite differences (nothing here re-types the oracle's formula)."""
import numpy as np
import pytest
from scipy.special import logsumexp

from oracle.sum_layer import sum_layer_fwd, sum_layer_bwd, sum_layer_bwd_literal
from workloads import layer_inputs


def _rand_layer(G, M, N, B, seed, cs=None, scale=3.0):
    d = layer_inputs(G, M, N, B, seed=seed, child_stride=cs, x_scale=scale, f_kind="uniform")
    return (d["theta"].astype(np.float64), d["x"].astype(np.float64), d["child_stride"],
            d["f"].astype(np.float64))


def test_uniform_theta_is_logsumexp_minus_logN():
    # theta rows = 1/N  =>  out = logsumexp_j x - log N  (scipy's logsumexp)
    rng = np.random.default_rng(10)
    N, B = 37, 9
    x = 20.0 * rng.standard_normal((N, B))
    theta = np.full((1, 5, N), 1.0 / N)
    out = sum_layer_fwd(theta, x)
    ref = logsumexp(x, axis=0) - np.log(N)
    np.testing.assert_allclose(out[0], np.broadcast_to(ref, (5, B)), rtol=0, atol=1e-12)


def test_one_hot_theta_selects_child():
    rng = np.random.default_rng(11)
    N, M, B = 16, 7, 5
    x = -500.0 + 10.0 * rng.standard_normal((N, B))        # far from 0: the shift matters
    js = rng.integers(0, N, size=M)
    theta = np.zeros((1, M, N))
    theta[0, np.arange(M), js] = 1.0
    out = sum_layer_fwd(theta, x)
    np.testing.assert_allclose(out[0], x[js], rtol=0, atol=1e-12)


def test_grouped_equals_independent_groups():
    # three groups at stride 5 > N = 4 (evenly strided children) and shared (stride 0, G=1)
    theta, x, cs, f = _rand_layer(3, 6, 4, 8, seed=12, cs=5)
    out = sum_layer_fwd(theta, x, cs)
    for g in range(3):
        og = sum_layer_fwd(theta[g:g + 1], x[g * cs:g * cs + 4], 0)
        np.testing.assert_array_equal(out[g], og[0])
    e, F = sum_layer_bwd(theta, x, cs, out, f)
    for g in range(3):
        eg, Fg = sum_layer_bwd(theta[g:g + 1], x[g * cs:g * cs + 4], 0, out[g:g + 1], f[g:g + 1])
        np.testing.assert_allclose(e[g * cs:g * cs + 4], eg, rtol=1e-13, atol=0)
        np.testing.assert_allclose(F[g], Fg[0], rtol=1e-13, atol=0)
    # the row between groups (row 4, 9) is nobody's child: zero element flow
    assert np.all(e[4] == 0) and np.all(e[9] == 0)


def test_groups_with_maxima_80_nats_apart():
    # the shift is per group: a group at -1000 nats next to one at +0 stays exact
    N, B = 8, 4
    rng = np.random.default_rng(13)
    x0 = rng.standard_normal((N, B))
    x1 = -1000.0 + rng.standard_normal((N, B))
    x = np.concatenate([x0, x1])
    theta = np.full((2, 3, N), 1.0 / N)
    out = sum_layer_fwd(theta, x, N)
    np.testing.assert_allclose(out[0], np.broadcast_to(logsumexp(x0, 0) - np.log(N), (3, B)), atol=1e-12)
    np.testing.assert_allclose(out[1], np.broadcast_to(logsumexp(x1, 0) - np.log(N), (3, B)), atol=1e-12)


def test_all_neg_inf_column_and_zero_rows():
    N, B = 6, 3
    x = np.random.default_rng(14).standard_normal((N, B))
    x[:, 1] = -np.inf                               # column with no probability mass
    theta = np.random.default_rng(15).uniform(size=(1, 4, N))
    theta[0, 2] = 0.0                               # a node with all-zero parameters
    out = sum_layer_fwd(theta, x)
    assert np.all(out[0, :, 1] == -np.inf)
    assert np.all(out[0, 2] == -np.inf)
    assert np.all(np.isfinite(np.delete(np.delete(out[0], 2, 0), 1, 1)))
    f = np.ones((1, 4, B))
    e, F = sum_layer_bwd(theta, x, 0, out, f)
    assert np.all(np.isfinite(e)) and np.all(np.isfinite(F))
    assert np.all(e[:, 1] == 0)
    assert np.all(F[0, 2] == 0)
    # one child at -inf in a finite column passes no flow to it
    x2 = x.copy()
    x2[3, 0] = -np.inf
    out2 = sum_layer_fwd(theta, x2)
    e2, _ = sum_layer_bwd(theta, x2, 0, out2, f)
    assert e2[3, 0] == 0


def test_bwd_factorisation_matches_literal_loops():
    theta, x, cs, f = _rand_layer(2, 5, 4, 6, seed=16, cs=4, scale=10.0)
    out = sum_layer_fwd(theta, x, cs)
    e, F = sum_layer_bwd(theta, x, cs, out, f)
    el, Fl = sum_layer_bwd_literal(theta, x, cs, out, f)
    np.testing.assert_allclose(e, el, rtol=1e-12, atol=0)
    np.testing.assert_allclose(F, Fl, rtol=1e-12, atol=0)


def test_flow_invariants():
    # sum_j F[i,j] = sum_b f[i,b]  and  sum_j e[j,b] = sum_i f[i,b]   (exp(out) = sum_j theta exp(x))
    theta, x, cs, f = _rand_layer(1, 64, 48, 32, seed=17, scale=3.0)
    out = sum_layer_fwd(theta, x, cs)
    e, F = sum_layer_bwd(theta, x, cs, out, f)
    np.testing.assert_allclose(F[0].sum(axis=1), f[0].sum(axis=1), rtol=1e-12)
    np.testing.assert_allclose(e.sum(axis=0), f[0].sum(axis=0), rtol=1e-12)


def test_flows_are_gradients_finite_differences():
    # e = d(sum f*out)/dx ;  F = d(sum f*out)/d(log theta)  (theta unnormalised)
    theta, x, cs, f = _rand_layer(2, 3, 4, 2, seed=18, cs=4, scale=2.0)
    out = sum_layer_fwd(theta, x, cs)
    e, F = sum_layer_bwd(theta, x, cs, out, f)

    def obj(th, xx):
        return float((f * sum_layer_fwd(th, xx, cs)).sum())

    eps = 1e-6
    for (r, b) in [(0, 0), (3, 1), (5, 0), (7, 1)]:
        xp, xm = x.copy(), x.copy()
        xp[r, b] += eps
        xm[r, b] -= eps
        fd = (obj(theta, xp) - obj(theta, xm)) / (2 * eps)
        assert abs(fd - e[r, b]) < 1e-8
    for (g, i, j) in [(0, 0, 0), (1, 2, 3), (0, 1, 2)]:
        tp, tm = theta.copy(), theta.copy()
        tp[g, i, j] *= np.exp(eps)
        tm[g, i, j] *= np.exp(-eps)
        fd = (obj(tp, x) - obj(tm, x)) / (2 * eps)
        assert abs(fd - F[g, i, j]) < 1e-8


def test_layer_workload_shapes():
    from workloads import layer
    d = layer()
    assert d["theta"].shape == (1, 1024, 1024) and d["x"].shape == (1024, 128)
    np.testing.assert_allclose(d["theta"].astype(np.float64).sum(-1), 1.0, atol=1e-5)
    # children log-values: a log-softmax over the 1024 children, spread over tens of nats
    lse = logsumexp(d["x"].astype(np.float64), axis=0)
    np.testing.assert_allclose(lse, 0.0, atol=1e-4)
    assert float(d["x"].max() - d["x"].min()) > 20.0
