"""Pins of the LowRank "sum_exp" oracle (pyjuice LowRank API doc, intro formulas):
finite differences of the flow-weighted objective against dA, dB and the element flows,
the rank-one form against "exp_sum" with an augmented rank two (exp(a) exp(b) = exp(a +
b)), a scale constant along the children (B = 0) against the plain sum layer, the
per-sample dense restatement through the sum-layer oracle, and the flow invariants."""
import numpy as np

from oracle.lowrank import lowrank_exp_sum_bwd, lowrank_sum_exp_bwd, lowrank_sum_exp_fwd
from oracle.sum_layer import sum_layer_bwd, sum_layer_fwd


def _case(seed, M=6, N=9, K=3, B=4, spread=1.0):
    rng = np.random.default_rng(seed)
    theta = rng.random((M, N)) + 0.05
    theta /= theta.sum(1, keepdims=True)
    A = rng.normal(0, spread, (B, M, K))
    Bm = rng.normal(0, spread, (B, K, N))
    x = rng.normal(0, 2, (N, B))
    f = rng.random((M, B)) + 0.1
    return theta, A, Bm, x, f


def test_finite_differences_of_the_objective():
    theta, A, Bm, x, f = _case(1)
    r = lowrank_sum_exp_bwd(theta, A, Bm, x, f)
    obj = lambda A_, B_, x_: float((f * lowrank_sum_exp_fwd(theta, A_, B_, x_)[0]).sum())
    h = 1e-6
    rng = np.random.default_rng(2)
    for _ in range(6):
        b, i, k = rng.integers(4), rng.integers(6), rng.integers(3)
        Ap, Am = A.copy(), A.copy()
        Ap[b, i, k] += h
        Am[b, i, k] -= h
        assert abs((obj(Ap, Bm, x) - obj(Am, Bm, x)) / (2 * h) - r["dA"][b, i, k]) <= 1e-7
        j = rng.integers(9)
        Bp, Bn = Bm.copy(), Bm.copy()
        Bp[b, k, j] += h
        Bn[b, k, j] -= h
        assert abs((obj(A, Bp, x) - obj(A, Bn, x)) / (2 * h) - r["dB"][b, k, j]) <= 1e-7
        xp, xn = x.copy(), x.copy()
        xp[j, b] += h
        xn[j, b] -= h
        assert abs((obj(A, Bm, xp) - obj(A, Bm, xn)) / (2 * h) - r["e"][j, b]) <= 1e-7


def test_rank_one_is_exp_sum_of_the_augmented_rank_two():
    theta, A, Bm, x, f = _case(3, K=1)
    B = x.shape[1]
    A2 = np.concatenate([A, np.ones_like(A)], axis=2)             # [A_i, 1]
    B2 = np.concatenate([np.ones_like(Bm), Bm], axis=1)           # [1; B_j]: A2 B2 = A_i + B_j
    s = lowrank_sum_exp_bwd(theta, A, Bm, x, f)
    e = lowrank_exp_sum_bwd(theta, A2, B2, x, f)
    for k in ("out", "logZ", "e", "Fplus", "W"):
        np.testing.assert_allclose(s[k], e[k], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dA"][:, :, 0], e["dA"][:, :, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(s["dB"][:, 0, :], e["dB"][:, 1, :], rtol=1e-10, atol=1e-12)
    assert B == 4


def test_scale_constant_along_children_is_the_plain_layer():
    theta, A, Bm, x, f = _case(4)
    Bm[:] = 0.0                                                   # g[i, j] = sum_r exp(A[i, r])
    r = lowrank_sum_exp_bwd(theta, A, Bm, x, f)
    out = sum_layer_fwd(theta[None], x, 0)[0]
    np.testing.assert_allclose(r["out"], out, rtol=1e-12, atol=1e-12)
    e, F = sum_layer_bwd(theta[None], x, 0, out[None], f[None])
    np.testing.assert_allclose(r["e"], e, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(r["Fplus"], F[0], rtol=1e-10, atol=1e-12)
    # W = sum_b f g / Z with g / Z = 1 / sum_j theta = 1 (theta's rows are normalized)
    np.testing.assert_allclose(r["W"], np.repeat(f.sum(1, keepdims=True), theta.shape[1], 1), rtol=1e-10)


def test_dense_restatement_through_the_sum_layer():
    theta, A, Bm, x, f = _case(5, spread=0.5)
    out, logZ = lowrank_sum_exp_fwd(theta, A, Bm, x)
    for b in range(x.shape[1]):
        g = np.exp(A[b]) @ np.exp(Bm[b])                          # the definition, unshifted
        Z = (theta * g).sum(1)
        tb = theta * g / Z[:, None]
        np.testing.assert_allclose(out[:, b], sum_layer_fwd(tb[None], x[:, b:b + 1], 0)[0, :, 0], rtol=1e-12)
        np.testing.assert_allclose(logZ[b], np.log(Z), rtol=1e-12)


def test_flow_invariants():
    theta, A, Bm, x, f = _case(6, spread=2.0)
    r = lowrank_sum_exp_bwd(theta, A, Bm, x, f)
    np.testing.assert_allclose(r["Fplus"].sum(1), f.sum(1), rtol=1e-12)      # sum_j p = 1
    np.testing.assert_allclose((theta * r["W"]).sum(1), f.sum(1), rtol=1e-12)  # sum_j theta g / Z = 1
    # sum_r dA[b, i, r] = sum_j (D / g) g = sum_j D[i, j] = f_i (sum_j p - sum_j q) = 0
    np.testing.assert_allclose(r["dA"].sum(2), 0.0, atol=1e-12)
