"""Pins of the LowRank exp_sum oracle: reductions to the plain sum layer, a scale
constant along the children, invariants, finite differences and a dense
per-sample restatement through the sum-layer oracle."""
import numpy as np

from oracle.lowrank import lowrank_exp_sum_fwd, lowrank_exp_sum_bwd
from oracle.sum_layer import sum_layer_fwd, sum_layer_bwd
from workloads import lowrank_inputs


def _inputs(M, N, K, B, spread, seed):
    d = lowrank_inputs(M, N, K, B, spread, seed, f_kind="uniform")
    return tuple(d[k].astype(np.float64) for k in ("theta", "A", "Bm", "x", "f"))


def test_zero_scale_reduces_to_sum_layer():
    th, A, Bm, x, f = _inputs(12, 10, 3, 5, 1.0, seed=40)
    A0, B0 = np.zeros_like(A), np.zeros_like(Bm)
    out, _ = lowrank_exp_sum_fwd(th, A0, B0, x)
    ref = sum_layer_fwd(th[None], x)[0]
    np.testing.assert_allclose(out, ref, atol=1e-12)
    r = lowrank_exp_sum_bwd(th, A0, B0, x, f)
    e, F = sum_layer_bwd(th[None], x, 0, ref[None], f[None])
    np.testing.assert_allclose(r["e"], e, rtol=1e-11)
    np.testing.assert_allclose(r["Fplus"], F[0], rtol=1e-11)
    # W = sum_b f_b[i] g/Z with g = 1 and Z = sum_j theta: row-constant sum_b f / sum_j theta
    wref = f.sum(1) / th.sum(1)
    np.testing.assert_allclose(r["W"], np.broadcast_to(wref[:, None], th.shape), rtol=1e-12)
    assert np.all(r["dA"] == 0) and np.all(r["dB"] == 0)
    # with only A = 0, dB = A^T D vanishes while dA = D B^T need not
    r2 = lowrank_exp_sum_bwd(th, A0, Bm, x, f)
    assert np.all(r2["dB"] == 0)


def test_scale_constant_along_children_leaves_theta():
    th, A, Bm, x, f = _inputs(8, 9, 4, 3, 4.0, seed=41)
    Bc = np.repeat(Bm[:, :, :1], Bm.shape[2], axis=2)     # every column of B_b equal
    out, logZ = lowrank_exp_sum_fwd(th, A, Bc, x)
    np.testing.assert_allclose(out, sum_layer_fwd(th[None], x)[0], atol=1e-12)
    # Z_b[i] = exp(A_b[i] . B_b[:,0]) * sum_j theta[i,j]
    s = np.einsum("bik,bk->bi", A, Bc[:, :, 0])
    np.testing.assert_allclose(logZ, s + np.log(th.sum(1))[None, :], atol=1e-12)


def test_invariants():
    th, A, Bm, x, f = _inputs(16, 20, 4, 6, 1.0, seed=42)
    r = lowrank_exp_sum_bwd(th, A, Bm, x, f)
    np.testing.assert_allclose(r["Fplus"].sum(1), f.sum(1), rtol=1e-11)
    np.testing.assert_allclose((th * r["W"]).sum(1), f.sum(1), rtol=1e-11)
    np.testing.assert_allclose(r["e"].sum(0), f.sum(0), rtol=1e-11)


def test_finite_differences():
    th, A, Bm, x, f = _inputs(4, 5, 2, 2, 4.0, seed=43)
    r = lowrank_exp_sum_bwd(th, A, Bm, x, f)
    eps = 1e-6

    def obj(t, a, bm, xx):
        return float((f * lowrank_exp_sum_fwd(t, a, bm, xx)[0]).sum())

    for idx in [(0, 0, 0), (1, 3, 1), (0, 2, 1)]:
        ap, am = A.copy(), A.copy()
        ap[idx] += eps
        am[idx] -= eps
        assert abs((obj(th, ap, Bm, x) - obj(th, am, Bm, x)) / (2 * eps) - r["dA"][idx]) < 1e-8
    for idx in [(0, 0, 0), (1, 1, 4), (0, 1, 2)]:
        bp, bm = Bm.copy(), Bm.copy()
        bp[idx] += eps
        bm[idx] -= eps
        assert abs((obj(th, A, bp, x) - obj(th, A, bm, x)) / (2 * eps) - r["dB"][idx]) < 1e-8
    # d/d log theta = F+ - theta * W  (F- = theta W)
    for (i, j) in [(0, 0), (2, 3), (3, 4)]:
        tp, tm = th.copy(), th.copy()
        tp[i, j] *= np.exp(eps)
        tm[i, j] *= np.exp(-eps)
        fd = (obj(tp, A, Bm, x) - obj(tm, A, Bm, x)) / (2 * eps)
        assert abs(fd - (r["Fplus"][i, j] - th[i, j] * r["W"][i, j])) < 1e-8
    # d/dx = element flows
    for (j, b) in [(0, 0), (4, 1)]:
        xp, xm = x.copy(), x.copy()
        xp[j, b] += eps
        xm[j, b] -= eps
        assert abs((obj(th, A, Bm, xp) - obj(th, A, Bm, xm)) / (2 * eps) - r["e"][j, b]) < 1e-8


def test_dense_per_sample_restatement():
    th, A, Bm, x, f = _inputs(10, 7, 3, 4, 1.0, seed=44)
    r = lowrank_exp_sum_bwd(th, A, Bm, x, f)
    Fp = np.zeros_like(th)
    for b in range(x.shape[1]):
        g = np.exp(A[b] @ Bm[b])
        tb = th * g / (th * g).sum(1, keepdims=True)
        ob = sum_layer_fwd(tb[None], x[:, b:b + 1])
        np.testing.assert_allclose(r["out"][:, b], ob[0, :, 0], atol=1e-12)
        eb, Fb = sum_layer_bwd(tb[None], x[:, b:b + 1], 0, ob, f[None, :, b:b + 1])
        np.testing.assert_allclose(r["e"][:, b], eb[:, 0], rtol=1e-11)
        Fp += Fb[0]
    np.testing.assert_allclose(r["Fplus"], Fp, rtol=1e-11)


def test_spread_recipe():
    d = lowrank_inputs(256, 256, 16, 4, 4.0, seed=8)
    S = np.einsum("bik,bkj->bij", d["A"].astype(np.float64), d["Bm"].astype(np.float64))
    assert 3.6 < S.std() < 4.4


def test_gradient_magnitudes_bound_gradients():
    th, A, Bm, x, f = _inputs(6, 7, 3, 2, 1.0, seed=44)
    r = lowrank_exp_sum_bwd(th, A, Bm, x, f)
    assert np.all(np.abs(r["dA"]) <= r["absdA"] * (1 + 1e-12))
    assert np.all(np.abs(r["dB"]) <= r["absdB"] * (1 + 1e-12))
    # with A = 0, |A|^T |f| (p + q) vanishes with dB
    r0 = lowrank_exp_sum_bwd(th, np.zeros_like(A), Bm, x, f)
    assert np.all(r0["absdB"] == 0)
