"""GPU parity of the whole HCLT circuit (pc_hclt_fwd_bwd through the C ABI) against the
float64 oracle: random, star, chain and single-variable trees with every size off the
tile sizes, in every mode; the 768-variable workload on every output and on the
uniform-emission closed form."""
import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from oracle.hclt import hclt_fwd_bwd
from tolerances import FLOW_TOL, LL_TOL, MODES, flow_err, ll_err
from workloads import hclt, hclt_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pc.load()


def _gpu_run(d, mode, flows=True):
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("data", "pi", "W", "E")}
    ll, dpi, dW, dE = pc.hclt_fwd_bwd(d["parent"], t["data"], t["pi"], t["W"], t["E"], precision=mode, flows=flows)
    torch.cuda.synchronize()
    pc.device_status()
    cpu = lambda v: None if v is None else v.cpu().numpy()
    return cpu(ll), cpu(dpi), cpu(dW), cpu(dE)


def _oracle(d):
    return hclt_fwd_bwd(d["parent"], d["data"], d["pi"], d["W"], d["E"])


@pytest.mark.parametrize("mode", MODES)
def test_random_tree_ragged(mode):
    d = hclt_inputs(40, 130, 17, 45, seed=200)
    rl, rpi, rW, rE = _oracle(d)
    ll, dpi, dW, dE = _gpu_run(d, mode)
    errs = ll_err(ll, rl), flow_err(dpi, rpi), flow_err(dW[1:], rW[1:]), flow_err(dE, rE)
    print(f"hclt 40x130 {mode}: ll {errs[0]:.3e} dpi {errs[1]:.3e} dW {errs[2]:.3e} dE {errs[3]:.3e}")
    assert errs[0] <= LL_TOL[mode]
    assert max(errs[1:]) <= FLOW_TOL[mode]
    assert np.all(dW[0] == 0)


@pytest.mark.parametrize("parent", [
    [-1],                                   # one variable: no edge
    [-1, 0],                                # one edge
    [-1, 0, 0, 0, 0, 0, 0],                 # star: six children in one level
    [-1, 0, 1, 2, 3, 4, 5, 6],              # chain: eight levels of one edge
])
def test_tree_shapes(parent):
    p = np.array(parent, dtype=np.int32)
    d = hclt_inputs(len(p), 70, 9, 33, seed=201, parent=p)
    rl, rpi, rW, rE = _oracle(d)
    ll, dpi, dW, dE = _gpu_run(d, "fp32")
    assert ll_err(ll, rl) <= LL_TOL["fp32"]
    assert flow_err(dpi, rpi) <= FLOW_TOL["fp32"]
    assert flow_err(dE, rE) <= FLOW_TOL["fp32"]
    if len(p) > 1:
        assert flow_err(dW[1:], rW[1:]) <= FLOW_TOL["fp32"]


def test_forward_only_and_accumulate():
    d = hclt_inputs(20, 96, 6, 40, seed=202)
    a = _gpu_run(d, "fp32", flows=False)
    assert a[1] is None
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("data", "pi", "W", "E")}
    ll, dpi, dW, dE = pc.hclt_fwd_bwd(d["parent"], t["data"], t["pi"], t["W"], t["E"], precision="fp32")
    assert np.array_equal(ll.cpu().numpy(), a[0])
    ll2, dpi2, dW2, dE2 = pc.hclt_fwd_bwd(d["parent"], t["data"], t["pi"], t["W"], t["E"], precision="fp32",
                                          dpi=dpi.clone(), dW=dW.clone(), dE=dE.clone(), accumulate=True)
    for x, y in ((dpi, dpi2), (dW, dW2), (dE, dE2)):
        torch.testing.assert_close(y, 2 * x, rtol=1e-6, atol=0)


@pytest.mark.parametrize("mode", MODES)
def test_latents_a_multiple_of_four(mode):
    # H % 4 == 0 but H % 8 != 0 and off the tile sizes: the parameter flows take the
    # persistent tiles with the theta ring (partial chunks), the element flows the staged
    # 128-wide tiles (bf16: u from the operand's hi and lo parts), dE a partial latent tile;
    # then accumulation, whose persistent epilogue adds with one reduction per element
    d = hclt_inputs(40, 100, 17, 45, seed=207)
    rl, rpi, rW, rE = _oracle(d)
    ll, dpi, dW, dE = _gpu_run(d, mode)
    errs = ll_err(ll, rl), flow_err(dpi, rpi), flow_err(dW[1:], rW[1:]), flow_err(dE, rE)
    print(f"hclt 40x100 {mode}: ll {errs[0]:.3e} dpi {errs[1]:.3e} dW {errs[2]:.3e} dE {errs[3]:.3e}")
    assert errs[0] <= LL_TOL[mode]
    assert max(errs[1:]) <= FLOW_TOL[mode]
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("data", "pi", "W", "E")}
    first = [torch.from_numpy(x).cuda() for x in (dpi, dW, dE)]
    _, dpi2, dW2, dE2 = pc.hclt_fwd_bwd(d["parent"], t["data"], t["pi"], t["W"], t["E"], precision=mode,
                                        dpi=first[0].clone(), dW=first[1].clone(), dE=first[2].clone(),
                                        accumulate=True)
    torch.cuda.synchronize()
    for x, y in zip(first, (dpi2, dW2, dE2)):
        torch.testing.assert_close(y, 2 * x, rtol=1e-6, atol=0)


@pytest.mark.parametrize("mode", ["auto", "fp32"])
def test_wide_tiles_ragged(mode):
    # enough edges on the lowest level for the 256-wide persistent element tiles, with H
    # and B off the tile sizes (H = 1000, B = 600): partial row and sample tiles
    d = hclt_inputs(24, 1000, 11, 600, seed=208)
    rl, rpi, rW, rE = _oracle(d)
    ll, dpi, dW, dE = _gpu_run(d, mode)
    errs = ll_err(ll, rl), flow_err(dpi, rpi), flow_err(dW[1:], rW[1:]), flow_err(dE, rE)
    print(f"hclt 24x1000 B600 {mode}: ll {errs[0]:.3e} dpi {errs[1]:.3e} dW {errs[2]:.3e} dE {errs[3]:.3e}")
    assert errs[0] <= LL_TOL[mode]
    assert max(errs[1:]) <= FLOW_TOL[mode]


@pytest.fixture(scope="module")
def hclt_full():
    d = hclt()
    return d, _oracle(d)


@pytest.mark.parametrize("mode", MODES)
def test_hclt_768_every_output(hclt_full, mode):
    # the full workload (767 edges, 256-wide element-flow tiles on the wide levels):
    # every log-likelihood and every flow element against the oracle
    d, (rl, rpi, rW, rE) = hclt_full
    ll, dpi, dW, dE = _gpu_run(d, mode)
    errs = ll_err(ll, rl), flow_err(dpi, rpi), flow_err(dW[1:], rW[1:]), flow_err(dE, rE)
    print(f"hclt 768 B512 {mode}: ll {errs[0]:.3e} dpi {errs[1]:.3e} dW {errs[2]:.3e} dE {errs[3]:.3e}")
    assert errs[0] <= LL_TOL[mode]
    assert max(errs[1:]) <= FLOW_TOL[mode]
    assert np.all(dW[0] == 0)
    B = d["data"].shape[0]
    tol = {"auto": 1e-2, "tf32": 1e-3, "fp32": 1e-5}[mode]
    assert abs(dpi.astype(np.float64).sum() - B) <= tol * B
    np.testing.assert_allclose(dW[1:].astype(np.float64).sum(axis=(1, 2)), B, rtol=tol)
    np.testing.assert_allclose(dE.astype(np.float64).sum(axis=(1, 2)), B, rtol=tol)


@pytest.mark.parametrize("mode", MODES)
def test_hclt_768_uniform_emissions(hclt_full, mode):
    # E = 1/C  =>  LL = -n log C exactly (up to the float32 rows of W and pi); every latent
    # of a node then sits within a rounding step of the node's maximum
    d = dict(hclt_full[0])
    d["E"] = np.full_like(d["E"], 1.0 / 512)
    ll, *_ = _gpu_run(d, mode, flows=False)
    W = d["W"].astype(np.float64)
    pi = d["pi"].astype(np.float64)
    n = len(d["parent"])
    # the float32 rows of W and pi sum to 1 only to ~1e-7; bound their effect on LL
    slack = np.abs(np.log(W[1:].sum(-1))).max(axis=1).sum() + abs(np.log(pi.sum()))
    err = np.abs(ll + n * np.log(512)).max()
    print(f"hclt 768 uniform {mode}: ll err {err:.3e} (slack {slack:.1e})")
    assert err <= LL_TOL[mode] + slack


def test_more_than_1024_latents():
    # H > 1024 takes the block-per-(node, sample) product layer instead of the warp one
    d = hclt_inputs(6, 1100, 7, 9, seed=203, parent=np.array([-1, 0, 0, 1, 1, 2], dtype=np.int32))
    rl, rpi, rW, rE = _oracle(d)
    ll, dpi, dW, dE = _gpu_run(d, "fp32")
    assert ll_err(ll, rl) <= LL_TOL["fp32"]
    assert flow_err(dpi, rpi) <= FLOW_TOL["fp32"]
    assert flow_err(dW[1:], rW[1:]) <= FLOW_TOL["fp32"]
    assert flow_err(dE, rE) <= FLOW_TOL["fp32"]


def test_more_than_1024_categories():
    # C > 1024: 35 category tiles of dE per variable, the last one partial (12 of 32)
    d = hclt_inputs(5, 64, 1100, 20, seed=204, parent=np.array([-1, 0, 0, 1, 2], dtype=np.int32))
    rl, rpi, rW, rE = _oracle(d)
    for mode in ("auto", "fp32"):
        ll, dpi, dW, dE = _gpu_run(d, mode)
        assert ll_err(ll, rl) <= LL_TOL[mode]
        assert max(flow_err(dpi, rpi), flow_err(dW[1:], rW[1:]), flow_err(dE, rE)) <= FLOW_TOL[mode]


@pytest.mark.parametrize("mode", MODES)
def test_prepared_parameters_match_the_plain_call(mode):
    # one prepared buffer serves two batches; every output equals pc_hclt_fwd_bwd's
    # (dpi within float-atomic rounding), and the prepared call matches the oracle
    d = hclt_inputs(40, 130, 17, 45, seed=205)
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("data", "pi", "W", "E")}
    prep = pc.hclt_prepare(d["parent"], t["W"], t["E"], precision=mode)
    rng = np.random.default_rng(206)
    for batch in range(2):
        data = t["data"] if batch == 0 else torch.from_numpy(
            rng.integers(0, 17, size=d["data"].shape, dtype=np.int64).astype(np.int32)).cuda()
        plain = pc.hclt_fwd_bwd(d["parent"], data, t["pi"], t["W"], t["E"], precision=mode)
        fast = pc.hclt_fwd_bwd(d["parent"], data, t["pi"], t["W"], None, precision=mode, prepared=prep)
        torch.cuda.synchronize()
        pc.device_status()
        for i, (a, b) in enumerate(zip(plain, fast)):
            if i == 1:
                torch.testing.assert_close(b, a, rtol=1e-6, atol=0)
            else:
                assert torch.equal(a, b)
        if batch == 0:
            rl, rpi, rW, rE = _oracle(d)
            ll, dpi, dW, dE = (x.cpu().numpy() for x in fast)
            assert ll_err(ll, rl) <= LL_TOL[mode]
            assert max(flow_err(dpi, rpi), flow_err(dW[1:], rW[1:]), flow_err(dE, rE)) <= FLOW_TOL[mode]
