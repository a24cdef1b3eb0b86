"""GPU parity of the whole HMM circuit (pc_hmm_fwd_bwd through the C ABI) against the
float64 oracle: the tiny workload in every mode, ragged and degenerate shapes, the
4096-state workload at batch 128 and 512 (every output), the 1024-state, 64-position
workload at batch 512 (every output), and the uniform-emission closed form."""
import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from oracle.hmm import hmm_fwd_bwd
from tolerances import FLOW_TOL, LL_TOL, MODES, flow_err, ll_err
from workloads import hmm, hmm_1024x64, hmm_inputs, tiny_hmm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pc.load()


def _gpu_run(d, mode, flows=True):
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("tokens", "pi", "A", "E")}
    ll, dpi, dA, dE = pc.hmm_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], precision=mode, flows=flows)
    torch.cuda.synchronize()
    pc.device_status()
    cpu = lambda v: None if v is None else v.cpu().numpy()
    return cpu(ll), cpu(dpi), cpu(dA), cpu(dE)


def _oracle(d):
    return hmm_fwd_bwd(d["pi"], d["A"], d["E"], d["tokens"])


@pytest.fixture(scope="module")
def tiny_case():
    d = tiny_hmm()
    return d, _oracle(d)


@pytest.mark.parametrize("mode", MODES)
def test_tiny_hmm_workload(tiny_case, mode):
    d, (rl, rpi, rA, rE) = tiny_case
    ll, dpi, dA, dE = _gpu_run(d, mode)
    errs = ll_err(ll, rl), flow_err(dpi, rpi), flow_err(dA, rA), flow_err(dE, rE)
    print(f"tiny hmm {mode}: ll {errs[0]:.3e} dpi {errs[1]:.3e} dA {errs[2]:.3e} dE {errs[3]:.3e}")
    assert errs[0] <= LL_TOL[mode]
    assert max(errs[1:]) <= FLOW_TOL[mode]


@pytest.mark.parametrize("mode", ["fp32", "auto"])
@pytest.mark.parametrize("shape", [(300, 5, 37, 45), (129, 3, 5, 130), (16, 2, 4, 1), (40, 1, 6, 9)])
def test_ragged_and_degenerate(shape, mode):
    H, T, V, B = shape
    d = hmm_inputs(H, T, V, B, seed=70 + H)
    rl, rpi, rA, rE = _oracle(d)
    ll, dpi, dA, dE = _gpu_run(d, mode)
    assert ll_err(ll, rl) <= LL_TOL[mode]
    assert flow_err(dpi, rpi) <= FLOW_TOL[mode]
    assert flow_err(dE, rE) <= FLOW_TOL[mode]
    if T >= 2:
        assert flow_err(dA, rA) <= FLOW_TOL[mode]
    else:
        assert np.all(dA == 0)


def test_forward_only_matches_forward_backward():
    d = hmm_inputs(256, 6, 20, 33, seed=80)
    a = _gpu_run(d, "fp32", flows=False)
    b = _gpu_run(d, "fp32", flows=True)
    assert a[1] is None and np.array_equal(a[0], b[0])


def test_accumulate_adds_flows():
    d = hmm_inputs(192, 4, 11, 40, seed=81)
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("tokens", "pi", "A", "E")}
    ll, dpi, dA, dE = pc.hmm_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], precision="fp32")
    ll2, dpi2, dA2, dE2 = pc.hmm_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], precision="fp32",
                                         dpi=dpi.clone(), dA=dA.clone(), dE=dE.clone(), accumulate=True)
    for a, b in ((dpi, dpi2), (dA, dA2), (dE, dE2)):
        torch.testing.assert_close(b, 2 * a, rtol=1e-6, atol=0)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("H", [300, 129])
def test_small_state_space_paths(H, mode):
    # H = 300 or 129 at batch 256: 128 x 64 split-K tiles on the chain (too few wider
    # pairs), and the dA contraction over K ranges (K = 8 x 256 divides into 4 ranges of
    # whole ring blocks); H = 129 leaves H^2 odd for the range sum's scalar path. Then
    # accumulation through the range sum doubles dA.
    d = hmm_inputs(H, 9, 23, 256, seed=90 + H)
    rl, rpi, rA, rE = _oracle(d)
    ll, dpi, dA, dE = _gpu_run(d, mode)
    errs = (ll_err(ll, rl), flow_err(dpi, rpi), flow_err(dA, rA), flow_err(dE, rE))
    print(f"hmm {H}x9 B256 {mode}: ll {errs[0]:.3e} dpi {errs[1]:.3e} dA {errs[2]:.3e} dE {errs[3]:.3e}")
    assert errs[0] <= LL_TOL[mode] and max(errs[1:]) <= FLOW_TOL[mode], errs
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("tokens", "pi", "A", "E")}
    base = torch.from_numpy(dA).cuda()
    _, _, dA2, _ = pc.hmm_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], precision=mode, dA=base.clone(),
                                  accumulate=True)
    torch.cuda.synchronize()
    torch.testing.assert_close(dA2, 2 * base, rtol=1e-6, atol=0)


def test_128_wide_split_tiles():
    # H = 1024, B = 768: 128 x 256 split-K pairs would give 48 CTAs, 128 x 128 pairs 96
    d = hmm_inputs(1024, 4, 19, 768, seed=97)
    rl, rpi, rA, rE = _oracle(d)
    ll, dpi, dA, dE = _gpu_run(d, "auto")
    assert ll_err(ll, rl) <= LL_TOL["auto"]
    assert max(flow_err(dpi, rpi), flow_err(dA, rA), flow_err(dE, rE)) <= FLOW_TOL["auto"]


@pytest.mark.parametrize("mode", ["auto", "fp32"])
def test_small_state_space_ragged_batch(mode):
    # 128 x 64 split-K tiles with a ragged last sample tile (B = 200)
    d = hmm_inputs(256, 4, 17, 200, seed=95)
    rl, rpi, rA, rE = _oracle(d)
    ll, dpi, dA, dE = _gpu_run(d, mode)
    assert ll_err(ll, rl) <= LL_TOL[mode]
    assert max(flow_err(dpi, rpi), flow_err(dA, rA), flow_err(dE, rE)) <= FLOW_TOL[mode]


@pytest.fixture(scope="module")
def hmm128():
    d = hmm(128)
    return d, _oracle(d)


@pytest.mark.parametrize("mode", MODES)
def test_hmm_4096_batch128_every_output(hmm128, mode):
    d, (rl, rpi, rA, rE) = hmm128
    ll, dpi, dA, dE = _gpu_run(d, mode)
    errs = ll_err(ll, rl), flow_err(dpi, rpi), flow_err(dA, rA), flow_err(dE, rE)
    print(f"hmm4096 B128 {mode}: ll {errs[0]:.3e} dpi {errs[1]:.3e} dA {errs[2]:.3e} dE {errs[3]:.3e}")
    assert errs[0] <= LL_TOL[mode]
    assert max(errs[1:]) <= FLOW_TOL[mode]


@pytest.fixture(scope="module")
def hmm1024():
    d = hmm_1024x64()
    return d, _oracle(d)


@pytest.mark.parametrize("mode", MODES)
def test_hmm_1024x64_batch512_every_output(hmm1024, mode):
    d, (rl, rpi, rA, rE) = hmm1024
    ll, dpi, dA, dE = _gpu_run(d, mode)
    errs = ll_err(ll, rl), flow_err(dpi, rpi), flow_err(dA, rA), flow_err(dE, rE)
    print(f"hmm1024x64 B512 {mode}: ll {errs[0]:.3e} dpi {errs[1]:.3e} dA {errs[2]:.3e} dE {errs[3]:.3e}")
    assert errs[0] <= LL_TOL[mode]
    assert max(errs[1:]) <= FLOW_TOL[mode]


@pytest.fixture(scope="module")
def hmm512():
    d = hmm(512)
    return d, _oracle(d)


@pytest.mark.parametrize("mode", MODES)
def test_hmm_4096_batch512_every_output(hmm512, mode):
    # the benchmarked configuration: in auto mode the chains take the 128 x 256 split-K
    # pairs that stage half of the emission block during the exchange
    d, (rl, rpi, rA, rE) = hmm512
    ll, dpi, dA, dE = _gpu_run(d, mode)
    errs = ll_err(ll, rl), flow_err(dpi, rpi), flow_err(dA, rA), flow_err(dE, rE)
    print(f"hmm4096 B512 {mode}: ll {errs[0]:.3e} dpi {errs[1]:.3e} dA {errs[2]:.3e} dE {errs[3]:.3e}")
    assert errs[0] <= LL_TOL[mode]
    assert max(errs[1:]) <= FLOW_TOL[mode]
    # flows are posterior expected counts: their totals are exact at any size
    B, T = d["tokens"].shape
    tol = {"auto": 1e-2, "tf32": 1e-3, "fp32": 1e-5}[mode]
    assert abs(dpi.astype(np.float64).sum() - B) <= tol * B
    assert abs(dA.astype(np.float64).sum() - B * (T - 1)) <= tol * B * (T - 1)
    counts = np.bincount(d["tokens"].ravel(), minlength=d["E"].shape[1])
    np.testing.assert_allclose(dE.astype(np.float64).sum(0), counts, rtol=tol, atol=tol)


@pytest.mark.parametrize("mode", MODES)
def test_uniform_emissions_closed_form(mode):
    # E = 1/V  =>  LL = -T log V exactly; 1/1024 is exact in bf16 and TF32 too
    d = dict(hmm(512))
    d["E"] = np.full_like(d["E"], 1.0 / 1024)
    ll, *_ = _gpu_run(d, mode, flows=False)
    A = d["A"].astype(np.float64)
    # rows of the float32 A sum to 1 only to ~1e-7: the exact LL is then -T log V plus
    # the log of the row sums along the path, bounded by T * max|log rowsum|
    slack = 32 * np.abs(np.log(A.sum(1))).max()
    assert np.abs(ll + 32 * np.log(1024)).max() <= LL_TOL[mode] + slack
