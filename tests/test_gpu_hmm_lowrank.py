"""GPU parity of the HMM circuit with LowRank exp_sum transitions (pc_hmm_lowrank_fwd_bwd
through the C ABI) against the float64 oracle: every output of ragged cases in every
mode, the 1024-state, 64-position, rank-16, batch-64 workload by sampled
log-likelihoods and the flow totals, accumulation, T = 1 and the refused rank."""
import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from oracle.hmm_lowrank import hmm_lowrank_forward, hmm_lowrank_fwd_bwd
from tolerances import FLOW_TOL, LL_TOL, MODES, flow_err, ll_err
from workloads import hmm_lowrank, hmm_lowrank_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pc.load()


def _grad_err(gpu, ref, mag):
    gpu = np.asarray(gpu, dtype=np.float64)
    if not np.all(np.isfinite(gpu)):
        return np.inf
    scale = mag + 1e-6 * mag.max()
    return float((np.abs(gpu - ref) / scale).max())


def _run(d, mode, **kw):
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("tokens", "pi", "A", "E", "FA", "FB")}
    r = pc.hmm_lowrank_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], t["FA"], t["FB"], precision=mode, **kw)
    torch.cuda.synchronize()
    pc.device_status()
    return {k: v.cpu().numpy() for k, v in r.items()}


@pytest.mark.parametrize("mode", MODES)
def test_ragged_every_output(mode):
    d = hmm_lowrank_inputs(130, 6, 20, 5, 4, 1.0, seed=600)
    r = hmm_lowrank_fwd_bwd(d["pi"], d["A"], d["E"], d["tokens"], d["FA"], d["FB"])
    g = _run(d, mode)
    errs = dict(ll=ll_err(g["ll"], r["ll"]), dpi=flow_err(g["dpi"], r["dpi"]), dA=flow_err(g["dA"], r["dA"]),
                W=flow_err(g["W"], r["W"]), dE=flow_err(g["dE"], r["dE"]),
                dFA=_grad_err(g["dFA"], r["dFA"], r["absdFA"]), dFB=_grad_err(g["dFB"], r["dFB"], r["absdFB"]))
    print(f"hmm-lowrank 130x6 k4 {mode}: " + " ".join(f"{k} {v:.2e}" for k, v in errs.items()))
    assert errs["ll"] <= LL_TOL[mode], errs
    for k in ("dpi", "dA", "W", "dE", "dFA", "dFB"):
        assert errs[k] <= FLOW_TOL[mode], (k, errs)


@pytest.mark.parametrize("mode", MODES)
def test_workload_sampled_and_totals(mode):
    d = hmm_lowrank()
    g = _run(d, mode)
    B, T = d["tokens"].shape
    pick = np.array([3, 40])
    ref, _, _ = hmm_lowrank_forward(d["pi"], d["A"], d["E"], d["tokens"][pick], d["FA"][:, pick], d["FB"][:, pick])
    err = ll_err(g["ll"][pick], ref)
    print(f"hmm-lowrank 1024x64 k16 B64 {mode}: sampled ll err {err:.3e}")
    assert err <= LL_TOL[mode]
    tol = {"auto": 1e-2, "tf32": 1e-3, "fp32": 1e-5}[mode]
    assert abs(g["dpi"].astype(np.float64).sum() - B) <= tol * B
    assert abs(g["dA"].astype(np.float64).sum() - B * (T - 1)) <= tol * B * (T - 1)
    assert abs((d["A"].astype(np.float64) * g["W"]).sum() - B * (T - 1)) <= tol * B * (T - 1)
    counts = np.bincount(d["tokens"].ravel(), minlength=d["E"].shape[1])
    np.testing.assert_allclose(g["dE"].astype(np.float64).sum(0), counts, rtol=tol, atol=tol)


def test_accumulate_doubles_and_t1():
    d = hmm_lowrank_inputs(64, 4, 10, 3, 2, 1.0, seed=601)
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("tokens", "pi", "A", "E", "FA", "FB")}
    r = pc.hmm_lowrank_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], t["FA"], t["FB"], precision="fp32")
    keys = ("dpi", "dA", "W", "dE", "dFA", "dFB")
    r2 = pc.hmm_lowrank_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], t["FA"], t["FB"], precision="fp32",
                                accumulate=True, **{k: r[k].clone() for k in keys})
    torch.cuda.synchronize()
    for k in keys:
        torch.testing.assert_close(r2[k], 2 * r[k], rtol=1e-6, atol=1e-12)
    d1 = hmm_lowrank_inputs(32, 1, 8, 4, 2, 1.0, seed=602)       # one position: no transition layer
    g = _run(d1, "fp32")
    ref = hmm_lowrank_fwd_bwd(d1["pi"], d1["A"], d1["E"], d1["tokens"], d1["FA"], d1["FB"])
    assert ll_err(g["ll"], ref["ll"]) <= LL_TOL["fp32"]
    assert flow_err(g["dE"], ref["dE"]) <= FLOW_TOL["fp32"]


def test_rank_above_the_fused_limit_is_refused():
    d = hmm_lowrank_inputs(16, 3, 4, 2, 65, 1.0, seed=603)
    with pytest.raises(pc.PCError, match="UNSUPPORTED"):
        _run(d, "auto")
