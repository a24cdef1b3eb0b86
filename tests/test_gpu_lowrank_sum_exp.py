"""GPU parity of the LowRank sum_exp layer (pc_lowrank_sum_exp_fwd / _bwd through the C
ABI) against the float64 oracle: ragged shapes over several tiles, ranks 1 .. 100, the
1024 x 1024 rank-16 batch-64 workload's factors at spreads 0.3, 1 and 4 in every mode,
B = 0 (a scale constant along the children) against the plain sum layer, accumulation,
partial outputs and the edge cases."""
import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from oracle.lowrank import lowrank_sum_exp_bwd
from oracle.sum_layer import sum_layer_fwd
from tolerances import FLOW_TOL, LL_TOL, MODES, flow_err, out_err
from workloads import lowrank, lowrank_inputs

pytestmark = pytest.mark.gpu

# TF32 flows of this form pass through two TF32 contractions in a row (the forward's P|Q,
# whose num and Z' make the node factors a s and a t, then the flow contraction): four
# operands rounded to nearest TF32, each within 2^-11 relative, bound an entry's error by
# 4 * 2^-11 = 1.95e-3 when the flow contraction is too short to average (rank 1, batch 2).
SE_FLOW_TOL = dict(FLOW_TOL, tf32=2e-3)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pc.load()


def _cuda(d):
    return {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("theta", "A", "Bm", "x", "f")}


def _grad_err(gpu, ref, mag):
    """Largest |gpu - ref| relative to the entry's sum of absolute terms before cancellation."""
    gpu = np.asarray(gpu, dtype=np.float64)
    if not np.all(np.isfinite(gpu)):
        return np.inf
    scale = mag + 1e-6 * mag.max()
    return float((np.abs(gpu - ref) / scale).max())


def _run(d, mode):
    t = _cuda(d)
    out, logZ = pc.lowrank_sum_exp_fwd(t["theta"], t["A"], t["Bm"], t["x"], precision=mode)
    g = pc.lowrank_sum_exp_bwd(t["theta"], t["A"], t["Bm"], t["x"], t["f"], precision=mode)
    torch.cuda.synchronize()
    pc.device_status()
    return out.cpu().numpy(), logZ.cpu().numpy(), {k: v.cpu().numpy() for k, v in g.items()}


def _errors(d, r, mode):
    out, logZ, g = _run(d, mode)
    return dict(out=out_err(out, r["out"]), logZ=out_err(logZ, r["logZ"]),
                dA=_grad_err(g["dA"], r["dA"], r["absdA"]), dB=_grad_err(g["dB"], r["dB"], r["absdB"]),
                e=flow_err(g["e"], r["e"]), Fplus=flow_err(g["Fplus"], r["Fplus"]), W=flow_err(g["W"], r["W"]))


def _check(errs, mode):
    assert errs["out"] <= LL_TOL[mode] and errs["logZ"] <= LL_TOL[mode], errs
    for k in ("dA", "dB", "e", "Fplus", "W"):
        assert errs[k] <= SE_FLOW_TOL[mode], (k, errs)


def _oracle(d):
    return lowrank_sum_exp_bwd(d["theta"], d["A"], d["Bm"], d["x"], d["f"])


@pytest.mark.parametrize("mode", MODES)
def test_ragged_tiles(mode):
    d = lowrank_inputs(200, 77, 5, 3, 1.0, seed=400, f_kind="uniform")
    errs = _errors(d, _oracle(d), mode)
    print(f"sum_exp 200x77 k5 {mode}: " + " ".join(f"{k} {v:.2e}" for k, v in errs.items()))
    _check(errs, mode)


@pytest.mark.parametrize("K", [1, 16, 17, 64, 100])
def test_ranks(K):
    d = lowrank_inputs(130, 100, K, 2, 1.0, seed=401 + K, f_kind="uniform")
    r = _oracle(d)
    for mode in MODES:
        _check(_errors(d, r, mode), mode)


@pytest.fixture(scope="module", params=[0.3, 1.0, 4.0])
def workload(request):
    d = lowrank(request.param)
    return request.param, d, _oracle(d)


def test_lowrank_sum_exp_1024_rank16_b64(workload):
    spread, d, r = workload
    for mode in MODES:
        errs = _errors(d, r, mode)
        print(f"sum_exp 1024 spread {spread} {mode}: " + " ".join(f"{k} {v:.2e}" for k, v in errs.items()))
        _check(errs, mode)


def test_scale_constant_along_children_is_the_sum_layer():
    d = lowrank_inputs(150, 140, 8, 4, 1.0, seed=410)
    d["Bm"] = np.zeros_like(d["Bm"])
    out, logZ, g = _run(d, "fp32")
    ref = sum_layer_fwd(d["theta"].astype(np.float64)[None], d["x"].astype(np.float64))[0]
    assert out_err(out, ref) <= LL_TOL["fp32"]
    r = _oracle(d)
    assert _grad_err(g["dB"], r["dB"], r["absdB"]) <= FLOW_TOL["fp32"]


def test_accumulate_and_partial_outputs():
    d = lowrank_inputs(64, 96, 4, 3, 1.0, seed=411, f_kind="uniform")
    t = _cuda(d)
    g = pc.lowrank_sum_exp_bwd(t["theta"], t["A"], t["Bm"], t["x"], t["f"], precision="fp32")
    g2 = pc.lowrank_sum_exp_bwd(t["theta"], t["A"], t["Bm"], t["x"], t["f"], precision="fp32",
                                **{k: v.clone() for k, v in g.items()}, accumulate=True)
    for k in g:
        torch.testing.assert_close(g2[k], 2 * g[k], rtol=1e-6, atol=0)
    s = pc.lowrank_sum_exp_bwd(t["theta"], t["A"], t["Bm"], t["x"], t["f"], precision="fp32", grads=False,
                               element_flows=False)
    assert s["dA"] is None and s["e"] is None
    assert torch.equal(s["Fplus"], g["Fplus"]) and torch.equal(s["W"], g["W"])
    q = pc.lowrank_sum_exp_bwd(t["theta"], t["A"], t["Bm"], t["x"], t["f"], precision="fp32", param_flows=False,
                               z_correction=False)
    assert torch.equal(q["dA"], g["dA"]) and torch.equal(q["dB"], g["dB"]) and torch.equal(q["e"], g["e"])


def test_edge_cases():
    d = lowrank_inputs(40, 30, 4, 2, 1.0, seed=412)
    t = _cuda(d)
    e0 = {k: v[..., :0] if k in ("x", "f") else v for k, v in t.items()}
    e0["A"], e0["Bm"] = t["A"][:0], t["Bm"][:0]
    out, logZ = pc.lowrank_sum_exp_fwd(e0["theta"], e0["A"], e0["Bm"], e0["x"].contiguous())
    assert out.shape == (40, 0) and logZ.shape == (0, 40)
    with pytest.raises(pc.PCError, match="SHAPE"):
        pc.lowrank_sum_exp_fwd(t["theta"], t["A"][:, :, :0].contiguous(), t["Bm"][:, :0].contiguous(), t["x"])
    with pytest.raises(pc.PCError, match="UNKNOWN_PRECISION"):
        pc.lowrank_sum_exp_fwd(t["theta"], t["A"], t["Bm"], t["x"], precision=7)
    # a sample whose children are all -inf: out = -inf, no flow
    d2 = lowrank_inputs(20, 24, 3, 2, 1.0, seed=413)
    d2["x"][:, 1] = -np.inf
    out, logZ, g = _run(d2, "fp32")
    assert np.all(np.isneginf(out[:, 1])) and np.all(np.isfinite(out[:, 0]))
    assert np.all(g["e"][:, 1] == 0) and np.all(g["dA"][1] == 0) and np.all(g["dB"][1] == 0)


@pytest.mark.parametrize("spread", [0.3, 1.0, 4.0])
def test_fp8_flow_products(spread):
    # F+ and W are sums of positive terms, each the product of two operands rounded to e4m3
    # (3 mantissa bits: within 2^-4 relative), so every entry is within 2 * 2^-4 (+ float32
    # rounding) of the exact sum; the gradients and element flows do not change.
    d = lowrank(spread)
    r = _oracle(d)
    t = _cuda(d)
    g = pc.lowrank_sum_exp_bwd(t["theta"], t["A"], t["Bm"], t["x"], t["f"], precision="auto")
    q = pc.lowrank_sum_exp_bwd(t["theta"], t["A"], t["Bm"], t["x"], t["f"], precision="auto", flow_precision="fp8")
    torch.cuda.synchronize()
    pc.device_status()
    for k in ("dA", "dB", "e"):
        assert torch.equal(q[k], g[k]), k
    rel = {}
    for k in ("Fplus", "W"):
        ref = r[k]
        got = q[k].cpu().numpy().astype(np.float64)
        rel[k] = np.abs(got - ref) / np.abs(ref)
        assert rel[k].max() <= 2 * 2.0 ** -4 * (1 + 1e-3), (k, rel[k].max())
    th = d["theta"].astype(np.float64)
    ratio = (q["Fplus"].cpu().numpy() / (th * q["W"].cpu().numpy())) / (r["Fplus"] / (th * r["W"]))
    print(f"fp8 flows spread {spread}: F+ median {np.median(rel['Fplus']):.2e} max {rel['Fplus'].max():.2e}; "
          f"W median {np.median(rel['W']):.2e} max {rel['W'].max():.2e}; F+/F- median "
          f"{np.median(np.abs(ratio - 1)):.2e} max {np.abs(ratio - 1).max():.2e}")
