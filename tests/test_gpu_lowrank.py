"""GPU parity of the LowRank exp_sum layer (pc_lowrank_exp_sum_fwd / _bwd through the C
ABI) against the float64 oracle: ragged shapes over several tiles, ranks 1 .. 64, the
1024 x 1024 rank-16 batch-64 workload at scale spreads 0.3, 1 and 4 nats in every mode,
the zero-scale reduction to the plain sum layer, accumulation and the edge cases."""
import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from oracle.lowrank import lowrank_exp_sum_bwd
from oracle.sum_layer import sum_layer_fwd
from tolerances import FLOW_TOL, LL_TOL, MODES, flow_err, out_err
from workloads import lowrank, lowrank_inputs

pytestmark = pytest.mark.gpu


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
    out, logZ = pc.lowrank_exp_sum_fwd(t["theta"], t["A"], t["Bm"], t["x"], precision=mode)
    g = pc.lowrank_exp_sum_bwd(t["theta"], t["A"], t["Bm"], t["x"], out, logZ, t["f"], precision=mode)
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
        assert errs[k] <= FLOW_TOL[mode], (k, errs)


def _oracle(d):
    return lowrank_exp_sum_bwd(d["theta"], d["A"], d["Bm"], d["x"], d["f"])


@pytest.mark.parametrize("mode", MODES)
def test_ragged_tiles(mode):
    d = lowrank_inputs(200, 77, 5, 3, 1.0, seed=300, f_kind="uniform")
    errs = _errors(d, _oracle(d), mode)
    print(f"lowrank 200x77 k5 {mode}: " + " ".join(f"{k} {v:.2e}" for k, v in errs.items()))
    _check(errs, mode)


# Ranks 1 .. 64 at a 1-nat spread. (At 4 nats and rank 64 the entries of S reach ~20 nats,
# and the accumulator's truncation over 8 TF32 k-steps moves exp(S) by ~1e-5 relative in
# fp32 mode: the spread-4 case is covered at the workload's rank 16 below.)
# (16 and 32 in bf16, 8 and 16 in TF32 take the operand layout with hi and lo in one row)
@pytest.mark.parametrize("K", [1, 8, 16, 17, 32, 40, 64])
def test_ranks(K):
    d = lowrank_inputs(130, 100, K, 2, 1.0, seed=301 + K, f_kind="uniform")
    r = _oracle(d)
    for mode in MODES:
        _check(_errors(d, r, mode), mode)


@pytest.fixture(scope="module", params=[0.3, 1.0, 4.0])
def workload(request):
    d = lowrank(request.param)
    return request.param, d, _oracle(d)


def test_lowrank_1024_rank16_b64(workload):
    spread, d, r = workload
    for mode in MODES:
        errs = _errors(d, r, mode)
        print(f"lowrank 1024 spread {spread} {mode}: " + " ".join(f"{k} {v:.2e}" for k, v in errs.items()))
        _check(errs, mode)


def test_zero_scale_is_the_sum_layer():
    d = lowrank_inputs(150, 140, 8, 4, 1.0, seed=310)
    d["A"] = np.zeros_like(d["A"])
    out, logZ, g = _run(d, "fp32")
    ref = sum_layer_fwd(d["theta"].astype(np.float64)[None], d["x"].astype(np.float64))[0]
    assert out_err(out, ref) <= LL_TOL["fp32"]
    assert np.all(g["dB"] == 0)
    np.testing.assert_allclose(logZ, np.log(d["theta"].astype(np.float64).sum(1))[None, :].repeat(4, 0),
                               atol=1e-6)


def test_accumulate_and_partial_outputs():
    d = lowrank_inputs(64, 96, 4, 3, 1.0, seed=311, f_kind="uniform")
    t = _cuda(d)
    out, logZ = pc.lowrank_exp_sum_fwd(t["theta"], t["A"], t["Bm"], t["x"], precision="fp32")
    g = pc.lowrank_exp_sum_bwd(t["theta"], t["A"], t["Bm"], t["x"], out, logZ, t["f"], precision="fp32")
    g2 = pc.lowrank_exp_sum_bwd(t["theta"], t["A"], t["Bm"], t["x"], out, logZ, t["f"], precision="fp32",
                                **{k: v.clone() for k, v in g.items()}, accumulate=True)
    for k in g:
        torch.testing.assert_close(g2[k], 2 * g[k], rtol=1e-6, atol=0)
    # only the statistics, only the gradients: the same values
    s = pc.lowrank_exp_sum_bwd(t["theta"], t["A"], t["Bm"], t["x"], out, logZ, t["f"], precision="fp32",
                               grads=False, element_flows=False)
    assert s["dA"] is None and s["e"] is None
    assert torch.equal(s["Fplus"], g["Fplus"]) and torch.equal(s["W"], g["W"])
    q = pc.lowrank_exp_sum_bwd(t["theta"], t["A"], t["Bm"], t["x"], out, logZ, t["f"], precision="fp32",
                               param_flows=False, z_correction=False)
    assert torch.equal(q["dA"], g["dA"]) and torch.equal(q["dB"], g["dB"]) and torch.equal(q["e"], g["e"])


def test_edge_cases():
    d = lowrank_inputs(40, 30, 4, 2, 1.0, seed=312)
    t = _cuda(d)
    # an empty batch and no nodes: nothing to do
    e0 = {k: v[..., :0] if k in ("x", "f") else v for k, v in t.items()}
    e0["A"], e0["Bm"] = t["A"][:0], t["Bm"][:0]
    out, logZ = pc.lowrank_exp_sum_fwd(e0["theta"], e0["A"], e0["Bm"], e0["x"].contiguous())
    assert out.shape == (40, 0) and logZ.shape == (0, 40)
    # rank above the fused kernels' limit, and rank 0
    big = lowrank_inputs(8, 8, 65, 1, 1.0, seed=313)
    tb = _cuda(big)
    with pytest.raises(pc.PCError, match="UNSUPPORTED"):
        pc.lowrank_exp_sum_fwd(tb["theta"], tb["A"], tb["Bm"], tb["x"])
    with pytest.raises(pc.PCError, match="SHAPE"):
        pc.lowrank_exp_sum_fwd(t["theta"], t["A"][:, :, :0].contiguous(), t["Bm"][:, :0].contiguous(), t["x"])
    with pytest.raises(pc.PCError, match="UNKNOWN_PRECISION"):
        pc.lowrank_exp_sum_fwd(t["theta"], t["A"], t["Bm"], t["x"], precision=7)


def test_theta_alignment_paths_agree():
    # theta's own rows feed the passes' tensor maps when they are 16-byte aligned (N % 4
    # == 0), through a padded copy otherwise: a theta stored 4 bytes off alignment takes
    # the copy, and every output keeps the same bits
    d = lowrank_inputs(130, 100, 16, 3, 1.0, seed=320, f_kind="uniform")
    t = _cuda(d)
    buf = torch.empty(t["theta"].numel() + 1, dtype=torch.float32, device="cuda")
    shifted = buf[1:].view(t["theta"].shape)
    shifted.copy_(t["theta"])
    assert shifted.data_ptr() % 16 != 0 and t["theta"].data_ptr() % 16 == 0
    for mode in MODES:
        res = []
        for th in (t["theta"], shifted):
            out, logZ = pc.lowrank_exp_sum_fwd(th, t["A"], t["Bm"], t["x"], precision=mode)
            g = pc.lowrank_exp_sum_bwd(th, t["A"], t["Bm"], t["x"], out, logZ, t["f"], precision=mode)
            res.append((out, logZ, g))
        torch.cuda.synchronize()
        pc.device_status()
        (o1, z1, g1), (o2, z2, g2) = res
        assert torch.equal(o1, o2) and torch.equal(z1, z2), mode
        for k in g1:
            assert torch.equal(g1[k], g2[k]), (mode, k)
