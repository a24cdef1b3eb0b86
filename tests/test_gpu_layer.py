"""GPU parity of the dense sum layer (pc_sum_layer_fwd / pc_sum_layer_bwd through the
C ABI) against the float64 oracle, in every precision mode."""
import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from oracle.sum_layer import sum_layer_fwd, sum_layer_bwd
from tolerances import FLOW_TOL, LL_TOL, MODES, flow_err, out_err
from workloads import layer, layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pc.load()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(d, mode):
    """GPU forward, and GPU backward on the oracle's node values rounded to float32:
    both sides of the backward comparison then get the same inputs (theta, x, out, f)."""
    th, x = _dev(d["theta"]), _dev(d["x"])
    cs = d["child_stride"]
    out = pc.sum_layer_fwd(th, x, child_stride=cs, precision=mode)
    out_in = _dev(_oracle_out(d).astype(np.float32))
    e, F = pc.sum_layer_bwd(th, x, out_in, _dev(d["f"]), child_stride=cs, precision=mode)
    torch.cuda.synchronize()
    pc.device_status()
    return out.cpu().numpy(), e.cpu().numpy(), F.cpu().numpy()


def _oracle_out(d):
    return sum_layer_fwd(d["theta"].astype(np.float64), d["x"].astype(np.float64), d["child_stride"])


def _ref(d):
    th, x = d["theta"].astype(np.float64), d["x"].astype(np.float64)
    out = _oracle_out(d)
    out32 = out.astype(np.float32).astype(np.float64)        # what the GPU backward receives
    e, F = sum_layer_bwd(th, x, d["child_stride"], out32, d["f"].astype(np.float64))
    return out, e, F


@pytest.fixture(scope="module")
def layer_case():
    d = layer()                              # M = N = 1024, batch 128, f = 1
    return d, _ref(d)


@pytest.mark.parametrize("mode", MODES)
def test_single_layer_workload(layer_case, mode):
    d, (ro, re, rF) = layer_case
    out, e, F = _run(d, mode)
    eo, ee, eF = out_err(out, ro), flow_err(e, re), flow_err(F, rF)
    print(f"layer {mode}: out {eo:.3e}  e {ee:.3e}  F {eF:.3e}")
    assert eo <= LL_TOL[mode]
    assert ee <= FLOW_TOL[mode]
    assert eF <= FLOW_TOL[mode]


@pytest.mark.parametrize("mode", MODES)
def test_grouped_ragged(mode):
    # three evenly strided groups; every size off the 128 tile and the K slice
    d = layer_inputs(3, 200, 150, 77, seed=60, child_stride=160, x_scale=5.0, f_kind="uniform")
    ro, re, rF = _ref(d)
    out, e, F = _run(d, mode)
    assert out_err(out, ro) <= LL_TOL[mode]
    assert flow_err(e, re) <= FLOW_TOL[mode]
    assert flow_err(F, rF) <= FLOW_TOL[mode]
    # rows between the groups are nobody's children: untouched (zero)
    assert np.all(e[150:160] == 0) and np.all(e[310:320] == 0)


def test_tiny_and_single_sample():
    for (G, M, N, B) in ((1, 1, 1, 1), (1, 3, 5, 1), (2, 1, 7, 3)):
        d = layer_inputs(G, M, N, B, seed=61, f_kind="uniform")
        ro, re, rF = _ref(d)
        out, e, F = _run(d, "fp32")
        assert out_err(out, ro) <= 1e-5
        assert flow_err(e, re) <= 1e-5 and flow_err(F, rF) <= 1e-5


def test_edge_cases_fp32():
    d = layer_inputs(2, 130, 70, 40, seed=62, child_stride=70, x_scale=3.0, f_kind="uniform")
    x = d["x"].copy()
    x[:70, 5] = -np.inf                       # group 0, sample 5: every child -inf
    x[70:, :] -= 1000.0                       # group 1 lives 1000 nats below group 0
    x[3, 7] = -np.inf                         # one -inf child in a finite column
    th = d["theta"].copy()
    th[0, 11] = 0.0                           # a node with all-zero parameters
    th[1, :, 4] = 0.0                         # a child no node of group 1 uses
    d = dict(d, x=x, theta=th)
    ro, re, rF = _ref(d)
    out, e, F = _run(d, "fp32")
    assert np.all(np.isneginf(out[0, :, 5])) and np.all(np.isneginf(out[0, 11]))
    assert out_err(out, ro) <= 1e-5
    assert np.all(np.isfinite(e)) and np.all(np.isfinite(F))
    assert flow_err(e, re) <= 1e-5 and flow_err(F, rF) <= 1e-5
    assert np.all(e[:70, 5] == 0) and e[3, 7] == 0 and np.all(F[0, 11] == 0)


def test_accumulate_and_optional_outputs():
    d = layer_inputs(1, 256, 192, 64, seed=63, f_kind="uniform")
    th, x, f = _dev(d["theta"]), _dev(d["x"]), _dev(d["f"])
    out = pc.sum_layer_fwd(th, x, precision="fp32")
    e1, F1 = pc.sum_layer_bwd(th, x, out, f, precision="fp32")
    e2, F2 = pc.sum_layer_bwd(th, x, out, f, precision="fp32", e=e1.clone(), F=F1.clone(), accumulate=True)
    torch.testing.assert_close(e2, 2 * e1, rtol=1e-6, atol=0)
    torch.testing.assert_close(F2, 2 * F1, rtol=1e-6, atol=0)
    e3, F3 = pc.sum_layer_bwd(th, x, out, f, precision="fp32", param_flows=False)
    assert F3 is None
    torch.testing.assert_close(e3, e1, rtol=0, atol=0)
    e4, F4 = pc.sum_layer_bwd(th, x, out, f, precision="fp32", element_flows=False)
    assert e4 is None
    torch.testing.assert_close(F4, F1, rtol=0, atol=0)


def test_tf32_downgrade_fails_the_fp32_bar(layer_case):
    # the fp32 bar is tight enough that one-pass TF32 products miss it (pyjuice PR #62,
    # Tests: downgrading either flow kernel's dots to TF32 fails the fp32 test)
    d, (ro, re, rF) = layer_case
    out, e, F = _run(d, "tf32")
    assert out_err(out, ro) > LL_TOL["fp32"]
    assert flow_err(e, re) > FLOW_TOL["fp32"]
    assert flow_err(F, rF) > FLOW_TOL["fp32"]


def test_profiler_reports_contractions():
    d = layer_inputs(1, 512, 256, 128, seed=64)
    th, x = _dev(d["theta"]), _dev(d["x"])
    pc.profile_start(16)
    out = pc.sum_layer_fwd(th, x, precision="auto")
    pc.sum_layer_bwd(th, x, out, _dev(d["f"]), precision="auto")
    rec = pc.profile_stop(16)
    assert [r[0] for r in rec] == ["layer_fwd", "layer_elem", "layer_param"]
    assert all(r[1] > 0 for r in rec) and all(r[2] == 2 * 512 * 256 * 128 for r in rec)
