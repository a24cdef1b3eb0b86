"""GPU parity of the HMM circuit on inputs at the edges of its numerical range, against
the float64 oracle (which works in log space and has no range limit):

* peaked emissions (rows of E a softmax of N(0, 10^2) logits: probabilities spread over
  tens of nats), in every mode. One path then carries nearly all of a sample's mass, so
  the operand roundings of the T - 1 chained layers do not average out: a flow's error
  is bounded by two roundings per layer, 2 (T - 1) u with u the mode's unit roundoff
  (2^-8 bf16, 2^-11 TF32); the flows are held to that where it exceeds the random-data
  bars (tolerances.FLOW_TOL), the log-likelihood to the stated bars;
* exact zeros in A and in E (half of A's entries, a third of E's), so that states are
  unreachable and tokens impossible for some states, in every mode;
* a token that every state emits with probability ~1e-30, and one with denormal
  probability ~1e-40 (scaled into range by the layer's shift before it is multiplied);
* a constructed HMM whose per-layer bound is looser than e^-55 for some samples: those
  samples are flagged (ll NaN, no flow, PC_ERR_RANGE from pc_device_status) while the
  others stay exact, and the same HMM with a milder gap is exact everywhere.
"""
import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from oracle.hmm import hmm_fwd_bwd
from tolerances import FLOW_TOL, LL_TOL, MODES, flow_err, ll_err
from workloads import hmm_edge_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pc.load()
    pc.device_status()


def _gpu_run(d, mode):
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("tokens", "pi", "A", "E")}
    ll, dpi, dA, dE = pc.hmm_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], precision=mode)
    torch.cuda.synchronize()
    return ll.cpu().numpy(), dpi.cpu().numpy(), dA.cpu().numpy(), dE.cpu().numpy()


UNIT_ROUNDOFF = {"auto": 2.0 ** -8, "tf32": 2.0 ** -11, "fp32": 0.0}


def _check(d, mode, label, flow_tol=None):
    rl, rpi, rA, rE = hmm_fwd_bwd(d["pi"], d["A"], d["E"], d["tokens"])
    ll, dpi, dA, dE = _gpu_run(d, mode)
    pc.device_status()
    errs = ll_err(ll, rl), flow_err(dpi, rpi), flow_err(dA, rA), flow_err(dE, rE)
    print(f"{label} {mode}: ll {errs[0]:.3e} dpi {errs[1]:.3e} dA {errs[2]:.3e} dE {errs[3]:.3e}")
    assert errs[0] <= LL_TOL[mode]
    assert max(errs[1:]) <= (FLOW_TOL[mode] if flow_tol is None else flow_tol)


@pytest.mark.parametrize("mode", MODES)
def test_peaked_emissions(mode):
    d = hmm_edge_inputs(300, 9, 40, 96, seed=500, e_scale=10.0)
    T = d["tokens"].shape[1]
    path_bound = 2 * (T - 1) * UNIT_ROUNDOFF[mode]
    _check(d, mode, "peaked E", flow_tol=max(FLOW_TOL[mode], path_bound))


@pytest.mark.parametrize("mode", MODES)
def test_zeros_in_transitions_and_emissions(mode):
    _check(hmm_edge_inputs(260, 7, 33, 80, seed=501, zero_A=0.5, zero_E=1 / 3), mode, "zeros in A, E")


@pytest.mark.parametrize("mode", ["auto", "fp32"])
def test_token_with_tiny_and_denormal_emissions(mode):
    d = hmm_edge_inputs(200, 6, 20, 64, seed=502)
    E = d["E"].astype(np.float64)
    rng = np.random.default_rng(503)
    E[:, 3] = 1e-30 * rng.uniform(0.5, 1.0, size=E.shape[0])
    E[:, 7] = 1e-40 * rng.uniform(0.5, 1.0, size=E.shape[0])  # float32 denormals
    d["E"] = E.astype(np.float32)
    tok = d["tokens"].copy()
    tok[::3, 2] = 3
    tok[1::4, 4] = 7
    tok[::5, 5] = 7  # the last position (the leaf) too
    d["tokens"] = tok
    _check(d, mode, "tiny emissions")


def _gap_hmm(H, eps):
    # states 0 and 1 swap (A), state 0 emits tokens 0 and 1, state 1 emits token 0 with
    # probability eps only; token 2 is emitted by both. After x_1 = 1 only state 0 is
    # possible, so at position 0 the bound max_k E[k,0] sum_l A[k,l] = 1 overestimates
    # the largest value eps. Further states (H > 2) are unreachable and emit nothing.
    pi = np.zeros(H); pi[:2] = 0.5
    A = np.zeros((H, H)); A[0, 1] = A[1, 0] = 1.0
    for k in range(2, H):
        A[k, k] = 1.0
    E = np.zeros((H, 3)); E[0] = [1.0, 1.0, 0.5]; E[1] = [eps, 0.0, 0.5]
    tokens = np.array([[0, 1], [1, 1], [0, 0], [1, 0], [2, 2], [2, 0]], dtype=np.int32)
    f = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    return dict(pi=f(pi), A=f(A), E=f(E), tokens=tokens)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("H", [2, 130])
def test_gap_within_range_is_exact(H, mode):
    _check(_gap_hmm(H, 1e-20), mode, f"gap 1e-20 H={H}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("H", [2, 130])
def test_gap_beyond_range_is_flagged(H, mode):
    d = _gap_hmm(H, 1e-30)
    ll, dpi, dA, dE = _gpu_run(d, mode)
    with pytest.raises(pc.PCError) as ei:
        pc.device_status()
    assert ei.value.status == 9, ei.value  # PC_ERR_RANGE
    pc.device_status()  # the read cleared it
    flagged = np.array([True, False, True, True, False, False])
    assert np.isnan(ll[flagged]).all()
    # the other samples are exact; the flagged ones pass no flow
    rest = dict(d, tokens=d["tokens"][~flagged])
    rl, rpi, rA, rE = hmm_fwd_bwd(rest["pi"], rest["A"], rest["E"], rest["tokens"])
    assert ll_err(ll[~flagged], rl) <= LL_TOL[mode]
    assert np.isneginf(ll[1])
    assert max(flow_err(dpi, rpi), flow_err(dA, rA), flow_err(dE, rE)) <= FLOW_TOL[mode]
