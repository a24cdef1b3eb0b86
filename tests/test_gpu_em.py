"""GPU parity of the EM M-step (pc_em_normalize through the C ABI) against the float64
oracle (oracle/em.py): the shapes of the HMM and LowRank workloads' parameters, ragged
and unaligned rows, rows without flow, zero denominators, and one whole Baum-Welch step
of the tiny HMM (GPU flows, GPU M-step) against the oracle's."""
import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from oracle.em import em_conditional, em_plain, hmm_em_step
from workloads import tiny_hmm

pytestmark = pytest.mark.gpu

REL = 1e-5  # float32 row sums and divisions against float64


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pc.load()


def _stats(shape, seed, zero_rows=0, zero_frac=0.0):
    rng = np.random.default_rng(seed)
    F = rng.gamma(0.5, 1.0, size=shape).astype(np.float32)
    if zero_frac:
        F[rng.random(shape) < zero_frac] = 0.0
    rows = F.reshape(-1, shape[-1])
    if zero_rows:
        rows[rng.choice(rows.shape[0], size=zero_rows, replace=False)] = 0.0
    theta = rng.random(shape).astype(np.float32)
    return F, theta


def _gpu(F, theta, W=None):
    t = torch.from_numpy(theta).cuda()
    pc.em_normalize(torch.from_numpy(F).cuda(), t, None if W is None else torch.from_numpy(W).cuda())
    torch.cuda.synchronize()
    return t.cpu().numpy()


@pytest.mark.parametrize("shape", [(1, 4096), (4096, 4096), (4096, 1024), (3, 5, 1000), (7, 7), (2, 1), (9, 4099)])
def test_plain_normalize(shape):
    F, theta = _stats(shape, seed=sum(shape), zero_rows=1 if len(shape) > 1 and shape[-2] > 1 else 0,
                      zero_frac=0.2)
    got = _gpu(F, theta)
    ref = em_plain(F, theta)
    np.testing.assert_allclose(got, ref, rtol=REL, atol=0)


@pytest.mark.parametrize("shape", [(1024, 1024), (5, 333), (64, 12)])
def test_conditional_normalize(shape):
    F, theta = _stats(shape, seed=7 + shape[0], zero_rows=1, zero_frac=0.1)
    rng = np.random.default_rng(shape[1])
    W = rng.gamma(2.0, 1.0, size=shape).astype(np.float32)
    W[rng.random(shape) < 0.05] = 0.0
    got = _gpu(F, theta, W)
    ref = em_conditional(F, W, theta)
    np.testing.assert_allclose(got, ref, rtol=REL, atol=0)


def test_rows_without_flow_keep_their_parameters():
    F = np.zeros((4, 8), np.float32)
    F[1, 3] = 2.0
    theta = np.arange(32, dtype=np.float32).reshape(4, 8) / 100
    got = _gpu(F, theta)
    np.testing.assert_array_equal(got[[0, 2, 3]], theta[[0, 2, 3]])
    np.testing.assert_array_equal(got[1], np.eye(8, dtype=np.float32)[3])


def test_baum_welch_step_of_the_tiny_hmm():
    d = tiny_hmm()
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("tokens", "pi", "A", "E")}
    _, dpi, dA, dE = pc.hmm_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], precision="fp32")
    new = [x.clone() for x in (t["pi"], t["A"], t["E"])]
    for flows, th in zip((dpi, dA, dE), new):
        pc.em_normalize(flows.reshape(th.shape).contiguous(), th)
    torch.cuda.synchronize()
    ref = hmm_em_step(d["pi"], d["A"], d["E"], d["tokens"])
    for got, r in zip(new, ref):
        np.testing.assert_allclose(got.cpu().numpy(), r, rtol=5e-5, atol=1e-7)
