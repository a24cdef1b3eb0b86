"""Failure detection on the GPU without a fault: device-side waits that run out.

Every wait in the library's kernels is bounded. The tensor-core contraction's first
waits (a free ring slot, a filled slot, a free or complete accumulator) take a limit
set from the host (pc_set_wait_limit_ns). With a 1 ns limit each such wait that does
not succeed at once gives up: the kernel records PC_ERR_TIMEOUT in the device status
word, waits (on the default limit) for the copies and MMAs it has already issued, frees
its tensor memory and exits. Nothing faults and nothing hangs.

Each case checks that the timeout is reported, that reading the status clears it, and
that, with the default limit restored, the same call on the same stream matches the
oracle. The cases cover an unsliced contraction (a long-K layer forward in bf16), the
sliced 3xTF32 accumulation, and the HMM chain's split-K CTA pairs, whose clusters meet
at barriers whatever a wait decided.
"""
import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from oracle.hmm import hmm_fwd_bwd
from oracle.sum_layer import sum_layer_fwd
from tolerances import LL_TOL, flow_err, FLOW_TOL, ll_err, out_err
from workloads import hmm_inputs, layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pc.load()
    pc.device_status()  # start from a clear status word
    yield
    pc.set_wait_limit_ns(0)


def _expect_timeout(run):
    pc.set_wait_limit_ns(1)
    try:
        run()
        torch.cuda.synchronize()
    finally:
        pc.set_wait_limit_ns(0)
    with pytest.raises(pc.PCError) as ei:
        pc.device_status()
    assert ei.value.status == 8, ei.value  # PC_ERR_TIMEOUT
    pc.device_status()  # the read cleared it
    torch.cuda.synchronize()  # the context is still usable


@pytest.mark.parametrize("mode", ["auto", "fp32"])
def test_layer_wait_runs_out_then_recovers(mode):
    # 65536 children: the epilogue's wait for its accumulator spans a K loop of at
    # least 128 ring blocks, far beyond the limit
    d = layer_inputs(1, 256, 65536, 64, seed=400)
    theta = torch.from_numpy(d["theta"]).cuda()
    x = torch.from_numpy(d["x"]).cuda()
    _expect_timeout(lambda: pc.sum_layer_fwd(theta, x, precision=mode))
    out = pc.sum_layer_fwd(theta, x, precision=mode)
    torch.cuda.synchronize()
    pc.device_status()
    ref = sum_layer_fwd(d["theta"], d["x"])
    assert out_err(out.cpu().numpy(), ref) <= LL_TOL[mode]


def test_hmm_split_pairs_wait_runs_out_then_recovers():
    # bf16 chain on 2-CTA clusters (split-K pairs) plus the stacked dA contraction
    d = hmm_inputs(1024, 4, 16, 512, seed=401)
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("tokens", "pi", "A", "E")}
    _expect_timeout(lambda: pc.hmm_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], precision="auto"))
    ll, dpi, dA, dE = pc.hmm_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], precision="auto")
    torch.cuda.synchronize()
    pc.device_status()
    rl, rpi, rA, rE = hmm_fwd_bwd(d["pi"], d["A"], d["E"], d["tokens"])
    assert ll_err(ll.cpu().numpy(), rl) <= LL_TOL["auto"]
    assert max(flow_err(dpi.cpu().numpy(), rpi), flow_err(dA.cpu().numpy(), rA),
               flow_err(dE.cpu().numpy(), rE)) <= FLOW_TOL["auto"]
