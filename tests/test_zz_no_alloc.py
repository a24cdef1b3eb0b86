"""pc_sum_layer_fwd_noalloc: the sum-layer forward for callers that cannot allocate
device memory (a plugin whose host framework owns all device memory and gives it no
allocator, or a hot path where an allocation is not allowed). It uses a 16 MiB scratch
array built into the library instead of a caller workspace.

Checked through the C ABI on calls in a row that share that scratch:
* the same kernels on the same inputs as pc_sum_layer_fwd (the workspace entry point),
  so the outputs must be bit-identical;
* a small call right after a larger one whose NaN inputs left NaN operands all over the
  scratch: a read of anything the small call did not write itself would show;
* one case against the float64 oracle at the per-mode bar;
and an oversize request must be refused before any launch. This file is collected last
on purpose: it must pass both alone in a fresh process and after every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from log_space_sum_gb300 import _native as N
from oracle.sum_layer import sum_layer_fwd
from tolerances import LL_TOL, MODES, out_err
from workloads import layer_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


def _noalloc(lib, theta, x, cs, out, mode):
    G, M, Nn = theta.shape
    B = x.shape[1]
    return lib.pc_sum_layer_fwd_noalloc(G, M, Nn, B, C.c_void_p(theta.data_ptr()), C.c_void_p(x.data_ptr()),
                                        cs, C.c_void_p(out.data_ptr()), pc.precision_code(mode),
                                        C.c_void_p(torch.cuda.current_stream().cuda_stream))


def _run_both(lib, d, mode):
    theta = torch.from_numpy(d["theta"]).cuda()
    x = torch.from_numpy(d["x"]).cuda()
    cs = d["child_stride"]
    nb = C.c_size_t(0)
    G, M, Nn = theta.shape
    assert lib.pc_sum_layer_workspace(G, M, Nn, x.shape[1], pc.precision_code(mode), C.byref(nb)) == 0
    assert nb.value <= SCRATCH_BYTES
    ref = pc.sum_layer_fwd(theta, x, child_stride=cs, precision=mode)
    out = torch.full_like(ref, float("nan"))
    assert _noalloc(lib, theta, x, cs, out, mode) == 0, lib.pc_last_error().decode()
    torch.cuda.synchronize()
    pc.device_status()
    return out, ref


@pytest.mark.parametrize("mode", MODES)
def test_noalloc_matches_workspace_entry_point(mode):
    assert torch.cuda.is_available(), "GPU test"
    lib = pc.load()
    # two calls in a row, different shapes and data, the second with strided groups
    for d in (layer_inputs(1, 640, 384, 96, seed=300), layer_inputs(3, 130, 200, 40, seed=301, child_stride=210)):
        out, ref = _run_both(lib, d, mode)
        assert torch.equal(out, ref), "the built-in scratch changed the result"
    # against the oracle, on the last case
    assert out_err(out.cpu().numpy(), sum_layer_fwd(d["theta"], d["x"], d["child_stride"])) <= LL_TOL[mode]


@pytest.mark.parametrize("mode", MODES)
def test_noalloc_after_a_larger_call_full_of_nan(mode):
    lib = pc.load()
    big = layer_inputs(1, 1024, 1024, 128, seed=302)
    big["theta"] = np.full_like(big["theta"], np.nan)  # NaN operands and partial sums all over the scratch
    out, _ = _run_both(lib, big, mode)
    assert not torch.isfinite(out).any()
    d = layer_inputs(2, 70, 90, 33, seed=303, child_stride=100)
    out, ref = _run_both(lib, d, mode)
    assert not torch.isnan(out).any()
    assert torch.equal(out, ref)
    assert out_err(out.cpu().numpy(), sum_layer_fwd(d["theta"], d["x"], d["child_stride"])) <= LL_TOL[mode]


def test_noalloc_refuses_requests_beyond_its_scratch():
    lib = pc.load()
    fake = C.c_void_p(0x1000)
    # 4096 x 4096 bf16 parameters alone are 32 MiB of scratch
    st = lib.pc_sum_layer_fwd_noalloc(1, 4096, 4096, 128, fake, fake, 0, fake, 0, None)
    assert N.STATUS[st] == "PC_ERR_UNSUPPORTED"
    msg = lib.pc_last_error().decode()
    assert "built-in scratch" in msg and "pc_sum_layer_fwd" in msg
