"""The precision emulator's rounding against torch's bf16 cast and hand-made TF32
bit patterns, and its prediction that each mode meets its error bound on the
single-layer workload's shape."""
import numpy as np
import pytest
import torch

from oracle import emulate
from oracle.sum_layer import sum_layer_fwd
from workloads import layer_inputs, hmm_inputs
from oracle.hmm import hmm_ll


def test_round_bf16_matches_torch_cast():
    rng = np.random.default_rng(50)
    v = (rng.standard_normal(100000) * np.exp(rng.uniform(-30, 30, 100000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(emulate.round_bf16(v), ref)


def test_round_tf32_ties_away_and_nearest():
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -10)
    cases = {
        1.0 + 2.0 ** -11: 1.0 + 2.0 ** -10,          # exact tie -> away from zero
        -(1.0 + 2.0 ** -11): -(1.0 + 2.0 ** -10),
        1.0 + 2.0 ** -12: 1.0,                       # below half -> down
        1.0 + 3 * 2.0 ** -12: 1.0 + 2.0 ** -10,      # above half -> up
        1.0 + 2.0 ** -10: 1.0 + 2.0 ** -10,          # representable -> unchanged
    }
    for a, b in cases.items():
        assert float(emulate.round_tf32(np.float32(a))) == b
    assert float(emulate.round_tf32(one)) == 1.0 and ulp > 0


def test_split_tf32_hi_lo():
    v = np.random.default_rng(51).standard_normal(10000).astype(np.float32)
    hi, lo = emulate.split_tf32(v)
    # hi and lo are TF32 values (13 low bits clear); hi + lo within 2^-22 relative of v
    assert np.all((hi.view(np.uint32) & 0x1FFF) == 0) and np.all((lo.view(np.uint32) & 0x1FFF) == 0)
    rel = np.abs((hi.astype(np.float64) + lo) - v) / np.abs(v)
    assert rel.max() < 2.0 ** -21


@pytest.mark.parametrize("mode,bound", [("auto", 8e-3), ("tf32", 1e-3), ("fp32", 1e-5)])
def test_layer_modes_reach_their_bounds(mode, bound):
    d = layer_inputs(1, 256, 512, 64, seed=2)
    th, x = d["theta"].astype(np.float64), d["x"].astype(np.float64)
    ref = sum_layer_fwd(th, x)
    emu = emulate.sum_layer_fwd(th, x, mode)
    err = np.abs(emu - ref).max()
    assert err < bound, (mode, err)


@pytest.mark.parametrize("mode,bound", [("auto", 8e-3), ("tf32", 1e-3), ("fp32", 1e-5)])
def test_hmm_chain_modes_reach_their_bounds(mode, bound):
    d = hmm_inputs(512, 32, 256, 8, seed=3)
    args = [d[k].astype(np.float64) for k in ("pi", "A", "E")] + [d["tokens"]]
    err = np.abs(emulate.hmm_ll(*args, mode) - hmm_ll(*args)).max()
    assert err < bound, (mode, err)
