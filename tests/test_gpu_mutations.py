"""The GPU parity checks catch plausible mistakes in the dense layer (pyjuice PR #62,
Tests: each of nine mutations of the dense path is caught). Mistakes are planted here,
in CPU restatements of the oracle, never in a GPU kernel: the GPU result (fp32 mode) must
pass against the oracle at the stated bars and fail against every mutated result, so a
GPU path with that mistake would fail the parity tests.

The layer has two evenly strided groups whose children sit 120 nats below and 100 nats
above zero, where a forward without the per-group column maximum over- or underflows in
float32.
"""
import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from oracle import emulate
from oracle.sum_layer import sum_layer_bwd, sum_layer_fwd
from tolerances import FLOW_TOL, LL_TOL, flow_err, out_err
from workloads import layer_inputs

pytestmark = pytest.mark.gpu

G, M, CS, B = 2, 256, 270, 96


@pytest.fixture(scope="module")
def case():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pc.load()
    d = layer_inputs(G, M, M, B, seed=610, child_stride=CS, f_kind="uniform")
    x = d["x"].astype(np.float64)
    x[:CS] -= 120.0
    x[CS:] += 100.0
    d["x"] = x.astype(np.float32)
    th, xx, f = (torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("theta", "x", "f"))
    out = pc.sum_layer_fwd(th, xx, child_stride=CS, precision="fp32")
    # the backward on the oracle's out rounded to float32, as the oracle's own check does
    ref_out = sum_layer_fwd(d["theta"], d["x"], CS)
    e, F = pc.sum_layer_bwd(th, xx, torch.from_numpy(ref_out.astype(np.float32)).cuda(), f, child_stride=CS,
                            precision="fp32")
    torch.cuda.synchronize()
    pc.device_status()
    out32 = ref_out.astype(np.float32).astype(np.float64)
    ref_e, ref_F = sum_layer_bwd(d["theta"], d["x"], CS, out32, d["f"])
    return d, (out.cpu().numpy(), e.cpu().numpy(), F.cpu().numpy()), (ref_out, ref_e, ref_F), out32


def _rows(g):
    return slice(g * CS, g * CS + M)


def _flows(theta, x, out, f, mutate):
    """The oracle's flows with one factor replaced by mutate(name, value)."""
    e = np.zeros_like(x)
    F = np.zeros_like(theta)
    for g in range(G):
        xs = x[_rows(g)]
        m = xs.max(axis=0)
        u = mutate("u", np.exp(xs - m))
        w = f[g] * mutate("r", np.exp(m - out[g]), m=m, out=out[g])
        e[_rows(g)] += mutate("e", u * (theta[g].T @ w), theta_t_w=theta[g].T @ w)
        F[g] = mutate("F", theta[g] * (w @ u.T), w_ut=w @ u.T)
    return e, F


def _keep(name, v, **kw):
    return v


MUTATIONS = {
    # forward
    "theta transposed": ("out", lambda d, o: sum_layer_fwd(np.swapaxes(d["theta"], 1, 2), d["x"], CS)),
    "no column max (float32)": ("out", lambda d, o: np.stack([
        np.log(d["theta"][g].astype(np.float32) @ np.exp(d["x"][_rows(g)].astype(np.float32))).astype(np.float64)
        for g in range(G)])),
    "children of the next row": ("out", lambda d, o: sum_layer_fwd(d["theta"], np.roll(d["x"], -1, axis=0), CS)),
    "one-pass TF32 products": ("out", lambda d, o: emulate.sum_layer_fwd(d["theta"], d["x"], "tf32", CS)),
    "lo*hi cross term dropped": ("out", lambda d, o: np.stack([
        (lambda xs: xs.max(0) + np.log(
            (lambda ph, pl, qh, ql: ph @ qh + ph @ ql)(
                *[t.astype(np.float64) for t in emulate.split_tf32(d["theta"][g])],
                *[t.astype(np.float64) for t in emulate.split_tf32(np.exp(xs - xs.max(0)))])))(
            d["x"][_rows(g)].astype(np.float64)) for g in range(G)])),
    "output rounded to bf16": ("out", lambda d, o: emulate.round_bf16(o[0].astype(np.float32)).astype(np.float64)),
    # backward
    "element flows without exp(x - m)": ("e", lambda d, o: _flows(
        d["theta"], d["x"], o[1], d["f"], lambda n, v, **k: k["theta_t_w"] if n == "e" else v)[0]),
    "parameter flows without theta": ("F", lambda d, o: _flows(
        d["theta"], d["x"], o[1], d["f"], lambda n, v, **k: k["w_ut"] if n == "F" else v)[1]),
    "flow scale exp(out - m)": ("e", lambda d, o: _flows(
        d["theta"], d["x"], o[1], d["f"], lambda n, v, **k: np.exp(k["out"] - k["m"]) if n == "r" else v)[0]),
}


def test_gpu_matches_the_oracle(case):
    d, (go, ge, gF), (ro, re, rF), _ = case
    assert out_err(go, ro) <= LL_TOL["fp32"]
    assert flow_err(ge, re) <= FLOW_TOL["fp32"] and flow_err(gF, rF) <= FLOW_TOL["fp32"]


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_mutation_is_caught(case, name):
    d64 = {k: (v.astype(np.float64) if isinstance(v, np.ndarray) else v) for k, v in case[0].items()}
    (go, ge, gF), (ro, _, _), out32 = case[1], case[2], case[3]
    which, fn = MUTATIONS[name]
    with np.errstate(all="ignore"):
        mut = fn(d64, (ro, out32))
    if which == "out":
        err = out_err(go, mut) if np.isfinite(mut).all() else np.inf
        print(f"{name}: out error against the mutation {err:.3e}")
        assert err > LL_TOL["fp32"]
    else:
        err = flow_err(ge if which == "e" else gF, mut) if np.isfinite(mut).all() else np.inf
        print(f"{name}: flow error against the mutation {err:.3e}")
        assert err > FLOW_TOL["fp32"]
