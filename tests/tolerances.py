"""Parity bars of the GPU tests.

Per-sample log-likelihood (for a single layer: every entry of ``out``), absolute:
fp32 1e-5, tf32 1e-3, auto (bf16 products) 8e-3.
Flows, elementwise relative with a floor: |gpu - ref| <= tol * (|ref| + 1e-6 max|ref|);
fp32 1e-5 is the stated bar; tf32 1e-3 and auto 3e-2 are the library's reading for
modes whose flow error the pages do not bound (the pages measured TF32 flows at
5e-5 / 3e-4 on one HMM layer, pyjuice PR #62 Summary 3).
"""
import numpy as np

LL_TOL = {"auto": 8e-3, "tf32": 1e-3, "fp32": 1e-5}
FLOW_TOL = {"auto": 3e-2, "tf32": 1e-3, "fp32": 1e-5}
MODES = ("auto", "tf32", "fp32")


def ll_err(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_inf = np.isneginf(gpu) & np.isneginf(ref)
    if np.any(np.isneginf(gpu) != np.isneginf(ref)):
        return np.inf
    d = np.abs(np.where(both_inf, 0.0, gpu - np.where(both_inf, 0.0, ref)))
    return float(d.max()) if d.size else 0.0


def out_err(gpu, ref):
    """ll_err for a float32 output array: the error beyond the float32 representation
    of the exact value (|fl32(ref) - ref|, up to half an ulp), which no float32
    result can avoid (at |out| = 1000 that alone is 3e-5)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if np.any(np.isneginf(gpu) != np.isneginf(ref)):
        return np.inf
    fin = np.isfinite(ref)
    rep = np.abs(ref[fin].astype(np.float32).astype(np.float64) - ref[fin])
    d = np.maximum(np.abs(gpu[fin] - ref[fin]) - rep, 0.0)
    return float(d.max()) if d.size else 0.0


def flow_err(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not np.all(np.isfinite(gpu)):
        return np.inf
    floor = 1e-6 * np.abs(ref).max() if ref.size else 0.0
    if floor == 0.0:
        return float(np.abs(gpu).max()) if gpu.size else 0.0
    return float((np.abs(gpu - ref) / (np.abs(ref) + floor)).max())
