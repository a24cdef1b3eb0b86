"""Precision emulator: the oracle's arithmetic with the operands of each product
rounded as a precision mode rounds them.

pyjuice PR #62, Summary 1 table: "auto" (bf16 products), "tf32" (round-to-nearest
TF32 products), "fp32" (fp32-level products from three TF32 terms, the tf32x3
split of Summary 3). Readings where the pages are silent: bf16 rounds to nearest
even; TF32 rounds to nearest with ties away from zero; the 3xTF32 split is
hi = rn(v), lo = rn(v - hi) and the lo*lo product is dropped.

This is not a pin of correctness. It predicts whether each mode's error bound is
reachable with the planned operand splits, with products exact and sums in
float64 (the hardware's fp32 accumulation adds its own small error).
"""
from __future__ import annotations

import numpy as np

MODES = ("auto", "tf32", "fp32")


def round_bf16(v) -> np.ndarray:
    """float32 -> nearest bfloat16 (ties to even), returned as float32."""
    a = np.asarray(v, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    r = ((bits + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32).view(np.float32)
    return np.where(np.isfinite(a), r, a)


def round_tf32(v) -> np.ndarray:
    """float32 -> nearest TF32 (10 explicit mantissa bits, ties away from zero)."""
    a = np.asarray(v, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    r = ((bits + 0x1000) & 0xFFFFE000).astype(np.uint32).view(np.float32)
    return np.where(np.isfinite(a), r, a)


def split_tf32(v):
    """(hi, lo) with hi = rn_tf32(v) and lo = rn_tf32(v - hi), both float32."""
    a = np.asarray(v, dtype=np.float32)
    hi = round_tf32(a)
    lo = round_tf32((a - hi).astype(np.float32))
    return hi, lo


def mode_matmul(P, Q, mode: str) -> np.ndarray:
    """P @ Q with the operands rounded (from float32) as ``mode`` rounds them."""
    P32 = np.asarray(P, dtype=np.float32)
    Q32 = np.asarray(Q, dtype=np.float32)
    if mode == "auto":
        return round_bf16(P32).astype(np.float64) @ round_bf16(Q32).astype(np.float64)
    if mode == "tf32":
        return round_tf32(P32).astype(np.float64) @ round_tf32(Q32).astype(np.float64)
    if mode == "fp32":
        ph, pl = (t.astype(np.float64) for t in split_tf32(P32))
        qh, ql = (t.astype(np.float64) for t in split_tf32(Q32))
        return ph @ qh + ph @ ql + pl @ qh
    raise ValueError(f"unknown precision mode {mode!r}; expected one of {MODES}")


def sum_layer_fwd(theta, x, mode: str, child_stride: int = 0) -> np.ndarray:
    """The oracle's forward with theta and exp(x - m_b) rounded to the mode's operands."""
    theta = np.asarray(theta, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    G, M, N = theta.shape
    out = np.empty((G, M, x.shape[1]))
    for g in range(G):
        xs = x[g * child_stride:g * child_stride + N]
        m = xs.max(axis=0)
        u = np.exp(xs - m[None, :])
        with np.errstate(divide="ignore"):
            out[g] = m[None, :] + np.log(mode_matmul(theta[g], u, mode))
    return out


def hmm_ll(pi, A, E, tokens, mode: str) -> np.ndarray:
    """HMM log-likelihood with every transition product in ``mode``; each layer's
    children are shifted by their column maximum before rounding."""
    A = np.asarray(A, dtype=np.float64)
    E = np.asarray(E, dtype=np.float64)
    pi = np.asarray(pi, dtype=np.float64)
    tokens = np.asarray(tokens)
    B, T = tokens.shape
    logE = np.log(E)
    x = logE[:, tokens[:, T - 1]]
    for t in range(T - 2, -1, -1):
        m = x.max(axis=0)
        u = np.exp(x - m[None, :])
        x = logE[:, tokens[:, t]] + m[None, :] + np.log(mode_matmul(A, u, mode))
    m = x.max(axis=0)
    return m + np.log(pi @ np.exp(x - m[None, :]))
