"""Seeded synthetic inputs for the log-space sum-layer workloads.

This module is shared by the CUDA path's tests/bench and by the float64 oracle.
It draws random numbers and shapes them into parameters (softmax rows), child
log-values and token/category indices. It holds none of the method's
arithmetic: no sum layer, no circuit, no flow is computed here.

Every generator draws in float64 with ``numpy.random.default_rng(seed)`` and
returns float32 arrays (what the GPU receives) plus int32 index arrays. The
oracle promotes the float32 arrays back to float64, so rounding of the inputs
is never counted as error.

Workloads (pyjuice PR #62, Results table; pyjuice LowRank API doc, Note):

* ``tiny_hmm``  - 32 latents, 8 positions, vocab 16, batch 16 (seed 1)
* ``layer``     - one dense shared-children layer, M=N=1024, batch 128 (seed 2)
* ``hmm``       - 4096 latents, 32 positions, vocab 1024, batch 128/512 (seeds 3/4)
* ``hclt``      - 768 variables, 1024 latents, 512 categories, batch 512 (seed 5)
* ``lowrank``   - 1024 states, rank 16, batch 64, spread 0.3/1/4 nats (seeds 6/7/8)
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "softmax_rows", "hmm_inputs", "hmm_edge_inputs", "tiny_hmm", "hmm", "layer_inputs", "layer",
    "hclt_parents", "hclt_inputs", "hclt", "lowrank_inputs", "lowrank",
    "SPREAD_SEEDS",
]


def softmax_rows(logits: np.ndarray) -> np.ndarray:
    """Rows of a softmax, float64 (the distribution recipe of the parameters)."""
    z = logits - logits.max(axis=-1, keepdims=True)
    p = np.exp(z)
    return p / p.sum(axis=-1, keepdims=True)


def _f32(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


# ---------------------------------------------------------------- HMM circuits
def hmm_inputs(H: int, T: int, V: int, B: int, seed: int):
    """HMM parameters and tokens.

    pi [H], A [H,H] (row k = P(z_{t+1} | z_t = k)), E [H,V] (row k = P(x | z = k)),
    each row a softmax of N(0,1) logits; tokens [B,T] int32 uniform in [0,V).
    """
    rng = np.random.default_rng(seed)
    pi = softmax_rows(rng.standard_normal(H))
    A = softmax_rows(rng.standard_normal((H, H)))
    E = softmax_rows(rng.standard_normal((H, V)))
    tokens = rng.integers(0, V, size=(B, T), dtype=np.int64).astype(np.int32)
    return dict(pi=_f32(pi), A=_f32(A), E=_f32(E), tokens=np.ascontiguousarray(tokens))


def hmm_edge_inputs(H: int, T: int, V: int, B: int, seed: int, e_scale: float = 1.0, zero_A: float = 0.0,
                    zero_E: float = 0.0):
    """HMM inputs with the structure of the numerical edge cases: emission rows a softmax
    of N(0, e_scale^2) logits (peaked for a large scale), and a fraction of exact zeros
    in the rows of A and of E (each row keeps its largest entry; rows renormalised).
    Tokens uniform in [0, V)."""
    rng = np.random.default_rng(seed)
    pi = softmax_rows(rng.standard_normal(H))
    A = softmax_rows(rng.standard_normal((H, H)))
    E = softmax_rows(e_scale * rng.standard_normal((H, V)))
    for M, frac in ((A, zero_A), (E, zero_E)):
        if frac > 0:
            keep = rng.uniform(size=M.shape) >= frac
            keep[np.arange(M.shape[0]), M.argmax(axis=1)] = True
            M *= keep
            M /= M.sum(axis=1, keepdims=True)
    tokens = rng.integers(0, V, size=(B, T), dtype=np.int64).astype(np.int32)
    return dict(pi=_f32(pi), A=_f32(A), E=_f32(E), tokens=np.ascontiguousarray(tokens))


def tiny_hmm():
    return hmm_inputs(32, 8, 16, 16, seed=1)


def hmm(B: int = 512):
    if B not in (128, 512):
        raise ValueError("the HMM workload is defined at batch 128 and 512")
    return hmm_inputs(4096, 32, 1024, B, seed=3 if B == 128 else 4)


def hmm_1024x64():
    """The second HMM workload of the pages' timing table: 1024 latents, 64 positions,
    batch 512 (the vocabulary is not stated there: 1024, as in the 4096-latent one)."""
    return hmm_inputs(1024, 64, 1024, 512, seed=9)


# ------------------------------------------------------- single dense layer
def layer_inputs(G: int, M: int, N: int, B: int, seed: int, child_stride: int | None = None,
                 x_scale: float = 3.0, f_kind: str = "ones"):
    """Dense sum-layer inputs.

    theta [G,M,N] rows softmax N(0,1); x [rows,B] child log-values, each group's
    column a log-softmax over its N children of N(0, x_scale^2) logits; f [G,M,B]
    node flows (ones, or uniform(0,1) with f_kind="uniform").
    """
    rng = np.random.default_rng(seed)
    cs = N if child_stride is None else child_stride
    theta = softmax_rows(rng.standard_normal((G, M, N)))
    rows = (G - 1) * cs + N if G > 0 else 0
    logits = x_scale * rng.standard_normal((rows, B))
    x = np.empty_like(logits)
    for g in range(G):
        blk = logits[g * cs:g * cs + N]
        mx = blk.max(axis=0, keepdims=True)
        x[g * cs:g * cs + N] = blk - mx - np.log(np.exp(blk - mx).sum(axis=0, keepdims=True))
    if f_kind == "ones":
        f = np.ones((G, M, B))
    elif f_kind == "uniform":
        f = rng.uniform(0.0, 1.0, size=(G, M, B))
    else:
        raise ValueError(f_kind)
    return dict(theta=_f32(theta), x=_f32(x), f=_f32(f), child_stride=cs)


def layer():
    return layer_inputs(1, 1024, 1024, 128, seed=2)


# ------------------------------------------------------------------- HCLT
def hclt_parents(nvars: int, seed: int) -> np.ndarray:
    """Random spanning tree: parent[0] = -1, parent[i] uniform in [0, i)."""
    rng = np.random.default_rng(seed)
    parent = np.empty(nvars, dtype=np.int32)
    parent[0] = -1
    for i in range(1, nvars):
        parent[i] = rng.integers(0, i)
    return parent


def hclt_inputs(nvars: int, H: int, C: int, B: int, seed: int, parent=None):
    """HCLT parameters: pi [H]; W [nvars,H,H] (W[c][z_parent][z_c], W[0] unused,
    left uniform); E [nvars,H,C]; data [B,nvars] uniform categories."""
    if parent is None:
        parent = hclt_parents(nvars, seed)
    rng = np.random.default_rng(seed + 1000)
    pi = softmax_rows(rng.standard_normal(H))
    W = np.empty((nvars, H, H), dtype=np.float32)
    W[0] = 1.0 / H
    for c in range(1, nvars):
        W[c] = softmax_rows(rng.standard_normal((H, H)))
    E = np.empty((nvars, H, C), dtype=np.float32)
    for v in range(nvars):
        E[v] = softmax_rows(rng.standard_normal((H, C)))
    data = rng.integers(0, C, size=(B, nvars), dtype=np.int64).astype(np.int32)
    return dict(parent=np.ascontiguousarray(parent, dtype=np.int32), pi=_f32(pi), W=W, E=E,
                data=np.ascontiguousarray(data))


def hclt():
    return hclt_inputs(768, 1024, 512, 512, seed=5)


# ---------------------------------------------------------------- LowRank
SPREAD_SEEDS = {0.3: 6, 1.0: 7, 4.0: 8}


def lowrank_inputs(M: int, N: int, K: int, B: int, spread: float, seed: int,
                   x_scale: float = 3.0, f_kind: str = "ones"):
    """LowRank exp_sum inputs: theta [M,N] rows softmax N(0,1); A [B,M,K] and
    Bm [B,K,N] drawn N(0, s^2) with s = sqrt(spread / sqrt(K)) so that the
    standard deviation of an entry of A_b B_b is ``spread`` nats; x [N,B] a
    log-softmax over the N children of N(0, x_scale^2) logits; f [M,B]."""
    rng = np.random.default_rng(seed)
    s = float(np.sqrt(spread / np.sqrt(K)))
    theta = softmax_rows(rng.standard_normal((M, N)))
    A = s * rng.standard_normal((B, M, K))
    Bm = s * rng.standard_normal((B, K, N))
    logits = x_scale * rng.standard_normal((N, B))
    mx = logits.max(axis=0, keepdims=True)
    x = logits - mx - np.log(np.exp(logits - mx).sum(axis=0, keepdims=True))
    f = np.ones((M, B)) if f_kind == "ones" else rng.uniform(0.0, 1.0, size=(M, B))
    return dict(theta=_f32(theta), A=_f32(A), Bm=_f32(Bm), x=_f32(x), f=_f32(f))


def lowrank(spread: float = 1.0):
    return lowrank_inputs(1024, 1024, 16, 64, spread, seed=SPREAD_SEEDS[spread])


def hmm_lowrank_inputs(H: int, T: int, V: int, B: int, K: int, spread: float, seed: int):
    """An HMM (as hmm_inputs) plus one pair of LowRank factors per transition copy:
    FA [T-1,B,H,K], FB [T-1,B,K,H] drawn N(0, s^2) with s = sqrt(spread / sqrt(K)), so
    that an entry of FA[t][b] FB[t][b] has standard deviation ``spread`` nats."""
    d = hmm_inputs(H, T, V, B, seed)
    rng = np.random.default_rng(seed + 500)
    s = float(np.sqrt(spread / np.sqrt(K)))
    d["FA"] = _f32(s * rng.standard_normal((T - 1, B, H, K)))
    d["FB"] = _f32(s * rng.standard_normal((T - 1, B, K, H)))
    return d


def hmm_lowrank():
    """The pages' LowRank measurement setting: an HMM of 1024 states, rank 16, batch 64
    (64 positions and vocabulary 1024, as the pages' 1024-state HMM), spread 1 nat."""
    return hmm_lowrank_inputs(1024, 64, 1024, 64, 16, 1.0, seed=11)


# ------------------------------------------------------------------- EM M-step
def em_statistics(seed: int = 10):
    """Synthetic parameter statistics of the M-step at the HMM 4096 x 32 workload's
    parameter shapes (initial dpi [1, 4096], transitions dA [4096, 4096], emissions
    dE [4096, 1024]) and of the LowRank 1024 x 1024 layer (F+ and W): flows drawn
    Gamma(0.5, 1) (many small entries, a few large ones, as expected counts are), W
    drawn Gamma(2, 1), and previous parameters uniform in [0, 1)."""
    rng = np.random.default_rng(seed)
    shapes = {"pi": (1, 4096), "A": (4096, 4096), "E": (4096, 1024), "lowrank": (1024, 1024)}
    out = {}
    for k, shp in shapes.items():
        out["F_" + k] = rng.gamma(0.5, 1.0, size=shp).astype(np.float32)
        out["theta_" + k] = rng.random(shp).astype(np.float32)
    out["W_lowrank"] = rng.gamma(2.0, 1.0, size=shapes["lowrank"]).astype(np.float32)
    return out
