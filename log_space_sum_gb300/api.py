"""PyTorch-facing wrappers of the C ABI: argument checks and marshalling only.

Every computation runs in libpcsum.so's CUDA kernels. PyTorch supplies device
memory (outputs and the scratch workspace) and the current CUDA stream.

Precision modes (pyjuice PR #62, Summary 1 table): "auto" (bf16 products),
"tf32" (TF32 products), "fp32" (3xTF32 products). The removed flags
``force_use_bf16`` / ``force_use_fp32`` raise a TypeError naming ``precision=``
when set to True and are accepted and ignored when False (same page, Breaking
change).
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _native as N

PRECISIONS = {"auto": 0, "tf32": 1, "fp32": 2}

_ws_cache: dict = {}


def precision_code(precision) -> int:
    if isinstance(precision, str):
        if precision not in PRECISIONS:
            raise ValueError(f"unknown precision {precision!r}; valid modes are 'auto' (bf16 "
                             "products), 'tf32' and 'fp32' (3xTF32)")
        return PRECISIONS[precision]
    if isinstance(precision, int) and not isinstance(precision, bool):
        return precision            # the library rejects unknown codes with PC_ERR_UNKNOWN_PRECISION
    raise TypeError(f"precision must be 'auto', 'tf32' or 'fp32', not {type(precision).__name__}")


def _removed_flags(kwargs: dict, where: str) -> None:
    for flag in ("force_use_bf16", "force_use_fp32"):
        if flag in kwargs:
            if kwargs.pop(flag):
                raise TypeError(f"{where}: {flag} was removed; pass precision='auto', 'tf32' or "
                                "'fp32' instead")
    if kwargs:
        raise TypeError(f"{where}: unexpected keyword arguments {sorted(kwargs)}")


def _check(t: torch.Tensor, name: str, dtype=torch.float32, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(device) -> C.c_void_p:
    return C.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def workspace(nbytes: int, device) -> torch.Tensor:
    """Scratch buffer of at least nbytes, cached per (device, stream)."""
    key = (device, torch.cuda.current_stream(device).cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def _query(name: str, *args) -> int:
    out = C.c_size_t(0)
    N.call(name, *args, C.byref(out))
    return out.value


# --------------------------------------------------------------------- sum layer
def sum_layer_fwd(theta, x, child_stride=None, precision="auto", out=None, **removed):
    """out[g,i,b] = m_b + log sum_j theta[g,i,j] exp(x[g*cs+j, b] - m_b) (pc_sum_layer_fwd)."""
    _removed_flags(removed, "sum_layer_fwd")
    prec = precision_code(precision)
    _check(theta, "theta")
    dev = theta.device
    _check(x, "x", device=dev)
    G, M, Nn = theta.shape
    B = x.shape[1]
    cs = (Nn if G > 1 else 0) if child_stride is None else int(child_stride)
    if out is None:
        out = torch.empty(G, M, B, dtype=torch.float32, device=dev)
    _check(out, "out", device=dev)
    nb = _query("pc_sum_layer_workspace", G, M, Nn, B, prec)
    ws = workspace(nb, dev)
    N.call("pc_sum_layer_fwd", G, M, Nn, B, _ptr(theta), _ptr(x), cs, _ptr(out), prec,
           _ptr(ws), ws.numel(), _stream(dev))
    return out


def sum_layer_bwd(theta, x, out, f, child_stride=None, precision="auto", element_flows=True,
                  param_flows=True, e=None, F=None, accumulate=False, **removed):
    """Element flows e (shaped like x) and parameter flows F (shaped like theta)
    (pc_sum_layer_bwd). Without ``accumulate`` the flows are overwritten; rows of x
    outside every group keep e's previous values (zeros for a fresh e)."""
    _removed_flags(removed, "sum_layer_bwd")
    prec = precision_code(precision)
    _check(theta, "theta")
    dev = theta.device
    for t, n in ((x, "x"), (out, "out"), (f, "f")):
        _check(t, n, device=dev)
    G, M, Nn = theta.shape
    B = x.shape[1]
    cs = (Nn if G > 1 else 0) if child_stride is None else int(child_stride)
    if element_flows and e is None:
        e = torch.zeros_like(x)
    if param_flows and F is None:
        F = torch.empty_like(theta)
    if e is not None:
        _check(e, "e", device=dev)
    if F is not None:
        _check(F, "F", device=dev)
    nb = _query("pc_sum_layer_workspace", G, M, Nn, B, prec)
    ws = workspace(nb, dev)
    N.call("pc_sum_layer_bwd", G, M, Nn, B, _ptr(theta), _ptr(x), cs, _ptr(out), _ptr(f),
           _ptr(e if element_flows else None), _ptr(F if param_flows else None), int(bool(accumulate)),
           prec, _ptr(ws), ws.numel(), _stream(dev))
    return (e if element_flows else None), (F if param_flows else None)


# --------------------------------------------------------------------------- HMM
def hmm_fwd_bwd(tokens, pi, A, E, precision="auto", flows=True, ll=None, dpi=None, dA=None, dE=None,
                accumulate=False, **removed):
    """Whole HMM circuit (pc_hmm_fwd_bwd): returns (ll [B] float64, dpi [H], dA [H,H],
    dE [H,V]); the flows are None when ``flows`` is False."""
    _removed_flags(removed, "hmm_fwd_bwd")
    prec = precision_code(precision)
    _check(A, "A")
    dev = A.device
    _check(tokens, "tokens", dtype=torch.int32, device=dev)
    _check(pi, "pi", device=dev)
    _check(E, "E", device=dev)
    B, T = tokens.shape
    H, V = E.shape
    if ll is None:
        ll = torch.empty(B, dtype=torch.float64, device=dev)
    _check(ll, "ll", dtype=torch.float64, device=dev)
    if flows:
        dpi = torch.empty(H, dtype=torch.float32, device=dev) if dpi is None else dpi
        dA = torch.empty(H, H, dtype=torch.float32, device=dev) if dA is None else dA
        dE = torch.empty(H, V, dtype=torch.float32, device=dev) if dE is None else dE
        for t, n in ((dpi, "dpi"), (dA, "dA"), (dE, "dE")):
            _check(t, n, device=dev)
    else:
        dpi = dA = dE = None
    nb = _query("pc_hmm_workspace", H, T, V, B, prec)
    ws = workspace(nb, dev)
    N.call("pc_hmm_fwd_bwd", H, T, V, B, _ptr(tokens), _ptr(pi), _ptr(A), _ptr(E), _ptr(ll),
           _ptr(dpi), _ptr(dA), _ptr(dE), int(bool(accumulate)), prec, _ptr(ws), ws.numel(),
           _stream(dev))
    return ll, dpi, dA, dE


def hmm_lowrank_fwd_bwd(tokens, pi, A, E, FA, FB, precision="auto", flows=True, accumulate=False, ll=None, dpi=None,
                        dA=None, W=None, dE=None, dFA=None, dFB=None, **removed):
    """HMM circuit with LowRank exp_sum transitions (pc_hmm_lowrank_fwd_bwd): FA
    [T-1,B,H,K], FB [T-1,B,K,H] the copies' factors. Returns a dict with ll [B] float64
    and, when ``flows``, dpi [H], dA [H,H] (sum of the copies' F+), W [H,H] (sum of their
    Z-correction statistics), dE [H,V], dFA, dFB (gradients of sum ll). Output tensors may
    be passed in (with ``accumulate`` the flows are added to them)."""
    _removed_flags(removed, "hmm_lowrank_fwd_bwd")
    prec = precision_code(precision)
    _check(A, "A")
    dev = A.device
    _check(tokens, "tokens", dtype=torch.int32, device=dev)
    for t, n in ((pi, "pi"), (E, "E"), (FA, "FA"), (FB, "FB")):
        _check(t, n, device=dev)
    B, T = tokens.shape
    H, V = E.shape
    K = FA.shape[-1]
    if tuple(FA.shape) != (max(T - 1, 0), B, H, K) or tuple(FB.shape) != (max(T - 1, 0), B, K, H):
        raise ValueError(f"FA {tuple(FA.shape)} and FB {tuple(FB.shape)}: expected [T-1,B,H,K] and [T-1,B,K,H]")
    out = dict(ll=torch.empty(B, dtype=torch.float64, device=dev) if ll is None else ll)
    _check(out["ll"], "ll", dtype=torch.float64, device=dev)
    if flows:
        new = lambda *shape: torch.empty(*shape, dtype=torch.float32, device=dev)  # noqa: E731
        given = dict(dpi=dpi, dA=dA, W=W, dE=dE, dFA=dFA, dFB=dFB)
        fresh = dict(dpi=lambda: new(H), dA=lambda: new(H, H), W=lambda: new(H, H), dE=lambda: new(H, V),
                     dFA=lambda: torch.empty_like(FA), dFB=lambda: torch.empty_like(FB))
        for k, v in given.items():
            out[k] = fresh[k]() if v is None else _check(v, k, device=dev)
    g = lambda k: _ptr(out.get(k))  # noqa: E731
    nb = _query("pc_hmm_lowrank_workspace", H, T, V, B, K, prec)
    ws = workspace(nb, dev)
    N.call("pc_hmm_lowrank_fwd_bwd", H, T, V, B, K, _ptr(tokens), _ptr(pi), _ptr(A), _ptr(E), _ptr(FA), _ptr(FB),
           g("ll"), g("dpi"), g("dA"), g("W"), g("dE"), g("dFA"), g("dFB"), int(bool(accumulate)), prec, _ptr(ws),
           ws.numel(), _stream(dev))
    return out


# -------------------------------------------------------------------------- HCLT
class HcltPrepared:
    """The HCLT's parameters in its contractions' formats (pc_hclt_prepare): reusable by
    every hclt_fwd_bwd call with the same tree, W, E and precision until they change."""

    def __init__(self, buf, parent, nvars, H, C, prec):
        self.buf, self.parent, self.nvars, self.H, self.C, self.prec = buf, parent, nvars, H, C, prec


def _host_parent(parent):
    import numpy as np
    return np.ascontiguousarray(np.asarray(parent.cpu() if isinstance(parent, torch.Tensor) else parent,
                                           dtype=np.int32))


def hclt_prepare(parent, W, E, precision="auto"):
    """Converts W and E once into the formats the HCLT's contractions read (pc_hclt_prepare)."""
    prec = precision_code(precision)
    _check(W, "W")
    dev = W.device
    _check(E, "E", device=dev)
    par = _host_parent(parent)
    n, H, Ccat = E.shape
    nb = _query("pc_hclt_prepare_bytes", n, H, Ccat, prec)
    buf = torch.empty(nb, dtype=torch.uint8, device=dev)
    N.call("pc_hclt_prepare", n, H, Ccat, par.ctypes.data_as(C.c_void_p), _ptr(W), _ptr(E), prec, _ptr(buf),
           buf.numel(), _stream(dev))
    return HcltPrepared(buf, par, n, H, Ccat, prec)


def hclt_fwd_bwd(parent, data, pi, W, E, precision="auto", flows=True, ll=None, dpi=None, dW=None, dE=None,
                 accumulate=False, prepared=None, **removed):
    """Whole HCLT circuit (pc_hclt_fwd_bwd). ``parent`` is a host int sequence
    (parent[0] = -1, parent[i] in [0, i)); data [B, nvars] int32 on the GPU; W
    [nvars, H, H]; E [nvars, H, C]. Returns (ll [B] float64, dpi, dW, dE). With
    ``prepared`` (from hclt_prepare for the same parent, W, E and precision) the call
    uses pc_hclt_fwd_bwd_prepared and E may be None."""
    import numpy as np

    _removed_flags(removed, "hclt_fwd_bwd")
    prec = precision_code(precision)
    _check(W, "W")
    dev = W.device
    _check(data, "data", dtype=torch.int32, device=dev)
    _check(pi, "pi", device=dev)
    par = _host_parent(parent)
    B, n = data.shape
    if prepared is not None:
        if prepared.prec != prec or prepared.nvars != n or not np.array_equal(prepared.parent, par):
            raise ValueError("prepared parameters were made for another tree or precision")
        H, Ccat = prepared.H, prepared.C
    else:
        _check(E, "E", device=dev)
        _, H, Ccat = E.shape
    if par.shape != (n,):
        raise ValueError(f"parent has shape {par.shape}, expected ({n},)")
    if ll is None:
        ll = torch.empty(B, dtype=torch.float64, device=dev)
    _check(ll, "ll", dtype=torch.float64, device=dev)
    if flows:
        dpi = torch.empty(H, dtype=torch.float32, device=dev) if dpi is None else dpi
        dW = torch.empty(n, H, H, dtype=torch.float32, device=dev) if dW is None else dW
        dE = torch.empty(n, H, Ccat, dtype=torch.float32, device=dev) if dE is None else dE
        for t, nm in ((dpi, "dpi"), (dW, "dW"), (dE, "dE")):
            _check(t, nm, device=dev)
    else:
        dpi = dW = dE = None
    if prepared is not None:
        nb = _query("pc_hclt_prepared_workspace", n, H, Ccat, B, prec)
        ws = workspace(nb, dev)
        N.call("pc_hclt_fwd_bwd_prepared", n, H, Ccat, B, par.ctypes.data_as(C.c_void_p), _ptr(data), _ptr(pi),
               _ptr(W), _ptr(prepared.buf), prepared.buf.numel(), _ptr(ll), _ptr(dpi), _ptr(dW), _ptr(dE),
               int(bool(accumulate)), prec, _ptr(ws), ws.numel(), _stream(dev))
        return ll, dpi, dW, dE
    nb = _query("pc_hclt_workspace", n, H, Ccat, B, prec)
    ws = workspace(nb, dev)
    N.call("pc_hclt_fwd_bwd", n, H, Ccat, B, par.ctypes.data_as(C.c_void_p), _ptr(data), _ptr(pi), _ptr(W), _ptr(E),
           _ptr(ll), _ptr(dpi), _ptr(dW), _ptr(dE), int(bool(accumulate)), prec, _ptr(ws), ws.numel(),
           _stream(dev))
    return ll, dpi, dW, dE


# ----------------------------------------------------------------------- LowRank
def _lowrank_shapes(theta, A, Bm, x):
    _check(theta, "theta")
    dev = theta.device
    for t, n in ((A, "A"), (Bm, "B"), (x, "x")):
        _check(t, n, device=dev)
    M, Nn = theta.shape
    Bs, Ma, K = A.shape
    if Ma != M or tuple(Bm.shape) != (Bs, K, Nn) or tuple(x.shape) != (Nn, Bs):
        raise ValueError(f"LowRank shapes: theta {tuple(theta.shape)}, A {tuple(A.shape)}, B {tuple(Bm.shape)}, "
                         f"x {tuple(x.shape)}; expected A [B,M,K], B [B,K,N], x [N,B]")
    return dev, M, Nn, K, Bs


def lowrank_exp_sum_fwd(theta, A, Bm, x, precision="auto", out=None, logZ=None, **removed):
    """LowRank exp_sum layer forward (pc_lowrank_exp_sum_fwd): returns out [M,B] and
    logZ [B,M] = log Z_b[i], which the backward reads."""
    _removed_flags(removed, "lowrank_exp_sum_fwd")
    prec = precision_code(precision)
    dev, M, Nn, K, Bs = _lowrank_shapes(theta, A, Bm, x)
    out = torch.empty(M, Bs, dtype=torch.float32, device=dev) if out is None else out
    logZ = torch.empty(Bs, M, dtype=torch.float32, device=dev) if logZ is None else logZ
    _check(out, "out", device=dev)
    _check(logZ, "logZ", device=dev)
    nb = _query("pc_lowrank_exp_sum_workspace", M, Nn, K, Bs, 0, prec)
    ws = workspace(nb, dev)
    N.call("pc_lowrank_exp_sum_fwd", M, Nn, K, Bs, _ptr(theta), _ptr(A), _ptr(Bm), _ptr(x), _ptr(out), _ptr(logZ),
           prec, _ptr(ws), ws.numel(), _stream(dev))
    return out, logZ


def lowrank_exp_sum_bwd(theta, A, Bm, x, out, logZ, f, precision="auto", grads=True, element_flows=True,
                        param_flows=True, z_correction=True, dA=None, dB=None, e=None, Fplus=None, W=None,
                        accumulate=False, **removed):
    """LowRank exp_sum layer backward (pc_lowrank_exp_sum_bwd): returns a dict with dA
    [B,M,K], dB [B,K,N] (``grads``), e [N,B] (``element_flows``), Fplus [M,N]
    (``param_flows``) and W [M,N] (``z_correction``); what is switched off is None."""
    _removed_flags(removed, "lowrank_exp_sum_bwd")
    prec = precision_code(precision)
    dev, M, Nn, K, Bs = _lowrank_shapes(theta, A, Bm, x)
    for t, n in ((out, "out"), (logZ, "logZ"), (f, "f")):
        _check(t, n, device=dev)
    new = lambda *shape: torch.empty(*shape, dtype=torch.float32, device=dev)  # noqa: E731
    dA = (new(Bs, M, K) if dA is None else dA) if grads else None
    dB = (new(Bs, K, Nn) if dB is None else dB) if grads else None
    e = (new(Nn, Bs) if e is None else e) if element_flows else None
    Fplus = (new(M, Nn) if Fplus is None else Fplus) if param_flows else None
    W = (new(M, Nn) if W is None else W) if z_correction else None
    for t, n in ((dA, "dA"), (dB, "dB"), (e, "e"), (Fplus, "Fplus"), (W, "W")):
        if t is not None:
            _check(t, n, device=dev)
    nb = _query("pc_lowrank_exp_sum_workspace", M, Nn, K, Bs, 1, prec)
    ws = workspace(nb, dev)
    N.call("pc_lowrank_exp_sum_bwd", M, Nn, K, Bs, _ptr(theta), _ptr(A), _ptr(Bm), _ptr(x), _ptr(out), _ptr(logZ),
           _ptr(f), _ptr(dA), _ptr(dB), _ptr(e), _ptr(Fplus), _ptr(W), int(bool(accumulate)), prec, _ptr(ws),
           ws.numel(), _stream(dev))
    return dict(dA=dA, dB=dB, e=e, Fplus=Fplus, W=W)


def lowrank_sum_exp_fwd(theta, A, Bm, x, precision="auto", out=None, logZ=None, **removed):
    """LowRank sum_exp layer forward (pc_lowrank_sum_exp_fwd), the scale g_b = exp(A_b)
    exp(B_b) summed over the rank: returns out [M,B] and logZ [B,M] = log Z_b[i]."""
    _removed_flags(removed, "lowrank_sum_exp_fwd")
    prec = precision_code(precision)
    dev, M, Nn, K, Bs = _lowrank_shapes(theta, A, Bm, x)
    out = torch.empty(M, Bs, dtype=torch.float32, device=dev) if out is None else out
    logZ = torch.empty(Bs, M, dtype=torch.float32, device=dev) if logZ is None else logZ
    _check(out, "out", device=dev)
    _check(logZ, "logZ", device=dev)
    nb = _query("pc_lowrank_sum_exp_workspace", M, Nn, K, Bs, 0, prec)
    ws = workspace(nb, dev)
    N.call("pc_lowrank_sum_exp_fwd", M, Nn, K, Bs, _ptr(theta), _ptr(A), _ptr(Bm), _ptr(x), _ptr(out), _ptr(logZ),
           prec, _ptr(ws), ws.numel(), _stream(dev))
    return out, logZ


def lowrank_sum_exp_bwd(theta, A, Bm, x, f, precision="auto", grads=True, element_flows=True, param_flows=True,
                        z_correction=True, dA=None, dB=None, e=None, Fplus=None, W=None, accumulate=False,
                        flow_precision="bf16", **removed):
    """LowRank sum_exp layer backward (pc_lowrank_sum_exp_bwd): the same outputs as
    lowrank_exp_sum_bwd (dA, dB, e, Fplus, W; what is switched off is None).
    ``flow_precision="fp8"`` (precision "auto"): Fplus and W from e4m3 products."""
    _removed_flags(removed, "lowrank_sum_exp_bwd")
    if flow_precision not in ("bf16", "fp8"):
        raise ValueError(f"flow_precision must be 'bf16' or 'fp8', got {flow_precision!r}")
    prec = precision_code(precision)
    dev, M, Nn, K, Bs = _lowrank_shapes(theta, A, Bm, x)
    _check(f, "f", device=dev)
    new = lambda *shape: torch.empty(*shape, dtype=torch.float32, device=dev)  # noqa: E731
    dA = (new(Bs, M, K) if dA is None else dA) if grads else None
    dB = (new(Bs, K, Nn) if dB is None else dB) if grads else None
    e = (new(Nn, Bs) if e is None else e) if element_flows else None
    Fplus = (new(M, Nn) if Fplus is None else Fplus) if param_flows else None
    W = (new(M, Nn) if W is None else W) if z_correction else None
    for t, n in ((dA, "dA"), (dB, "dB"), (e, "e"), (Fplus, "Fplus"), (W, "W")):
        if t is not None:
            _check(t, n, device=dev)
    nb = _query("pc_lowrank_sum_exp_workspace", M, Nn, K, Bs, 1, prec)
    ws = workspace(nb, dev)
    N.call("pc_lowrank_sum_exp_bwd", M, Nn, K, Bs, _ptr(theta), _ptr(A), _ptr(Bm), _ptr(x), _ptr(f), _ptr(dA),
           _ptr(dB), _ptr(e), _ptr(Fplus), _ptr(W), int(bool(accumulate)), int(flow_precision == "fp8"), prec,
           _ptr(ws), ws.numel(), _stream(dev))
    return dict(dA=dA, dB=dB, e=e, Fplus=Fplus, W=W)


# -------------------------------------------------------------------- EM M-step
def em_normalize(F: torch.Tensor, theta: torch.Tensor, W: torch.Tensor | None = None) -> torch.Tensor:
    """EM M-step (pc_em_normalize), in place on ``theta`` (shape [..., N], rows = nodes):
    theta = normalize(F) over the last axis, or with ``W`` the LowRank conditional update
    normalize(F / W) (0 where W <= 0). A row whose statistic sums to 0 keeps theta."""
    _check(F, "F")
    _check(theta, "theta", device=F.device)
    if W is not None:
        _check(W, "W", device=F.device)
    if F.shape != theta.shape or (W is not None and W.shape != F.shape):
        raise ValueError(f"F {tuple(F.shape)}, theta {tuple(theta.shape)} and W must have one shape")
    if F.dim() < 1 or F.numel() == 0:
        raise ValueError("F must have at least one element")
    Nn = F.shape[-1]
    rows = F.numel() // Nn
    N.call("pc_em_normalize", 1, rows, Nn, _ptr(F), _ptr(W), _ptr(theta), _stream(F.device))
    return theta


# -------------------------------------------------------------------- diagnostics
def device_status(device=None) -> None:
    """Synchronises the current stream and raises PCError if a kernel gave up a bounded wait."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    N.call("pc_device_status", _stream(dev))


def set_wait_limit_ns(ns: int = 0) -> None:
    """Limit of the contraction kernel's first device-side waits on the current device
    (0 restores the 2 s default); a wait that runs out is reported by device_status()."""
    N.call("pc_set_wait_limit_ns", int(ns))


def profile_start(capacity: int = 4096) -> None:
    N.call("pc_profile_start", int(capacity))


def profile_stop(capacity: int = 4096):
    """Returns [(kind, ms, flops, launches)] for every record since profile_start: one
    contraction launch, or a chain of consecutive launches of one kind timed together."""
    cnt = C.c_int(0)
    ms = (C.c_float * capacity)()
    kind = (C.c_int * capacity)()
    flops = (C.c_longlong * capacity)()
    launches = (C.c_int * capacity)()
    N.call("pc_profile_stop", C.byref(cnt), ms, kind, flops, launches, int(capacity))
    return [(N.KINDS.get(kind[i], str(kind[i])), float(ms[i]), int(flops[i]), int(launches[i]))
            for i in range(cnt.value)]
