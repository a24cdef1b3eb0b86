"""Every entry point can be captured into a CUDA graph: the calls are asynchronous on the
caller's stream, issue no host synchronisation and no copy from pageable host memory (the
HCLT's tree plan travels in kernel arguments), and join their side stream back before
returning. Each case runs eagerly once (lazy set-up, workspace), is captured with
torch.cuda.graph, replayed, and compared with the eager result: bit-identical where the
kernels are deterministic, else (float atomic sums: the HMM's dpi, the LowRank flows of
the HMM) within 1e-6 relative.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import log_space_sum_gb300 as pc
from workloads import hclt_inputs, hmm_inputs, hmm_lowrank_inputs, layer_inputs, lowrank_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pc.load()


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        eager = [x.clone() if isinstance(x, torch.Tensor) else x for x in fn()]
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    for x in out:
        if isinstance(x, torch.Tensor):
            x.fill_(float("nan"))  # the replay must write every output
    g.replay()
    torch.cuda.synchronize()
    pc.device_status()
    return eager, list(out)


def _same(eager, graph, exact=True):
    for a, b in zip(eager, graph):
        if a is None:
            assert b is None
            continue
        if exact:
            assert torch.equal(a, b)
        else:
            torch.testing.assert_close(b, a, rtol=1e-6, atol=0, equal_nan=True)


def _t(a, dtype=None):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("mode", ["auto", "fp32"])
def test_sum_layer(mode):
    d = layer_inputs(2, 200, 130, 70, seed=600, child_stride=150, f_kind="uniform")
    th, x, f = _t(d["theta"]), _t(d["x"]), _t(d["f"])
    fwd = lambda: [pc.sum_layer_fwd(th, x, child_stride=150, precision=mode)]
    _same(*_capture(fwd))
    out = fwd()[0]
    _same(*_capture(lambda: list(pc.sum_layer_bwd(th, x, out, f, child_stride=150, precision=mode))))


def test_sum_layer_noalloc():
    lib = pc.load()
    d = layer_inputs(1, 256, 320, 64, seed=601)
    th, x = _t(d["theta"]), _t(d["x"])
    out = torch.empty(1, 256, 64, device="cuda")

    def run():
        st = lib.pc_sum_layer_fwd_noalloc(1, 256, 320, 64, C.c_void_p(th.data_ptr()), C.c_void_p(x.data_ptr()), 0,
                                          C.c_void_p(out.data_ptr()), 0,
                                          C.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, lib.pc_last_error().decode()
        return [out]
    _same(*_capture(run))


@pytest.mark.parametrize("mode", ["auto", "tf32", "fp32"])
def test_hmm(mode):
    d = hmm_inputs(300, 6, 17, 96, seed=602)
    t = {k: _t(d[k]) for k in ("tokens", "pi", "A", "E")}
    eager, graph = _capture(lambda: list(pc.hmm_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], precision=mode)))
    _same(eager[:1], graph[:1])        # ll
    _same(eager[2:], graph[2:])        # dA, dE: deterministic sums
    _same(eager[1:2], graph[1:2], exact=False)  # dpi: float atomics


@pytest.mark.parametrize("mode", ["auto", "fp32"])
def test_hclt(mode):
    d = hclt_inputs(12, 130, 7, 40, seed=603)
    t = {k: _t(d[k]) for k in ("data", "pi", "W", "E")}
    eager, graph = _capture(lambda: list(pc.hclt_fwd_bwd(d["parent"], t["data"], t["pi"], t["W"], t["E"],
                                                         precision=mode)))
    _same(eager[:1] + eager[2:], graph[:1] + graph[2:])
    _same(eager[1:2], graph[1:2], exact=False)  # dpi: float atomics


@pytest.mark.parametrize("mode", ["auto", "tf32"])
def test_hclt_prepared_and_persistent_tiles(mode):
    # H a multiple of 8: the forward and parameter contractions run on persistent tiles;
    # the prepared parameters are made outside the graph, the batch call is captured
    d = hclt_inputs(24, 256, 9, 256, seed=604)
    t = {k: _t(d[k]) for k in ("data", "pi", "W", "E")}
    prep = pc.hclt_prepare(d["parent"], t["W"], t["E"], precision=mode)
    torch.cuda.synchronize()
    eager, graph = _capture(lambda: list(pc.hclt_fwd_bwd(d["parent"], t["data"], t["pi"], t["W"], None,
                                                         precision=mode, prepared=prep)))
    _same(eager[:1] + eager[2:], graph[:1] + graph[2:])
    _same(eager[1:2], graph[1:2], exact=False)  # dpi: float atomics


@pytest.mark.parametrize("form", ["exp_sum", "sum_exp"])
def test_lowrank(form):
    d = lowrank_inputs(200, 150, 5, 24, spread=1.0, seed=604)
    th, A, Bm, x, f = (_t(d[k]) for k in ("theta", "A", "Bm", "x", "f"))
    if form == "exp_sum":
        fwd = lambda: list(pc.lowrank_exp_sum_fwd(th, A, Bm, x, precision="auto"))
        _same(*_capture(fwd))
        out, logZ = fwd()
        _same(*_capture(lambda: list(pc.lowrank_exp_sum_bwd(th, A, Bm, x, out, logZ, f, precision="auto").values())))
    else:
        _same(*_capture(lambda: list(pc.lowrank_sum_exp_fwd(th, A, Bm, x, precision="auto"))))
        _same(*_capture(lambda: list(pc.lowrank_sum_exp_bwd(th, A, Bm, x, f, precision="auto").values())))


def test_hmm_lowrank():
    d = hmm_lowrank_inputs(130, 5, 9, 6, 4, 1.0, seed=605)
    t = {k: _t(d[k]) for k in ("tokens", "pi", "A", "E", "FA", "FB")}
    eager, graph = _capture(lambda: list(pc.hmm_lowrank_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], t["FA"],
                                                                t["FB"], precision="auto").values()))
    _same(eager, graph, exact=False)


def test_em_normalize():
    rng = np.random.default_rng(606)
    F = _t(rng.gamma(0.5, 1.0, size=(300, 257)).astype(np.float32))
    th0 = _t(rng.uniform(size=(300, 257)).astype(np.float32))
    th = th0.clone()

    def run():
        th.copy_(th0)  # device to device: capturable
        return [pc.em_normalize(F, th)]
    _same(*_capture(run))
