"""Benchmark of the hot path: forward + backward of the HMM circuit (the headline), and
of the single sum layer, the HCLT circuit and the LowRank exp_sum layer.

Workloads (synthetic, seeded; see workloads/):
  hmm      HMM with 4096 latent states, 32 positions, vocabulary 1024, batch 512
           (pyjuice PR #62, Results table). One step = one pc_hmm_fwd_bwd call: 31 tied
           4096x4096 sum layers forward, the 31 element-flow contractions backward and
           the depth-15872 parameter-flow contraction.
  hmm1024  the table's second HMM: 1024 latent states, 64 positions, batch 512
           (vocabulary 1024): 63 + 63 tied 1024x1024 layers, depth-32256 dA.
  layer    one dense sum layer M = N = 1024, batch 128: pc_sum_layer_fwd + _bwd.
  hclt     HCLT, 768 variables, 1024 latents, 512 categories, batch 512: pc_hclt_fwd_bwd.
  lowrank  LowRank exp_sum layer M = N = 1024, rank 16, batch 64, scale spread 1 nat:
           pc_lowrank_exp_sum_fwd + _bwd (dA, dB, e, F+, W).
  lowrank_sum_exp  the same factors in the LowRank sum_exp form (pc_lowrank_sum_exp_*).
  hmm_lowrank  HMM 1024x64, batch 64, with LowRank rank-16 transitions (pc_hmm_lowrank_fwd_bwd).
  mstep    the EM M-step (pc_em_normalize) of the HMM 4096x32 parameters (dpi, dA, dE)
           and of the LowRank 1024x1024 layer (normalize F+ / W); unit: nodes/s.

python bench.py [--gpus N --steps K --warmup W --precision auto|tf32|fp32
                 --impl ours|reference --workload hmm|hmm1024|layer|hclt|lowrank|lowrank_sum_exp|hmm_lowrank|mstep]

Prints one JSON line (rank 0). Under torchrun each rank runs its own batch (weak
scaling; no data-path collective). Between timed steps a 256 MiB buffer is written to
flush the 126 MB L2. The value comes from a timed pass with only the step events;
the roofline entry from a second timed pass of the same steps in which the library
records a CUDA event pair around every contraction on the launching stream, or around
each HMM chain of same-kind contractions as a whole (pc_profile_start/stop) — events
between kernels serialise them, so they stay out of the first pass. ``--impl reference`` times the float64 CPU oracle on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

UNIT = "samples/s"
HMM_METRIC = "HMM 4096x32 fwd+bwd samples/s @batch 512 (1 GB300); % tensor/HBM roofline"
# pages' RTX PRO 6000 figures for the HMM workload (context, other hardware)
# The pages' whole-circuit figures (RTX PRO 6000, batch 512, forward + backward): another
# machine's numbers, the denominators of vs_baseline only.
PAGES_SAMPLES_PER_S = {
    "hmm": {"auto": 512 / 32.1e-3, "fp32": 512 / 49.9e-3},
    "hmm1024": {"auto": 512 / 10.2e-3, "fp32": 512 / 12.3e-3},
    "hclt": {"auto": 512 / 48.1e-3, "fp32": 512 / 64.3e-3},
}
DTYPE = {"auto": "bf16", "tf32": "tf32", "fp32": "3xtf32"}
# nominal dense tensor rates relative to bf16 (2.25 PF bf16, 1.1 PF tf32)
TF32_OVER_BF16 = 1.1 / 2.25
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# special-function unit: 16 exp2 results per SM per clock (the SM count comes from the device)
MUFU_PER_SM_CLK = 16
MEMORY_KINDS = ("hmm_mem", "hclt_mem", "em_mstep")


def choose_bf16_peak(peaks, clk):
    """The measured bf16 peak that applies to this run: the burst figure (a kernel timed
    at full clock), unless the clocks sampled during the timed region show a power-capped
    run well below the maximum, where the sustained figure (measured under the power cap)
    applies. Returns (TFLOP/s, which)."""
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    if clk and clk.get("sm_mhz") and clk.get("sm_max_mhz"):
        capped = "sw_power_cap" in (clk.get("reasons") or [])
        if capped and clk["sm_mhz"] < 0.9 * clk["sm_max_mhz"]:
            return sustained, "bf16 sustained (power-capped clocks)"
    return burst, "bf16 burst"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--precision", default="auto", choices=["auto", "tf32", "fp32"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--other-modes", type=int, default=1,
                    help="with --precision auto, also time the tf32 and fp32 modes (extra keys)")
    ap.add_argument("--workload", default="hmm",
                    choices=["hmm", "hmm1024", "layer", "hclt", "lowrank", "lowrank_sum_exp", "hmm_lowrank", "mstep"])
    ap.add_argument("--flow-fp8", action="store_true",
                    help="lowrank_sum_exp: e4m3 operands for the two flow contractions (precision auto)")
    ap.add_argument("--hclt-nvars", type=int, default=768,
                    help="HCLT variables (768 = the workload; fewer for a profiler-sized case)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ workloads
class Workload:
    """One benchmarked call sequence: its inputs (numpy, seeded), the GPU step through
    the public API on device-resident tensors, and the oracle on the first b samples."""

    name = metric = desc = ""
    batch = 0
    unit = UNIT  # a "sample" is one unit of the workload's batch
    unit_noun, oracle_what = "samples", "forward + backward"
    roofline_bound = "tensor"

    def dtype(self, prec):
        return DTYPE[prec]

    def config(self):
        return {}


class HmmWorkload(Workload):
    name, metric, batch = "hmm", HMM_METRIC, 512
    H, T, V = 4096, 32, 1024
    desc = "HMM 4096 latents x 32 positions, vocab 1024, batch 512: forward LL + backward flows dpi, dA, dE"
    data = "synthetic (seeded: softmax N(0,1) rows for pi, A, E; uniform tokens)"

    def inputs(self):
        from workloads import hmm
        return hmm(512)

    def config(self):
        return {"H": self.H, "T": self.T, "V": self.V, "B": self.batch}

    def oracle(self, d, b):
        from oracle.hmm import hmm_fwd_bwd
        hmm_fwd_bwd(d["pi"], d["A"], d["E"], d["tokens"][:b])

    def device(self, pc, d, dev, prec):
        import torch
        t = {k: torch.from_numpy(d[k]).to(dev) for k in ("tokens", "pi", "A", "E")}
        H, V = d["E"].shape
        out = dict(ll=torch.empty(self.batch, dtype=torch.float64, device=dev),
                   dpi=torch.empty(H, device=dev), dA=torch.empty(H, H, device=dev), dE=torch.empty(H, V, device=dev))

        def step(tok=None):
            pc.hmm_fwd_bwd(t["tokens"] if tok is None else tok, t["pi"], t["A"], t["E"], precision=prec, **out)
        host_in = torch.from_numpy(d["tokens"]).pin_memory()
        host_out = torch.empty(self.batch, dtype=torch.float64).pin_memory()
        dev_in = torch.empty_like(t["tokens"])

        def e2e():
            dev_in.copy_(host_in, non_blocking=True)
            step(dev_in)
            host_out.copy_(out["ll"], non_blocking=True)
        # the same, reading the flows back too (an EM loop keeps them on the device)
        host_flows = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in out.items() if k != "ll"}

        def e2e_flows():
            e2e()
            for k, h in host_flows.items():
                h.copy_(out[k], non_blocking=True)
        self.e2e_flows = (e2e_flows, host_out.numel() * 8 + sum(h.numel() * 4 for h in host_flows.values()))
        return step, e2e, host_in.numel() * 4, host_out.numel() * 8


class Hmm1024Workload(HmmWorkload):
    name, batch = "hmm1024", 512
    H, T, V = 1024, 64, 1024
    metric = "HMM 1024x64 fwd+bwd samples/s @batch 512 (1 GB300); % tensor/HBM roofline"
    desc = "HMM 1024 latents x 64 positions, vocab 1024, batch 512: forward LL + backward flows dpi, dA, dE"

    def inputs(self):
        from workloads import hmm_1024x64
        return hmm_1024x64()


class HmmLowRankWorkload(Workload):
    """An HMM whose 63 transition copies each carry the LowRank exp_sum scale with their own
    per-sample factors: every transition layer is the fused exp_sum layer."""
    name, batch = "hmm_lowrank", 64
    metric = "HMM 1024x64 with LowRank rank-16 transitions fwd+bwd samples/s @batch 64 (1 GB300)"
    desc = ("HMM 1024 latents x 64 positions, vocab 1024, batch 64, LowRank exp_sum rank 16 (spread 1 nat) on each "
            "transition copy: forward LL + backward dpi, dA (F+), W, dE and the factor gradients")
    data = "synthetic (seeded: softmax N(0,1) rows for pi, A, E; uniform tokens; factors N(0, s^2))"
    roofline_bound = "alu"

    def inputs(self):
        from workloads import hmm_lowrank
        return hmm_lowrank()

    def config(self):
        # M, N, B: the exp unit's work per transition layer (one exp per sample, node, child)
        return {"H": 1024, "T": 64, "V": 1024, "B": 64, "K": 16, "spread": 1.0, "M": 1024, "N": 1024}

    def oracle(self, d, b):
        from oracle.hmm_lowrank import hmm_lowrank_fwd_bwd
        hmm_lowrank_fwd_bwd(d["pi"], d["A"], d["E"], d["tokens"][:b], d["FA"][:, :b], d["FB"][:, :b])

    def device(self, pc, d, dev, prec):
        import torch
        t = {k: torch.from_numpy(d[k]).to(dev) for k in ("tokens", "pi", "A", "E", "FA", "FB")}
        out = pc.hmm_lowrank_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], t["FA"], t["FB"], precision=prec)
        bufs = {k: v for k, v in out.items()}

        def step(FA=None, FB=None):
            pc.hmm_lowrank_fwd_bwd(t["tokens"], t["pi"], t["A"], t["E"], t["FA"] if FA is None else FA,
                                   t["FB"] if FB is None else FB, precision=prec, **bufs)
        hA = torch.from_numpy(d["FA"]).pin_memory()
        hB = torch.from_numpy(d["FB"]).pin_memory()
        h_ll = torch.empty(self.batch, dtype=torch.float64).pin_memory()
        dA_in, dB_in = torch.empty_like(t["FA"]), torch.empty_like(t["FB"])

        def e2e():
            dA_in.copy_(hA, non_blocking=True)
            dB_in.copy_(hB, non_blocking=True)
            step(dA_in, dB_in)
            h_ll.copy_(bufs["ll"], non_blocking=True)
        return step, e2e, (hA.numel() + hB.numel()) * 4, h_ll.numel() * 8


class LayerWorkload(Workload):
    name, batch = "layer", 128
    metric = "sum layer 1024x1024 fwd+bwd samples/s @batch 128 (1 GB300)"
    desc = "dense sum layer M = N = 1024, batch 128: forward out + backward element flows e and parameter flows F"
    data = "synthetic (seeded: softmax N(0,1) theta rows; x log-softmax of N(0,9) logits; f = 1)"

    def inputs(self):
        from workloads import layer
        return layer()

    def config(self):
        return {"M": 1024, "N": 1024, "B": 128}

    def oracle(self, d, b):
        from oracle.sum_layer import sum_layer_bwd, sum_layer_fwd
        th = d["theta"].astype("float64")
        x = d["x"][:, :b].astype("float64")
        out = sum_layer_fwd(th, x)
        sum_layer_bwd(th, x, 0, out, d["f"][:, :, :b].astype("float64"))

    def device(self, pc, d, dev, prec):
        import torch
        th = torch.from_numpy(d["theta"]).to(dev)
        x = torch.from_numpy(d["x"]).to(dev)
        f = torch.from_numpy(d["f"]).to(dev)
        out = torch.empty(1, 1024, self.batch, device=dev)
        e = torch.zeros_like(x)
        F = torch.empty_like(th)

        def step(xin=None):
            xx = x if xin is None else xin
            pc.sum_layer_fwd(th, xx, precision=prec, out=out)
            pc.sum_layer_bwd(th, xx, out, f, precision=prec, e=e, F=F)
        host_in = torch.from_numpy(d["x"]).pin_memory()
        host_out = torch.empty(1024, self.batch).pin_memory()
        dev_in = torch.empty_like(x)

        def e2e():
            dev_in.copy_(host_in, non_blocking=True)
            step(dev_in)
            host_out.copy_(out[0], non_blocking=True)
        return step, e2e, host_in.numel() * 4, host_out.numel() * 4


class HcltWorkload(Workload):
    name, batch = "hclt", 512
    metric = "HCLT 768 vars x 1024 latents fwd+bwd samples/s @batch 512 (1 GB300)"
    desc = ("HCLT 768 variables, 1024 latents, 512 categories, random tree, batch 512: forward LL + backward "
            "flows dpi, dW, dE")
    data = "synthetic (seeded: parent[i] ~ U[0, i); softmax N(0,1) rows for pi, W, E; uniform categories)"

    nvars = 768

    def inputs(self):
        from workloads import hclt, hclt_inputs
        return hclt() if self.nvars == 768 else hclt_inputs(self.nvars, 1024, 512, 512, seed=5)

    def config(self):
        return {"nvars": self.nvars, "H": 1024, "C": 512, "B": 512}

    def oracle(self, d, b):
        from oracle.hclt import hclt_fwd_bwd
        hclt_fwd_bwd(d["parent"], d["data"][:b], d["pi"], d["W"], d["E"])

    def device(self, pc, d, dev, prec):
        import torch
        t = {k: torch.from_numpy(d[k]).to(dev) for k in ("data", "pi", "W", "E")}
        n, H, C = d["E"].shape
        out = dict(ll=torch.empty(self.batch, dtype=torch.float64, device=dev), dpi=torch.empty(H, device=dev),
                   dW=torch.empty(n, H, H, device=dev), dE=torch.empty(n, H, C, device=dev))

        def step(data=None):
            pc.hclt_fwd_bwd(d["parent"], t["data"] if data is None else data, t["pi"], t["W"], t["E"],
                            precision=prec, **out)
        host_in = torch.from_numpy(d["data"]).pin_memory()
        host_out = torch.empty(self.batch, dtype=torch.float64).pin_memory()
        dev_in = torch.empty_like(t["data"])

        def e2e():
            dev_in.copy_(host_in, non_blocking=True)
            step(dev_in)
            host_out.copy_(out["ll"], non_blocking=True)

        # the same step with the parameters prepared once (pc_hclt_prepare): an EM
        # iteration's batches share W and E
        prep = {}

        def prepare():
            prep["p"] = pc.hclt_prepare(d["parent"], t["W"], t["E"], precision=prec)

        def step_prepared():
            pc.hclt_fwd_bwd(d["parent"], t["data"], t["pi"], t["W"], None, precision=prec, prepared=prep["p"], **out)
        self.prepared = (prepare, step_prepared)
        return step, e2e, host_in.numel() * 4, host_out.numel() * 8


class LowRankWorkload(Workload):
    name, batch = "lowrank", 64
    metric = "LowRank exp_sum 1024x1024 rank 16 fwd+bwd samples/s @batch 64 (1 GB300); % exp-unit roofline"
    desc = ("LowRank exp_sum layer M = N = 1024, rank 16, batch 64, scale spread 1 nat: forward out, logZ + "
            "backward dA, dB, e, F+, W")
    data = "synthetic (seeded: softmax N(0,1) theta rows; A, B ~ N(0, s^2); x log-softmax of N(0,9) logits; f = 1)"
    roofline_bound = "alu"

    def inputs(self):
        from workloads import lowrank
        return lowrank(1.0)

    def config(self):
        return {"M": 1024, "N": 1024, "K": 16, "B": 64, "spread": 1.0}

    def oracle(self, d, b):
        from oracle.lowrank import lowrank_exp_sum_bwd
        lowrank_exp_sum_bwd(d["theta"], d["A"][:b], d["Bm"][:b], d["x"][:, :b], d["f"][:, :b])

    def device(self, pc, d, dev, prec):
        import torch
        t = {k: torch.from_numpy(d[k]).to(dev) for k in ("theta", "A", "Bm", "x", "f")}
        M, N = d["theta"].shape
        Bs, _, K = d["A"].shape
        out = torch.empty(M, Bs, device=dev)
        logZ = torch.empty(Bs, M, device=dev)
        g = dict(dA=torch.empty(Bs, M, K, device=dev), dB=torch.empty(Bs, K, N, device=dev),
                 e=torch.empty(N, Bs, device=dev), Fplus=torch.empty(M, N, device=dev), W=torch.empty(M, N, device=dev))

        def step(A=None, Bm=None):
            A = t["A"] if A is None else A
            Bm = t["Bm"] if Bm is None else Bm
            pc.lowrank_exp_sum_fwd(t["theta"], A, Bm, t["x"], precision=prec, out=out, logZ=logZ)
            pc.lowrank_exp_sum_bwd(t["theta"], A, Bm, t["x"], out, logZ, t["f"], precision=prec, **g)
        hA = torch.from_numpy(d["A"]).pin_memory()
        hB = torch.from_numpy(d["Bm"]).pin_memory()
        h_out = torch.empty(M, Bs).pin_memory()
        dA_in, dB_in = torch.empty_like(t["A"]), torch.empty_like(t["Bm"])

        def e2e():
            dA_in.copy_(hA, non_blocking=True)
            dB_in.copy_(hB, non_blocking=True)
            step(dA_in, dB_in)
            h_out.copy_(out, non_blocking=True)
        return step, e2e, (hA.numel() + hB.numel()) * 4, h_out.numel() * 4


class LowRankSumExpWorkload(LowRankWorkload):
    """The second form of the LowRank scale, g_b = sum_r exp(A_b[:, r]) exp(B_b[r, :]), on
    the same factors: every pass is tensor-core contractions over the (sample, rank)
    virtual batch, so the roofline is the tensor pipe's."""
    name = "lowrank_sum_exp"
    metric = "LowRank sum_exp 1024x1024 rank 16 fwd+bwd samples/s @batch 64 (1 GB300); % tensor roofline"
    desc = ("LowRank sum_exp layer M = N = 1024, rank 16, batch 64 (the exp_sum workload's factors): forward "
            "out, logZ + backward dA, dB, e, F+, W")
    roofline_bound = "tensor"

    def oracle(self, d, b):
        from oracle.lowrank import lowrank_sum_exp_bwd
        lowrank_sum_exp_bwd(d["theta"], d["A"][:b], d["Bm"][:b], d["x"][:, :b], d["f"][:, :b])

    flow_precision = "bf16"

    def config(self):
        return {**super().config(), "flow_precision": self.flow_precision}

    def device(self, pc, d, dev, prec):
        import torch
        t = {k: torch.from_numpy(d[k]).to(dev) for k in ("theta", "A", "Bm", "x", "f")}
        M, N = d["theta"].shape
        Bs, _, K = d["A"].shape
        out = torch.empty(M, Bs, device=dev)
        logZ = torch.empty(Bs, M, device=dev)
        g = dict(dA=torch.empty(Bs, M, K, device=dev), dB=torch.empty(Bs, K, N, device=dev),
                 e=torch.empty(N, Bs, device=dev), Fplus=torch.empty(M, N, device=dev), W=torch.empty(M, N, device=dev))
        fp = self.flow_precision

        def step(A=None, Bm=None):
            A = t["A"] if A is None else A
            Bm = t["Bm"] if Bm is None else Bm
            pc.lowrank_sum_exp_fwd(t["theta"], A, Bm, t["x"], precision=prec, out=out, logZ=logZ)
            pc.lowrank_sum_exp_bwd(t["theta"], A, Bm, t["x"], t["f"], precision=prec, flow_precision=fp, **g)
        hA = torch.from_numpy(d["A"]).pin_memory()
        hB = torch.from_numpy(d["Bm"]).pin_memory()
        h_out = torch.empty(M, Bs).pin_memory()
        dA_in, dB_in = torch.empty_like(t["A"]), torch.empty_like(t["Bm"])

        def e2e():
            dA_in.copy_(hA, non_blocking=True)
            dB_in.copy_(hB, non_blocking=True)
            step(dA_in, dB_in)
            h_out.copy_(out, non_blocking=True)
        return step, e2e, (hA.numel() + hB.numel()) * 4, h_out.numel() * 4


class MstepWorkload(Workload):
    """The EM M-step after a backward: every node's parameters normalized over its
    children (plain, for the HMM's dpi, dA, dE) or the LowRank conditional update
    normalize(F+ / W). A step updates all 9217 nodes; the unit is nodes/s."""
    name, unit, roofline_bound = "mstep", "nodes/s", "hbm"
    unit_noun, oracle_what = "nodes", "M-step"
    PARTS = (("pi", 1, 4096), ("A", 4096, 4096), ("E", 4096, 1024), ("lowrank", 1024, 1024))
    batch = sum(m for _, m, _ in PARTS)
    metric = "EM M-step nodes/s (HMM 4096x32 + LowRank 1024x1024 parameters, 1 GB300); % HBM roofline"
    desc = ("EM M-step: normalize dpi [1x4096], dA [4096x4096], dE [4096x1024] of the HMM 4096x32 workload "
            "and the LowRank 1024x1024 conditional update normalize(F+/W)")
    data = "synthetic (seeded: flows Gamma(0.5,1), W Gamma(2,1), previous parameters U[0,1))"

    def inputs(self):
        from workloads import em_statistics
        return em_statistics()

    def dtype(self, prec):
        return "f32"  # the M-step has no precision modes

    def config(self):
        return {"parts": {k: [m, n] for k, m, n in self.PARTS}, "nodes": self.batch}

    def oracle(self, d, b):
        from oracle.em import em_conditional, em_plain
        left = b
        for k, m, _ in self.PARTS:
            r = min(left, m)
            if r <= 0:
                break
            if k == "lowrank":
                em_conditional(d["F_lowrank"][:r], d["W_lowrank"][:r], d["theta_lowrank"][:r])
            else:
                em_plain(d["F_" + k][:r], d["theta_" + k][:r])
            left -= r

    def device(self, pc, d, dev, prec):
        import torch
        t = {k: torch.from_numpy(v).to(dev) for k, v in d.items()}
        names = [k for k, _, _ in self.PARTS]

        def step(src=None):
            s = t if src is None else src
            for k in names:
                pc.em_normalize(s["F_" + k], t["theta_" + k], s["W_lowrank"] if k == "lowrank" else None)
        host_in = {k: torch.from_numpy(d[k]).pin_memory() for k in d if k.startswith(("F_", "W_"))}
        dev_in = {k: torch.empty_like(t[k]) for k in host_in}
        host_out = {k: torch.empty(t["theta_" + k].shape, dtype=torch.float32).pin_memory() for k in names}

        def e2e():
            for k in host_in:
                dev_in[k].copy_(host_in[k], non_blocking=True)
            step(dev_in)
            for k in names:
                host_out[k].copy_(t["theta_" + k], non_blocking=True)
        h2d = sum(v.numel() * 4 for v in host_in.values())
        d2h = sum(v.numel() * 4 for v in host_out.values())
        return step, e2e, h2d, d2h


WORKLOADS = {w.name: w for w in (HmmWorkload(), Hmm1024Workload(), LayerWorkload(), HcltWorkload(), LowRankWorkload(),
                                 LowRankSumExpWorkload(), HmmLowRankWorkload(), MstepWorkload())}


# ------------------------------------------------------------------ CPU oracle
def oracle_sample_rate(w, d, target_s: float = 12.0):
    """The float64 oracle on a bounded sample of the workload: returns (samples/s,
    description, cores, b, seconds). The sample is the first b samples of the batch, b
    grown until one run takes about target_s seconds (at most the whole batch)."""
    b = 1
    while True:
        t0 = time.perf_counter()
        w.oracle(d, b)
        dt = time.perf_counter() - t0
        if dt >= target_s / 2 or b >= w.batch:
            break
        b = min(w.batch, max(b * 2, int(b * target_s / max(dt, 1e-3))))
    desc = (f"float64 NumPy oracle ({w.name}): the same {w.oracle_what} for the first {b} of the "
            f"{w.batch} {w.unit_noun} of the workload, {dt:.1f} s")
    return b / dt, desc, os.cpu_count(), b, dt


def pick_workload(args):
    w = WORKLOADS[args.workload]
    if w.name == "lowrank_sum_exp" and args.flow_fp8:
        w.flow_precision = "fp8"
        w.desc += " (flow contractions on e4m3 operands)"
    if w.name == "hclt" and args.hclt_nvars != 768:
        w.nvars = args.hclt_nvars
        w.desc = w.desc.replace("768 variables", f"{args.hclt_nvars} variables")
    return w


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = pick_workload(args)
    d = w.inputs()
    rate, desc, cores, b, _ = oracle_sample_rate(w, d, target_s=8.0)
    times = []
    for _ in range(args.steps):  # the sizing run above served as the warm-up
        t0 = time.perf_counter()
        w.oracle(d, b)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = b / (ms / 1e3)
    line = {
        "impl": "reference", "metric": w.metric, "value": value, "unit": w.unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.desc + f" (oracle on {b}-sample slices)", **w.config(), "sample_batch": b},
        "cpu_baseline": {"value": value, "unit": w.unit, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": w.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid):
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="pcsum_clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if device_uuid:
            cmd += ["-i", device_uuid]
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for row in fh:
                f = [c.strip() for c in row.split(",")]
                if len(f) < 8:
                    continue
                try:
                    sm.append(float(f[0]))
                    mx.append(float(f[1]))
                except ValueError:
                    continue
                for n, v in zip(names, f[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ traffic
def kernel_source_hash():
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "log_space_sum_gb300", "csrc", "*"))):
        with open(p, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kind: str, precision: str, workload: str):
    """DRAM bytes per launch of a contraction from a committed ncu capture of this
    workload, or None when there is none or the kernel sources changed since it was
    taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    ent = d.get(f"{workload}/{kind}:{precision}")
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ ranks
def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over all ranks (the slowest rank's time); x itself for one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, batch: int, steps: int, total_ms: float) -> float:
    """Whole-job samples/s: every rank processes its own batch per step (weak scaling)."""
    return world * batch * steps / (total_ms / 1e3)


# ------------------------------------------------------------------ GPU arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    import log_space_sum_gb300 as pc

    w = pick_workload(args)
    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    lib = pc.load()

    d = w.inputs()
    step, e2e_step, h2d_bytes, d2h_bytes = w.device(pc, d, dev, args.precision)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    pc.device_status(dev)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid) if rank == 0 else None

    # Timed pass 1 (the value): only the step events. The library's per-contraction
    # events would sit between the kernels of a step, serialise launches that otherwise
    # overlap (programmatic dependent launch) and slow the step down (measured 18% on
    # the HMM workload), so they are recorded in a second timed pass below.
    def timed_pass(profile: bool):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        n0 = lib.pc_launch_count()
        cap = 2000 * args.steps
        if profile:
            pc.profile_start(cap)
        for i in range(args.steps):
            flush.random_(0, 255) if i == 0 else flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        prof = pc.profile_stop(cap) if profile else []
        torch.cuda.synchronize(dev)
        n = lib.pc_launch_count() - n0
        if world > 1:
            dist.barrier()
        return [a.elapsed_time(b) for a, b in ev], prof, n

    ms_steps, _, launches = timed_pass(False)
    clk = clocks.stop() if clocks else None
    pc.device_status(dev)
    # Timed pass 2 (the roofline): the same steps with a CUDA event pair around every
    # contraction, recorded by the library on the launching stream.
    ms_steps_prof, prof, _ = timed_pass(True)
    pc.device_status(dev)
    total_ms = sum(ms_steps)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = job_rate(world, w.batch, args.steps, total_ms)

    # ---- roofline of the dominant kernel kind (by total time in the timed region)
    peaks, peak_src = load_peaks()
    by_kind = {}
    for kind, ms, fl, nl in prof:
        k = by_kind.setdefault(kind, [0.0, 0, 0])
        k[0] += ms
        k[1] += fl
        k[2] += nl
    # the dominant contraction kind (memory-bound kinds are reported in the hbm block)
    cands = [k for k in by_kind if k not in MEMORY_KINDS] or list(by_kind)
    dom = max(cands, key=lambda k: by_kind[k][0])
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # the memory-bound passes of the step (operand copies, transposes, gathers, product
    # and flow kernels): algorithmic bytes over their summed device time
    mem = {k: v for k, v in by_kind.items() if k in MEMORY_KINDS and k != dom}
    hbm = None
    if mem:
        mb = sum(v[1] for v in mem.values())
        mms = sum(v[0] for v in mem.values())
        hpeak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        hbm = {"kinds": sorted(mem), "launches_per_step": sum(v[2] for v in mem.values()) / args.steps,
               "bytes_per_step": mb / args.steps, "ms_per_step": mms / args.steps,
               "achieved": mb / (mms / 1e3) / 1e9, "peak": hpeak, "unit": "GB/s",
               "frac": mb / (mms / 1e3) / 1e9 / hpeak, "peak_source": f"{peak_src} copy bandwidth",
               "note": "summed event time of each memory-bound launch (side-stream ones overlap the chain)"}
    dms, dfl, dn = by_kind[dom]
    if w.roofline_bound == "hbm":
        # the kind's recorded count is its algorithmic bytes (read once, written once)
        achieved = dfl / (dms / 1e3) / 1e9
        peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        roofline = {
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": recorded_traffic(dom, args.precision, w.name), "kernel": f"k_em_normalize ({dom})",
            "launches_timed": dn, "ms_per_launch": dms / dn,
            "peak_source": f"{peak_src} copy bandwidth",
            "share_of_step": sum(v[0] for v in by_kind.values()) / sum(ms_steps_prof) if world == 1 else None,
        }
    elif w.roofline_bound == "alu":
        # one exp per (sample, node, child) in every LowRank pass
        cfg = w.config()
        exps = cfg["M"] * cfg["N"] * cfg["B"]
        mhz = (clk or {}).get("sm_max_mhz") or 2070.0
        peak = n_sms * MUFU_PER_SM_CLK * mhz * 1e6 / 1e12
        achieved = exps * dn / (dms / 1e3) / 1e12
        roofline = {
            "bound": "alu", "achieved": achieved, "peak": peak, "unit": "Texp/s", "frac": achieved / peak,
            "traffic": recorded_traffic(dom, args.precision, w.name), "kernel": f"k_lowrank* ({dom})",
            "launches_timed": dn, "ms_per_launch": dms / dn,
            "peak_source": f"derived: {n_sms} SMs x {MUFU_PER_SM_CLK} exp/clk x {mhz:.0f} MHz",
            "share_of_step": sum(v[0] for v in by_kind.values()) / sum(ms_steps_prof) if world == 1 else None,
        }
    else:
        achieved = dfl / (dms / 1e3) / 1e12
        bf16_peak, which = choose_bf16_peak(peaks, clk)
        peak = bf16_peak if args.precision == "auto" else bf16_peak * TF32_OVER_BF16
        con = {k: v for k, v in by_kind.items() if k not in MEMORY_KINDS}
        roofline = {
            "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": recorded_traffic(dom, args.precision, w.name), "kernel": f"k_umma_gemm ({dom})",
            "launches_timed": dn, "ms_per_launch": dms / dn,
            "peak_source": f"{peak_src} {which}" + ("" if args.precision == "auto"
                                                     else " x 1.1/2.25 (nominal tf32/bf16)"),
            "sm_mhz_during_timed_region": (clk or {}).get("sm_mhz"),
            "all_contractions_frac": sum(v[1] for v in con.values()) / (sum(v[0] for v in con.values())
                                                                       / 1e3) / 1e12 / peak,
            "share_of_step": sum(v[0] for v in con.values()) / sum(ms_steps_prof) if world == 1 else None,
        }
        if args.precision == "fp32":
            roofline["issued_frac"] = 3 * achieved / peak

    # ---- end to end through the public API with pinned host buffers
    e2e_ms = []
    for i in range(max(3, min(args.steps, 10))):
        flush.fill_(i & 0xFF)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e2e_step()
        torch.cuda.synchronize(dev)
        e2e_ms.append(1e3 * (time.perf_counter() - t0))
    e2e_value = job_rate(world, w.batch, 1, max_over_ranks(statistics.mean(e2e_ms), world, dev))
    e2e_flows = None
    if getattr(w, "e2e_flows", None):
        fn, fbytes = w.e2e_flows
        fms = []
        for i in range(max(3, min(args.steps, 10))):
            flush.fill_(i & 0xFF)
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            fms.append(1e3 * (time.perf_counter() - t0))
        e2e_flows = {"value": job_rate(world, w.batch, 1, max_over_ranks(statistics.mean(fms), world, dev)),
                     "unit": w.unit, "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(fbytes)}

    # a workload whose parameters can be prepared once per EM iteration (the HCLT): the
    # per-batch step with prepared parameters, and the preparation's own time
    prepared = None
    if getattr(w, "prepared", None):
        prep_fn, pstep = w.prepared
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        prep_fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        prep_ms = e0.elapsed_time(e1)
        for _ in range(3):
            pstep()
        torch.cuda.synchronize(dev)
        k = max(3, min(args.steps, 10))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        for i in range(k):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            pstep()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        pc.device_status(dev)
        tot = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), world, dev)
        prepared = {"value": job_rate(world, w.batch, k, tot), "ms_per_step": tot / k, "steps": k,
                    "prepare_ms": prep_ms,
                    "note": "W and E converted once per EM iteration (pc_hclt_prepare, prepare_ms) and read by "
                            "every batch's pc_hclt_fwd_bwd_prepared; value = the per-batch step"}

    # the other precision modes of the same workload, same timing rules (value only)
    modes = None
    if args.precision == "auto" and args.other_modes and w.name in ("hmm", "hmm1024", "hclt"):
        modes = {}
        for prec in ("tf32", "fp32"):
            mstep, *_ = w.device(pc, d, dev, prec)
            for _ in range(3):
                mstep()
            torch.cuda.synchronize(dev)
            k = max(3, min(args.steps, 10))
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize(dev)
            for i in range(k):
                flush.fill_(i & 0xFF)
                ev[i][0].record(stream)
                mstep()
                ev[i][1].record(stream)
            torch.cuda.synchronize(dev)
            pc.device_status(dev)
            tot = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), world, dev)
            modes[prec] = {"value": job_rate(world, w.batch, k, tot), "ms_per_step": tot / k, "steps": k,
                           "warmup": 3, "dtype": w.dtype(prec)}
            del mstep

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, cores, b, dt = oracle_sample_rate(w, d)
        cpu = {"value": rate, "unit": w.unit, "cores": cores, "kind": "oracle", "sample": desc}

    if rank == 0:
        ref = PAGES_SAMPLES_PER_S.get(w.name, {}).get(args.precision)
        if w.name == "hclt" and w.nvars != 768:
            ref = None
        line = {
            "metric": w.metric, "value": value, "unit": w.unit, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": (value / world / ref) if ref else None,
            "dtype": w.dtype(args.precision), "data": w.data,
            "config": {"workload": w.desc, **w.config(), "precision": args.precision,
                       "l2": "flushed between timed steps (256 MiB write)", "launch": "eager stream",
                       "parallelism": f"replicas x{world}"},
            "clocks": clk,
            "e2e": {"value": e2e_value, "unit": w.unit, "h2d_bytes_per_step": int(h2d_bytes),
                    "d2h_bytes_per_step": int(d2h_bytes)},
            "gpu_launches": int(launches),
            "roofline": roofline,
            "hbm": hbm,
            "e2e_with_flows": e2e_flows,
            "prepared_parameters": prepared,
            "modes": modes,
            "cpu_baseline": cpu,
            "step_ms": {"min": min(ms_steps), "median": statistics.median(ms_steps), "max": max(ms_steps),
                        "instrumented_median": statistics.median(ms_steps_prof)},
            "kernels": {k: {"launches": v[2], "ms": v[0], "tflops": v[1] / (v[0] / 1e3) / 1e12}
                        for k, v in by_kind.items()},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
