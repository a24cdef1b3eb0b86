"""GB300-native log-space sum layers for probabilistic circuits.

The computation lives in ``libpcsum.so`` (hand-written sm_103a CUDA behind the C
ABI declared in ``include/pcsum.h``); this package is a thin ctypes binding that
passes PyTorch device memory and streams to it. Build the library with
``python -m log_space_sum_gb300.build``.
"""
from ._native import PCError, declared_symbols, load  # noqa: F401
from .api import (  # noqa: F401
    PRECISIONS,
    device_status,
    em_normalize,
    hclt_fwd_bwd,
    hclt_prepare,
    hmm_fwd_bwd,
    hmm_lowrank_fwd_bwd,
    lowrank_exp_sum_bwd,
    lowrank_exp_sum_fwd,
    lowrank_sum_exp_bwd,
    lowrank_sum_exp_fwd,
    precision_code,
    profile_start,
    set_wait_limit_ns,
    profile_stop,
    sum_layer_bwd,
    sum_layer_fwd,
)

__version__ = "0.1.0"
