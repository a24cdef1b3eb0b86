"""ctypes declarations of libpcsum.so (the C ABI in include/pcsum.h).

Loading fails loudly when the library has not been built: there is no fallback
implementation of any computation in this package.
"""
from __future__ import annotations

import ctypes as C
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpcsum.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "pcsum.h")

STATUS = {
    0: "PC_OK", 1: "PC_ERR_NULL", 2: "PC_ERR_SHAPE", 3: "PC_ERR_ALIGNMENT",
    4: "PC_ERR_UNKNOWN_PRECISION", 5: "PC_ERR_WORKSPACE", 6: "PC_ERR_UNSUPPORTED",
    7: "PC_ERR_CUDA", 8: "PC_ERR_TIMEOUT", 9: "PC_ERR_RANGE",
}

KINDS = {
    0: "layer_fwd", 1: "layer_elem", 2: "layer_param", 3: "hmm_fwd", 4: "hmm_elem",
    5: "hmm_param", 6: "hclt_fwd", 7: "hclt_elem", 8: "hclt_param", 9: "lowrank_fwd",
    10: "lowrank_bwd", 11: "em_mstep", 12: "hmm_mem", 13: "hclt_mem",
}
# kinds whose flops field holds algorithmic bytes
MEMORY_KINDS = {"em_mstep", "hmm_mem", "hclt_mem"}

_i, _ll, _sz, _p, _f, _d = C.c_int, C.c_longlong, C.c_size_t, C.c_void_p, C.c_float, C.c_double

# name -> argtypes (restype is the int status unless listed in _STR)
SIGNATURES = {
    "pc_version": [],
    "pc_status_string": [_i],
    "pc_last_error": [],
    "pc_device_status": [_p],
    "pc_set_wait_limit_ns": [C.c_ulonglong],
    "pc_launch_count": [],
    "pc_profile_start": [_i],
    "pc_profile_stop": [_p, _p, _p, _p, _p, _i],
    "pc_sum_layer_workspace": [_i, _i, _i, _i, _i, _p],
    "pc_sum_layer_fwd": [_i, _i, _i, _i, _p, _p, _ll, _p, _i, _p, _sz, _p],
    "pc_sum_layer_bwd": [_i, _i, _i, _i, _p, _p, _ll, _p, _p, _p, _p, _i, _i, _p, _sz, _p],
    "pc_sum_layer_fwd_noalloc": [_i, _i, _i, _i, _p, _p, _ll, _p, _i, _p],
    "pc_hmm_workspace": [_i, _i, _i, _i, _i, _p],
    "pc_hmm_fwd_bwd": [_i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _p, _sz, _p],
    "pc_hclt_workspace": [_i, _i, _i, _i, _i, _p],
    "pc_hclt_fwd_bwd": [_i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _p, _sz, _p],
    "pc_hclt_prepare_bytes": [_i, _i, _i, _i, _p],
    "pc_hclt_prepare": [_i, _i, _i, _p, _p, _p, _i, _p, _sz, _p],
    "pc_hclt_prepared_workspace": [_i, _i, _i, _i, _i, _p],
    "pc_hclt_fwd_bwd_prepared": [_i, _i, _i, _i, _p, _p, _p, _p, _p, _sz, _p, _p, _p, _p, _i, _i, _p, _sz, _p],
    "pc_lowrank_exp_sum_workspace": [_i, _i, _i, _i, _i, _i, _p],
    "pc_lowrank_sum_exp_workspace": [_i, _i, _i, _i, _i, _i, _p],
    "pc_lowrank_sum_exp_fwd": [_i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _i, _p, _sz, _p],
    "pc_lowrank_sum_exp_bwd": [_i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _p, _sz, _p],
    "pc_lowrank_exp_sum_fwd": [_i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _i, _p, _sz, _p],
    "pc_em_normalize": [_i, _i, _i, _p, _p, _p, _p],
    "pc_hmm_lowrank_workspace": [_i, _i, _i, _i, _i, _i, _p],
    "pc_hmm_lowrank_fwd_bwd": [_i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _p,
                               _sz, _p],
    "pc_lowrank_exp_sum_bwd": [_i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _p, _sz,
                               _p],
}
_STR = {"pc_version", "pc_status_string", "pc_last_error"}

_lib = None


class PCError(RuntimeError):
    """A non-PC_OK status from the library, with its name and pc_last_error() detail."""

    def __init__(self, func: str, status: int, detail: str):
        self.func, self.status, self.detail = func, status, detail
        super().__init__(f"{func}: {STATUS.get(status, status)}: {detail}")


def declared_symbols(header: str = HEADER):
    """Function names the public header declares."""
    with open(header) as fh:
        text = fh.read()
    return sorted(set(re.findall(r"PCSUM_API\s+[\w\s\*]+?\b(pc_\w+)\s*\(", text)))


def load() -> C.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m log_space_sum_gb300.build` "
            "(there is no non-CUDA fallback)")
    lib = C.CDLL(LIB_PATH)
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = C.c_char_p if name in _STR else (C.c_ulonglong if name == "pc_launch_count" else C.c_int)
    _lib = lib
    return lib


def call(name: str, *args) -> None:
    """Calls an entry point and raises PCError on a non-PC_OK status."""
    lib = load()
    st = getattr(lib, name)(*args)
    if st != 0:
        raise PCError(name, st, lib.pc_last_error().decode())
