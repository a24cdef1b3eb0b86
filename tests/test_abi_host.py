"""The C ABI without a GPU: the library loads, exports every function the public
header declares, and rejects bad arguments with the documented status before
launching anything (no CUDA call is reached in these cases)."""
import ctypes as C

import pytest

from log_space_sum_gb300 import _native as N
from log_space_sum_gb300 import build as B


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.load()


def test_every_declared_symbol_is_exported(lib):
    names = N.declared_symbols()
    assert {"pc_sum_layer_fwd", "pc_sum_layer_bwd", "pc_hmm_fwd_bwd"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name
        assert name in N.SIGNATURES, f"{name} has no ctypes signature"


def test_version_and_status_strings(lib):
    assert lib.pc_version().decode().startswith("pcsum")
    for code, name in N.STATUS.items():
        assert lib.pc_status_string(code).decode() == name


def _size():
    return C.c_size_t(0)


def test_unknown_precision_names_the_modes(lib):
    nb = _size()
    st = lib.pc_sum_layer_workspace(1, 8, 8, 8, 7, C.byref(nb))
    assert N.STATUS[st] == "PC_ERR_UNKNOWN_PRECISION"
    msg = lib.pc_last_error().decode()
    assert "PC_PREC_AUTO" in msg and "PC_PREC_FP32" in msg
    st = lib.pc_hmm_workspace(8, 4, 4, 4, -1, C.byref(nb))
    assert N.STATUS[st] == "PC_ERR_UNKNOWN_PRECISION"


@pytest.mark.parametrize("args,status", [
    ((0, 8, 8, 8), "PC_ERR_SHAPE"),
    ((1, -1, 8, 8), "PC_ERR_SHAPE"),
    ((1, 8, 0, 8), "PC_ERR_SHAPE"),
    ((1, 8, 8, 1 << 24), "PC_ERR_SHAPE"),
])
def test_layer_shape_checks(lib, args, status):
    nb = _size()
    assert N.STATUS[lib.pc_sum_layer_workspace(*args, 0, C.byref(nb))] == status


def test_layer_workspace_grows_with_precision(lib):
    sizes = []
    for prec in range(3):
        nb = _size()
        assert lib.pc_sum_layer_workspace(1, 1024, 1024, 128, prec, C.byref(nb)) == 0
        sizes.append(nb.value)
    assert sizes[0] < sizes[1] < sizes[2]


def test_layer_argument_errors_before_launch(lib):
    fake = C.c_void_p(0x1000)
    # NULL theta
    st = lib.pc_sum_layer_fwd(1, 8, 8, 8, None, fake, 0, fake, 0, fake, 1 << 30, None)
    assert N.STATUS[st] == "PC_ERR_NULL"
    # groups that overlap
    st = lib.pc_sum_layer_fwd(2, 8, 8, 8, fake, fake, 4, fake, 0, fake, 1 << 30, None)
    assert N.STATUS[st] == "PC_ERR_SHAPE"
    assert "overlap" in lib.pc_last_error().decode()
    # workspace missing / too small
    st = lib.pc_sum_layer_fwd(1, 8, 8, 8, fake, fake, 0, fake, 0, None, 0, None)
    assert N.STATUS[st] == "PC_ERR_WORKSPACE"
    st = lib.pc_sum_layer_fwd(1, 8, 8, 8, fake, fake, 0, fake, 0, fake, 16, None)
    assert N.STATUS[st] == "PC_ERR_WORKSPACE"
    # backward: NULL flows input
    st = lib.pc_sum_layer_bwd(1, 8, 8, 8, fake, fake, 0, fake, None, fake, fake, 0, 0, fake, 1 << 30, None)
    assert N.STATUS[st] == "PC_ERR_NULL"
    # backward with neither output requested is a no-op (nothing to launch)
    st = lib.pc_sum_layer_bwd(1, 8, 8, 8, fake, fake, 0, fake, fake, None, None, 0, 0, None, 0, None)
    assert st == 0


def test_hmm_argument_errors_before_launch(lib):
    fake = C.c_void_p(0x1000)
    nb = _size()
    assert lib.pc_hmm_workspace(4096, 32, 1024, 512, 0, C.byref(nb)) == 0
    assert nb.value > 4096 * 4096 * 2
    assert N.STATUS[lib.pc_hmm_workspace(0, 32, 1024, 512, 0, C.byref(nb))] == "PC_ERR_SHAPE"
    assert N.STATUS[lib.pc_hmm_workspace(20000, 32, 1024, 512, 0, C.byref(nb))] == "PC_ERR_SHAPE"
    st = lib.pc_hmm_fwd_bwd(8, 4, 4, 4, None, fake, fake, fake, fake, None, None, None, 0, 0, fake,
                            1 << 30, None)
    assert N.STATUS[st] == "PC_ERR_NULL"
    st = lib.pc_hmm_fwd_bwd(8, 4, 4, 4, fake, fake, fake, fake, fake, None, None, None, 0, 0, fake,
                            8, None)
    assert N.STATUS[st] == "PC_ERR_WORKSPACE"


def test_profile_capacity_check(lib):
    assert N.STATUS[lib.pc_profile_start(0)] == "PC_ERR_SHAPE"
    # every output but the count may be NULL; a NULL count is refused before any CUDA call
    assert N.STATUS[lib.pc_profile_stop(None, None, None, None, None, 4)] == "PC_ERR_NULL"


def test_split_workspaces_hold_the_partial_products(lib):
    # the single-group layer at M = N = 1024, B = 128 runs its forward over 8 K ranges: the
    # workspace holds the 8 x M x B float32 partial sums that G = 2 groups do not need
    one, two = _size(), _size()
    assert lib.pc_sum_layer_workspace(1, 1024, 1024, 128, 0, C.byref(one)) == 0
    assert lib.pc_sum_layer_workspace(2, 1024, 1024, 128, 0, C.byref(two)) == 0
    assert one.value - two.value / 2 >= 8 * 1024 * 128 * 4 - 4096  # two groups: twice the rest
    # the HMM with H = 1024, T = 64, B = 512 runs its stacked dA contraction over 4 K ranges
    # (4 x H x H float32 partial products); with B = 500 the ranges do not divide K evenly
    small, odd = _size(), _size()
    assert lib.pc_hmm_workspace(1024, 64, 1024, 512, 0, C.byref(small)) == 0
    assert lib.pc_hmm_workspace(1024, 64, 1024, 500, 0, C.byref(odd)) == 0
    assert small.value - odd.value >= 4 * 1024 * 1024 * 4 - (1 << 20)


def test_em_normalize_argument_errors_before_launch(lib):
    fake = C.c_void_p(0x1000)
    assert N.STATUS[lib.pc_em_normalize(1, 4, 4, None, None, fake, None)] == "PC_ERR_NULL"
    assert N.STATUS[lib.pc_em_normalize(1, 4, 4, fake, None, None, None)] == "PC_ERR_NULL"
    assert N.STATUS[lib.pc_em_normalize(0, 4, 4, fake, None, fake, None)] == "PC_ERR_SHAPE"
    assert N.STATUS[lib.pc_em_normalize(1, 4, 0, fake, fake, fake, None)] == "PC_ERR_SHAPE"
    assert N.STATUS[lib.pc_em_normalize(1 << 16, 1 << 16, 4, fake, None, fake, None)] == "PC_ERR_SHAPE"


def test_lowrank_sum_exp_argument_errors_before_launch(lib):
    fake = C.c_void_p(0x1000)
    nb = _size()
    assert lib.pc_lowrank_sum_exp_workspace(1024, 1024, 16, 64, 1, 0, C.byref(nb)) == 0
    fwd_only = _size()
    assert lib.pc_lowrank_sum_exp_workspace(1024, 1024, 16, 64, 0, 0, C.byref(fwd_only)) == 0
    assert 0 < fwd_only.value < nb.value
    assert N.STATUS[lib.pc_lowrank_sum_exp_workspace(8, 8, 0, 4, 0, 0, C.byref(nb))] == "PC_ERR_SHAPE"
    assert N.STATUS[lib.pc_lowrank_sum_exp_workspace(8, 8, 4, 4, 0, 9, C.byref(nb))] == "PC_ERR_UNKNOWN_PRECISION"
    st = lib.pc_lowrank_sum_exp_fwd(8, 8, 4, 4, fake, fake, fake, fake, None, fake, 0, fake, 1 << 30, None)
    assert N.STATUS[st] == "PC_ERR_NULL"
    st = lib.pc_lowrank_sum_exp_fwd(8, 8, 4, 4, fake, fake, fake, fake, fake, fake, 0, fake, 16, None)
    assert N.STATUS[st] == "PC_ERR_WORKSPACE"
    st = lib.pc_lowrank_sum_exp_bwd(8, 8, 4, 4, fake, fake, fake, fake, None, None, None, None, None, None, 0, 0, 0,
                                    fake, 1 << 30, None)
    assert N.STATUS[st] == "PC_ERR_NULL"


def test_hmm_lowrank_argument_errors_before_launch(lib):
    fake = C.c_void_p(0x1000)
    nb = _size()
    assert lib.pc_hmm_lowrank_workspace(1024, 64, 1024, 64, 16, 0, C.byref(nb)) == 0
    assert N.STATUS[lib.pc_hmm_lowrank_workspace(64, 4, 8, 4, 65, 0, C.byref(nb))] == "PC_ERR_UNSUPPORTED"
    assert N.STATUS[lib.pc_hmm_lowrank_workspace(64, 0, 8, 4, 4, 0, C.byref(nb))] == "PC_ERR_SHAPE"
    args = [None] * 13
    st = lib.pc_hmm_lowrank_fwd_bwd(64, 4, 8, 4, 4, None, fake, fake, fake, fake, fake, fake, *args[:6], 0, 0,
                                    fake, 1 << 30, None)
    assert N.STATUS[st] == "PC_ERR_NULL"
    st = lib.pc_hmm_lowrank_fwd_bwd(64, 4, 8, 4, 4, fake, fake, fake, fake, None, None, fake, *args[:6], 0, 0,
                                    fake, 1 << 30, None)
    assert N.STATUS[st] == "PC_ERR_NULL"                 # factors required when T > 1
    st = lib.pc_hmm_lowrank_fwd_bwd(64, 4, 8, 4, 4, fake, fake, fake, fake, fake, fake, fake, *args[:6], 0, 0,
                                    fake, 64, None)
    assert N.STATUS[st] == "PC_ERR_WORKSPACE"
