"""The Python binding's host-side checks (no GPU needed): the removed flags and
unknown precision modes (pyjuice PR #62, Breaking change and Tests), and the
refusal to run on CPU tensors (there is no CPU path)."""
import pytest
import torch

import log_space_sum_gb300 as pc


def test_removed_flags_raise_type_error_naming_precision():
    t = torch.zeros(1, 2, 2)
    for fn, args in ((pc.sum_layer_fwd, (t, t[0])), (pc.sum_layer_bwd, (t, t[0], t, t)),
                     (pc.hmm_fwd_bwd, (t, t, t, t))):
        for flag in ("force_use_bf16", "force_use_fp32"):
            with pytest.raises(TypeError, match="precision="):
                fn(*args, **{flag: True})


def test_removed_flags_false_is_accepted_and_ignored():
    t = torch.zeros(1, 2, 2)
    # False passes the flag check; the call then stops at the CPU-tensor check
    with pytest.raises(ValueError, match="CUDA tensor"):
        pc.sum_layer_fwd(t, t[0], force_use_bf16=False, force_use_fp32=False)


def test_unknown_precision():
    with pytest.raises(ValueError, match="'auto'"):
        pc.precision_code("fp16")
    with pytest.raises(TypeError):
        pc.precision_code(1.0)
    assert [pc.precision_code(m) for m in ("auto", "tf32", "fp32")] == [0, 1, 2]


def test_cpu_tensors_are_refused():
    t = torch.zeros(1, 4, 4)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pc.sum_layer_fwd(t, t[0])
