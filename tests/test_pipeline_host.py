"""Host-side checks of the pipeline objects (no GPU): tensors handed to the
C ABI must have the shape, dtype, device and layout the calls assume, since
the library cannot see buffer sizes and would read out of bounds."""
import pytest
import torch

from ulysses_sequence_attention_usp_gb300.pipeline import _check_input


def test_accepts_the_expected_tensor():
    _check_input("q", torch.zeros(5, 4, 64, dtype=torch.bfloat16), 5, 4, 64,
                 torch.device("cpu"))


@pytest.mark.parametrize("t,err", [
    (torch.zeros(5, 4, 64), TypeError),                                  # fp32
    (torch.zeros(6, 4, 64, dtype=torch.bfloat16), ValueError),           # rows
    (torch.zeros(5, 2, 64, dtype=torch.bfloat16), ValueError),           # heads
    (torch.zeros(5, 4, 128, dtype=torch.bfloat16), ValueError),          # head dim
    (torch.zeros(4, 5, 64, dtype=torch.bfloat16).transpose(0, 1), ValueError),  # strided
    (None, TypeError),
])
def test_rejects_what_the_kernels_would_misread(t, err):
    with pytest.raises(err):
        _check_input("q", t, 5, 4, 64, torch.device("cpu"))


def test_device_index_only_checked_when_given():
    t = torch.zeros(5, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        _check_input("q", t, 5, 4, 64, torch.device("cuda"))
