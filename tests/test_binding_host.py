"""Host-side checks of the binding's caller-output validation (no GPU: the
checks compare tensors' device, dtype, element count and layout only)."""
import pytest
import torch

rl = pytest.importorskip("linear_recurrence_scan_affine_gb300")
from linear_recurrence_scan_affine_gb300.binding import _out  # noqa: E402


def like(shape=(6, 300), dtype=torch.float32):
    return torch.zeros(shape, dtype=dtype)


def test_accepts_a_contiguous_output_of_the_same_size_and_dtype():
    o = torch.empty(6 * 300)
    assert _out(o, "out", like()) is o
    assert _out(torch.empty(6, 300, dtype=torch.int32), "out", like(dtype=torch.int32)) is not None
    # an explicit dtype overrides the inputs' (compact inputs, float32 output)
    assert _out(torch.empty(6, 300), "out", like(dtype=torch.int16), dtype=torch.float32) is not None


@pytest.mark.parametrize("bad,exc", [
    (torch.empty(5, 300), ValueError),                 # too few elements
    (torch.empty(7, 300), ValueError),                 # too many
    (torch.empty(300, 6).T, ValueError),               # not contiguous
    (torch.empty(6, 300, dtype=torch.float64), TypeError),
    ([0.0] * 1800, TypeError),                         # not a tensor
])
def test_refuses_outputs_the_library_could_overrun_or_misread(bad, exc):
    with pytest.raises(exc):
        _out(bad, "out", like())


def test_refuses_an_output_on_another_device():
    meta = torch.empty(6, 300, device="meta")
    with pytest.raises(ValueError):
        _out(meta, "out", like())
