"""Host-side argument checks of the Python binding (CPU only: they raise
before any call reaches the library)."""
import pytest
import torch

from sliding_window_attention_prefill_gb300 import swa


def test_out_is_new_when_not_given():
    q = torch.zeros(2, 3, 8, dtype=torch.bfloat16)
    o = swa._out(None, q, torch.bfloat16)
    assert o.shape == q.shape and o.dtype == q.dtype and o.data_ptr() != q.data_ptr()


@pytest.mark.parametrize("shape", [(2, 3, 4), (6, 8), (2, 3, 8, 1), (1, 3, 8)])
def test_out_of_another_shape_is_refused(shape):
    # a smaller or reshaped buffer would take writes past its end
    q = torch.zeros(2, 3, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="shape of q"):
        swa._out(torch.zeros(shape, dtype=torch.bfloat16), q, torch.bfloat16)


def test_out_of_the_right_shape_still_needs_a_cuda_tensor_of_the_type():
    q = torch.zeros(2, 3, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        swa._out(torch.zeros(2, 3, 8, dtype=torch.float16), q, torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        swa._out(torch.zeros(2, 3, 8, dtype=torch.bfloat16), q, torch.bfloat16)
    with pytest.raises(TypeError):
        swa._out([0.0] * 48, q, torch.bfloat16)
