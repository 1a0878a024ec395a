"""The Python binding's own checks, which run before the C ABI is called and
need no GPU: a tensor argument must be a torch tensor on a CUDA device (dense
and of the call's element type are checked next, on the device)."""
import pytest
import torch


@pytest.fixture(scope="module")
def gbf():
    import fusion_add_rmsnorm_gb300 as g
    return g


def test_host_tensors_are_refused_before_the_call(gbf):
    x = torch.zeros(2, 8, dtype=torch.bfloat16)
    q = torch.zeros(2, 8, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        gbf.add_rmsnorm_fp8(x, x, x, q, gbf.NORM_NOWEIGHT)
    with pytest.raises(ValueError, match="CUDA"):
        gbf.gated_act(torch.zeros(2, 16, dtype=torch.bfloat16), x)


def test_non_tensors_are_refused(gbf):
    with pytest.raises(TypeError, match="torch.Tensor"):
        gbf.copy([1, 2, 3], [4, 5, 6], nbytes=3)


def test_optional_arguments_pass_through(gbf):
    assert gbf._ptr(None, torch.bfloat16, "bias") is None
