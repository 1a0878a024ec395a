"""gbf_copy moves every byte, including a tail shorter than 16 bytes."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [16, 1000, 4096 + 7, 1 << 22, (1 << 24) + 3])
def test_copy_exact(n):
    import fusion_add_rmsnorm_gb300 as gbf
    src = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda")
    dst = torch.zeros_like(src)
    gbf.copy(src, dst)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)
