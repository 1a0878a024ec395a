"""Device-side failure detection without a GPU fault: a kernel's bounded wait
on a barrier nothing arrives at gives up after about a second, the error word
reports GBF_ETIMEOUT, and the context keeps working afterwards."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import fusion_add_rmsnorm_gb300 as gbf
    assert gbf.device_status()[0] == gbf.OK
    t0 = time.time()
    gbf.selftest_bounded_wait()
    status, msg = gbf.device_status()           # synchronises the stream
    elapsed = time.time() - t0
    assert status == gbf.ETIMEOUT, msg
    assert 0.5 < elapsed < 30
    assert gbf.device_status()[0] == gbf.OK     # the read cleared the word
    src = torch.arange(1 << 20, dtype=torch.int32, device="cuda")
    dst = torch.zeros_like(src)
    gbf.copy(src, dst)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)
