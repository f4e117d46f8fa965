"""A device-side wait that nothing completes runs out at its deadline, reports
MOE_ERR_TIMEOUT with a record of where it waited, and leaves the context usable:
how the pipelined kernels report a lost producer without faulting or hanging the
GPU (the flag is simply never set)."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def test_unfinished_phase_times_out_and_reports():
    import moe_decode_host_gb300 as m

    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    diag = torch.zeros(16, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert m.lib.moe_debug_wait_timeout(status.data_ptr(), diag.data_ptr(), None) == m.MOE_OK
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == m.MOE_ERR_TIMEOUT
    d = diag.cpu().tolist()
    assert d[0] == 1 and d[1] == 0 and d[2] == 0 and d[3] == 1  # set; block 0, warp 0, a "stage full" wait
    assert d[4] == 0 and d[5] == 0  # ring slot 0, waited for parity 0
    assert 1.5 < waited < 60.0
    # the context is still usable
    x = torch.arange(1000, dtype=torch.float32, device="cuda")
    assert float(x.sum().item()) == 499500.0
