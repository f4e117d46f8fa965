"""moe_grouped_ffn_noalloc: the grouped expert FFN for callers that cannot allocate
device memory (an engine that gave all free HBM to its own pools, code running
during a global-mode stream capture, embedders with their own allocator).  Its
workspace is a fixed array inside the library, so its results must match the
regular entry point's, call after call, with nothing allocated by the call.

This file is collected after the layer parity tests on purpose; it also passes when run alone in a fresh
process (the first call on the device looks up the array's address)."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import LayerFixture, rel_l2

pytestmark = pytest.mark.gpu

OUT_TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _both(fx, T, seed):
    """Routes one batch, gathers, then runs the regular FFN and the no-allocation
    FFN on the same inputs; returns both y tensors."""
    import moe_decode_host_gb300 as m

    logits = torch.from_numpy(synth.gen_logits_uniform(T, fx.E, seed=seed)).cuda()
    x = synth.gen_x(T, fx.H, seed=seed + 1).cuda()
    buf = m.StepBuffers(fx.layer, T)
    m.moe_route(fx.layer, logits, T, buf.topk_ids, buf.topk_w, buf.counts, buf.offsets, buf.entries)
    m.cold_gather(fx.layer, buf.topk_ids, T, buf.phys_ids, buf.cold_list, buf.n_cold_picked)
    m.moe_grouped_ffn(fx.layer, x, T, buf.phys_ids, buf.counts, buf.offsets, buf.entries, buf.y, buf.workspace)
    y_ref = buf.y.clone()
    y_na = torch.full_like(buf.y, float("nan"))
    m.moe_grouped_ffn_noalloc(fx.layer, x, T, buf.phys_ids, buf.counts, buf.offsets, buf.entries, y_na)
    torch.cuda.synchronize()
    assert fx.layer.status() == 0, fx.layer.diag().tolist()
    return y_ref.cpu().numpy(), y_na.cpu().numpy()


@pytest.mark.parametrize("H,I,E,n_hot,k,T", [
    (256, 512, 16, 12, 2, 4),       # the small test layer
    (4096, 3072, 16, 12, 6, 8),     # full-size experts
])
def test_noalloc_matches_regular_entry_point_twice(H, I, E, n_hot, k, T):
    fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=E - n_hot, k=k, seed=77 + H)
    for call in range(2):
        y_ref, y_na = _both(fx, T, seed=1000 * call + T)
        assert np.all(np.isfinite(y_na))
        assert rel_l2(y_na, y_ref) <= OUT_TOL
    fx.layer.close()


def test_noalloc_rejects_batches_beyond_its_array():
    import moe_decode_host_gb300 as m

    fx = LayerFixture(H=256, I=512, E=16, n_hot=12, n_cold=4, k=2, seed=5)
    T = 4096  # needs far more workspace than the static array holds
    assert fx.layer.ffn_workspace_bytes(T) > m.MOE_NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = m.lib.moe_grouped_ffn_noalloc(fx.layer.handle, dummy.data_ptr(), T, dummy.data_ptr(), dummy.data_ptr(),
                                       dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), None)
    assert rc == m.MOE_ERR_SCRATCH_TOO_SMALL
    fx.layer.close()
