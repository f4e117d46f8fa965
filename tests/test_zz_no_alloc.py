"""moe_grouped_ffn_noalloc: the grouped expert FFN for callers that cannot allocate
device memory (an engine that gave all free HBM to its own pools, code running
during a global-mode stream capture, embedders with their own allocator).  Its
workspace is a fixed array inside the library, and it runs the same kernels as the
regular entry point on the same inputs, so its results must equal the regular
entry point's bit for bit, call after call, with nothing allocated by the call.

This file is collected after the layer parity tests on purpose; it also passes when
run alone in a fresh process (the first call on the device looks up the array's
address)."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import LayerFixture

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _logits(T, E, seed, favour=()):
    lg = synth.gen_logits_uniform(T, E, seed=seed)
    for e in favour:  # every token picks these experts (their buckets hold all T tokens)
        lg[:, e] += 12.0
    return torch.from_numpy(lg).cuda()


def _both(fx, T, seed, favour=()):
    """Routes one batch, gathers, then runs the regular FFN and the no-allocation
    FFN on the same inputs; returns both y tensors on the host."""
    import moe_decode_host_gb300 as m

    logits = _logits(T, fx.E, seed, favour)
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
    counts = buf.counts.cpu().numpy()
    return y_ref.cpu().numpy(), y_na.cpu().numpy(), counts


@pytest.mark.parametrize("H,I,E,n_hot,k,T,zero_copy", [
    (256, 512, 16, 12, 2, 4, False),       # the small test layer
    (4096, 3072, 16, 12, 6, 8, False),     # full-size experts
    (4096, 3072, 16, 12, 6, 8, True),      # cold experts read in place on the layer's copy stream
])
def test_noalloc_matches_regular_entry_point_twice(H, I, E, n_hot, k, T, zero_copy):
    fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=E - n_hot, k=k, seed=77 + H, zero_copy=zero_copy)
    for call in range(2):
        y_ref, y_na, counts = _both(fx, T, seed=1000 * call + T)
        assert np.all(np.isfinite(y_na))
        assert np.array_equal(y_na, y_ref), call
    fx.layer.close()


def test_noalloc_tensor_core_buckets_at_the_size_limit():
    """H=4096, I=3072, k=6: the static array holds the workspace of 68 tokens
    (2*max(H, I) + 4*I + 4 bytes per pick, sections 256-byte aligned).  Two experts
    get all 68 tokens, so their buckets run on the tensor-core kernel through the
    static array; 69 tokens are rejected."""
    import moe_decode_host_gb300 as m

    H, I, E, n_hot, k = 4096, 3072, 16, 12, 6
    fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=E - n_hot, k=k, seed=31)
    assert fx.layer.ffn_workspace_bytes(68) <= m.MOE_NOALLOC_SCRATCH_BYTES < fx.layer.ffn_workspace_bytes(69)
    for call in range(2):
        y_ref, y_na, counts = _both(fx, 68, seed=500 + call, favour=(3, 13))  # 3 hot, 13 cold
        assert counts[3] == 68 and counts[13] == 68
        assert np.array_equal(y_na, y_ref), call
    dummy = torch.zeros(69 * k, dtype=torch.int32, device="cuda")
    rc = m.lib.moe_grouped_ffn_noalloc(fx.layer.handle, dummy.data_ptr(), 69, dummy.data_ptr(), dummy.data_ptr(),
                                       dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), None)
    assert rc == m.MOE_ERR_SCRATCH_TOO_SMALL
    fx.layer.close()


def test_noalloc_call_leaves_free_device_memory_unchanged():
    """A first call on a fresh layer allocates nothing: free device memory is the
    same before and after it (the library's module, which holds the array, is
    loaded by an earlier call, as it is once per process)."""
    import moe_decode_host_gb300 as m

    warm = LayerFixture(H=256, I=512, E=16, n_hot=12, n_cold=4, k=2, seed=3)
    _both(warm, 4, seed=9)
    fx = LayerFixture(H=256, I=512, E=16, n_hot=12, n_cold=4, k=2, seed=4)
    T = 6
    logits = _logits(T, fx.E, 21)
    x = synth.gen_x(T, fx.H, seed=22).cuda()
    buf = m.StepBuffers(fx.layer, T)
    m.moe_route(fx.layer, logits, T, buf.topk_ids, buf.topk_w, buf.counts, buf.offsets, buf.entries)
    m.cold_gather(fx.layer, buf.topk_ids, T, buf.phys_ids, buf.cold_list, buf.n_cold_picked)
    m.moe_gather_join(fx.layer)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    m.moe_grouped_ffn_noalloc(fx.layer, x, T, buf.phys_ids, buf.counts, buf.offsets, buf.entries, buf.y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert fx.layer.status() == 0
    assert bool(torch.isfinite(buf.y[:T * fx.k]).all())
    fx.layer.close()
    warm.layer.close()


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
