"""MXFP4 quantisation of bf16 activations on the GPU (the all-FP4 prefill mode's
first step) against the oracle's quantiser: codes and scale bytes bit-exact.
The inputs are bf16, so both sides decide every code exactly (a power-of-two
scaling of a bf16 value is exact in either precision)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _rows():
    rng = np.random.default_rng(17)
    out = []
    # five full-width rows, one magnitude per 32-block (finite in bf16)
    out.append((4096, rng.standard_normal(5 * 4096) * np.repeat(2.0 ** rng.integers(-140, 120, 5 * 128), 32)))
    # three rows of ties of the E2M1 grid at several block scales, both signs
    v = rng.choice([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 3.0, 6.0], 3 * 96) * rng.choice([-1.0, 1.0], 3 * 96)
    v[::32] = 4.0
    out.append((96, v * np.repeat(2.0 ** rng.integers(-100, 100, 9), 32)))
    # zero, negative zero, a lone bf16 subnormal, saturation just below the next power
    special = np.zeros(128)
    special[32:64] = -0.0
    special[64 + 5] = 2.0 ** -133
    special[96:100] = [7.96875, 6.5, -6.0625, 5.96875]
    out.append((128, special))
    return out


def test_quant_mxfp4_matches_oracle():
    import moe_decode_host_gb300 as m

    for K, v in _rows():
        x = torch.tensor(v.reshape(-1, K), dtype=torch.float32).to(torch.bfloat16)
        assert torch.isfinite(x.float()).all()
        rows = x.shape[0]
        xd = x.cuda()
        nib = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
        sc = torch.empty((rows, K // 32), dtype=torch.uint8, device="cuda")
        m.quant_mxfp4(xd, rows, K, nib, sc)
        torch.cuda.synchronize()
        want_n, want_s = oracle.quant_mxfp4(x.float().numpy().astype(np.float64).ravel())
        assert np.array_equal(sc.cpu().numpy().ravel(), want_s)
        assert np.array_equal(nib.cpu().numpy().ravel(), want_n)


def test_quant_mxfp4_arguments():
    import moe_decode_host_gb300 as m

    lib = m.lib
    x = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
    nib = torch.empty((2, 32), dtype=torch.uint8, device="cuda")
    sc = torch.empty((2, 2), dtype=torch.uint8, device="cuda")
    assert lib.moe_quant_mxfp4(x.data_ptr(), 0, 64, nib.data_ptr(), sc.data_ptr(), None) == m.MOE_OK
    assert lib.moe_quant_mxfp4(x.data_ptr(), 2, 48, nib.data_ptr(), sc.data_ptr(), None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_mxfp4(x.data_ptr(), -1, 64, nib.data_ptr(), sc.data_ptr(), None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_mxfp4(None, 2, 64, nib.data_ptr(), sc.data_ptr(), None) == m.MOE_ERR_INVALID_ARG


def test_hardware_e2m1_rounding_matches_the_comparison_rule():
    """The block-scaled kernels round h with the hardware pair conversion; it must
    take the same code as the comparison rule (the OCP rule: nearest, ties to the
    even code, saturating at 6) for every value below 8: each tie point and its two
    float neighbours, a dense grid, tiny and subnormal values, both signs, +-0."""
    import moe_decode_host_gb300 as m

    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 7.0, 7.999999], np.float32)
    near = np.concatenate([np.nextafter(ties, np.float32(0)), ties, np.nextafter(ties, np.float32(8))])
    dense = np.linspace(0, 7.99, 200001, dtype=np.float32)
    tiny = np.array([1e-45, 1e-38, 1e-20, 1e-3, 0.2499], np.float32)
    v = np.concatenate([ties, grid, near, dense, tiny]).astype(np.float32)
    v = np.concatenate([v, -v, np.array([-0.0], np.float32)])
    d = torch.from_numpy(v).cuda()
    out = torch.zeros(2 * v.size, dtype=torch.int32, device="cuda")
    m.debug_e2m1_round(d, out)
    torch.cuda.synchronize()
    o = out.cpu().numpy().reshape(-1, 2)
    bad = np.nonzero(o[:, 0] != o[:, 1])[0]
    assert bad.size == 0, [(float(v[i]), int(o[i, 0]), int(o[i, 1])) for i in bad[:10]]
