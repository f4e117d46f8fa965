"""CPU checks of the C-ABI library: it builds, loads, exports every function that
include/moehost.h declares, and rejects bad arguments on the host before any
CUDA call (no compute, no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "moehost.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def mlib():
    import __graft_entry__

    __graft_entry__.build()
    import moe_decode_host_gb300 as m

    return m


def test_header_declares_the_five_entry_points():
    names = _declared_functions()
    for n in ("moe_route", "cold_gather", "moe_grouped_ffn", "moe_combine", "residency_update"):
        assert n in names


def test_library_exports_every_declared_symbol(mlib):
    lib = ctypes.CDLL(mlib.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_side_argument_checks(mlib):
    lib = mlib.lib
    assert lib.moe_expert_bytes(100, 128) == 0
    assert lib.moe_expert_bytes(4096, 3072) == 20054016
    assert lib.moe_expert_bytes(256, 512) == 208896
    out = ctypes.c_void_p()
    assert lib.moe_scratch_create(-1, 208896, None, ctypes.byref(out)) == mlib.MOE_ERR_INVALID_ARG
    assert lib.moe_scratch_create(4, 208896, None, ctypes.byref(out)) == mlib.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(None, None, -1, 2, 256, None, 0, None) == mlib.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(None, None, 4, 0, 256, None, 0, None) == mlib.MOE_ERR_INVALID_ARG
    assert lib.moe_route(None, None, 1, None, None, None, None, None, None) == mlib.MOE_ERR_INVALID_ARG
    assert lib.cold_gather(None, None, 1, None, None, None, None) == mlib.MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_ffn(None, None, 1, None, None, None, None, None, None, 0, None) == \
        mlib.MOE_ERR_INVALID_ARG
    n = ctypes.c_int32()
    assert lib.residency_update(None, ctypes.byref(n), None) == mlib.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_destroy(None) == mlib.MOE_ERR_INVALID_ARG
    p = mlib.moe_params(16, 2, 256, 512, 12, 4, 0, 16, 8, 3.0)
    loc = (ctypes.c_int32 * 16)(*range(16))
    bad = mlib.moe_params(16, 0, 256, 512, 12, 4, 0, 16, 8, 3.0)
    assert lib.moe_layer_create(ctypes.byref(bad), None, None, None, loc, ctypes.byref(out)) == \
        mlib.MOE_ERR_INVALID_ARG
    bad = mlib.moe_params(16, 2, 200, 512, 12, 4, 0, 16, 8, 3.0)
    assert lib.moe_layer_create(ctypes.byref(bad), None, None, None, loc, ctypes.byref(out)) == \
        mlib.MOE_ERR_INVALID_ARG
    bad = mlib.moe_params(16, 2, 256, 512, 12, 5, 0, 16, 8, 3.0)
    assert lib.moe_layer_create(ctypes.byref(bad), None, None, None, loc, ctypes.byref(out)) == \
        mlib.MOE_ERR_INVALID_ARG
    for field, value in (("host_mirror", 2), ("zero_copy", 2), ("zero_copy", -1), ("renorm", 3)):
        bad = mlib.moe_params(16, 2, 256, 512, 12, 4, 0, 16, 8, 3.0)
        setattr(bad, field, value)
        assert lib.moe_layer_create(ctypes.byref(bad), None, None, None, loc, ctypes.byref(out)) == \
            mlib.MOE_ERR_INVALID_ARG, field
    # cold experts but no scratch
    assert lib.moe_layer_create(ctypes.byref(p), None, None, None, loc, ctypes.byref(out)) == \
        mlib.MOE_ERR_INVALID_ARG
    # a map that is not a bijection
    dup = (ctypes.c_int32 * 16)(*([0] + list(range(1, 15)) + [0]))
    assert lib.moe_layer_create(ctypes.byref(p), None, None, None, dup, ctypes.byref(out)) == \
        mlib.MOE_ERR_INVALID_ARG
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, -99):
        assert lib.moe_strerror(code)


def test_package_has_no_oracle_dependency():
    pkg = os.path.join(ROOT, "moe_decode_host_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "moe_oracle" not in src, f


def _random_window(rng, E, n_hot):
    loc = rng.permutation(E).astype("int32")
    kind = rng.integers(0, 3)
    if kind == 0:    # sparse window: most experts unpicked, small counts (many ties)
        counts = rng.binomial(3, 0.15, E)
    elif kind == 1:  # skewed window
        counts = rng.zipf(1.5, E).clip(max=200) - 1
    else:            # counts on the hysteresis boundary: cold = 3 x hot exactly
        counts = rng.integers(0, 4, E) * rng.choice([1, 3], E)
    return counts.astype("int32"), loc


def test_residency_plan_matches_the_oracle_on_random_windows(mlib):
    """The library's host planner (the one residency_update applies) against the
    oracle's residency rule: identical placements and swap lists, bit for bit."""
    import numpy as np

    import oracle

    rng = np.random.default_rng(2024)
    cases = 0
    for _ in range(400):
        E = int(rng.choice([8, 16, 64, 384]))
        n_hot = int(rng.integers(0, E + 1))
        max_swaps = int(rng.choice([0, 1, 2, 8, 64]))
        hyst = float(rng.choice([0.0, 1.5, 3.0, 6.0]))
        counts, loc = _random_window(rng, E, n_hot)
        got_loc, got_pro, got_dem = mlib.residency_plan(counts, loc, n_hot, max_swaps, hyst)
        want_loc, want_pro, want_dem = oracle.residency(counts, loc, n_hot, max_swaps, hyst)
        assert np.array_equal(got_loc, want_loc)
        assert np.array_equal(got_pro, want_pro) and np.array_equal(got_dem, want_dem)
        cases += int(got_pro.size > 0)
    assert cases > 100  # most windows make at least one swap


def test_residency_plan_rejects_bad_input(mlib):
    import numpy as np

    lib = mlib.lib
    ok_counts = np.zeros(8, np.int32)
    out = np.empty(8, np.int32)
    pro = np.empty(8, np.int32)
    dem = np.empty(8, np.int32)
    P = mlib._lib.ptr

    def plan(counts, loc, n_hot=4, max_swaps=8, hyst=3.0):
        return lib.moe_residency_plan(P(counts), P(loc), counts.size, n_hot, max_swaps, hyst, P(out), P(pro), P(dem))

    assert plan(ok_counts, np.arange(8, dtype=np.int32)) == 0
    assert plan(ok_counts, np.array([0, 1, 2, 3, 4, 5, 6, 6], np.int32)) == mlib.MOE_ERR_INVALID_ARG  # not a permutation
    assert plan(ok_counts, np.array([0, 1, 2, 3, 4, 5, 6, 8], np.int32)) == mlib.MOE_ERR_INVALID_ARG  # out of range
    bad = ok_counts.copy()
    bad[3] = -1
    assert plan(bad, np.arange(8, dtype=np.int32)) == mlib.MOE_ERR_INVALID_ARG
    assert plan(ok_counts, np.arange(8, dtype=np.int32), n_hot=9) == mlib.MOE_ERR_INVALID_ARG
    assert plan(ok_counts, np.arange(8, dtype=np.int32), max_swaps=65) == mlib.MOE_ERR_INVALID_ARG
    assert plan(ok_counts, np.arange(8, dtype=np.int32), hyst=float("nan")) == mlib.MOE_ERR_INVALID_ARG
    assert plan(ok_counts, np.arange(8, dtype=np.int32), hyst=-1.0) == mlib.MOE_ERR_INVALID_ARG


def test_quant_mxfp4_host_checks(mlib):
    lib = mlib.lib
    assert lib.moe_quant_mxfp4(None, 0, 64, None, None, None) == mlib.MOE_OK  # nothing to do
    assert lib.moe_quant_mxfp4(None, 2, 64, None, None, None) == mlib.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_mxfp4(None, 2, 48, None, None, None) == mlib.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_mxfp4(None, -1, 64, None, None, None) == mlib.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_mxfp4(None, 1, 0, None, None, None) == mlib.MOE_ERR_INVALID_ARG
