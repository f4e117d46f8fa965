"""The bench's CPU oracle leg stays bounded on large batches: each oracle call
takes the first few tokens of a seeded step (the oracle runs every pick on its
own token, so its time per token does not depend on the batch)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _cfg(T, routing="uniform"):
    return {"name": "tiny", "H": 128, "I": 128, "E": 16, "k": 2, "T": T, "routing": routing, "s": 1.1}


def test_prefill_step_is_sampled_by_its_first_tokens():
    v, tok, secs, sample = bench.oracle_tokens_per_s(_cfg(8192), 0.0, seed_tag="t")
    assert tok == bench.ORACLE_TOKENS_PER_CALL
    assert v > 0 and secs > 0
    assert "the first 8 of a 8192-token step" in sample


def test_small_batches_run_whole_steps():
    for T in (1, 6):
        v, tok, secs, sample = bench.oracle_tokens_per_s(_cfg(T, "verify" if T == 6 else "zipf"), 0.0)
        assert tok == T
        assert f"the first {T} of a {T}-token step" in sample


def test_first_tokens_route_as_in_the_whole_step():
    import oracle
    import synth

    E, k = 16, 2
    full = synth.gen_logits_uniform(8192, E, seed=5)
    _, ids_full, w_full, _, _, _ = oracle.route(full, k)
    _, ids_head, w_head, _, _, _ = oracle.route(np.ascontiguousarray(full[:8]), k)
    assert np.array_equal(ids_full[:8], ids_head)
    assert np.array_equal(w_full[:8], w_head)


def _args(*argv):
    old = sys.argv
    sys.argv = ["bench.py", *argv]
    try:
        return bench.parse()
    finally:
        sys.argv = old


def test_default_run_is_the_batch1_decode_layer():
    a = _args()
    assert (a.gpus, a.config, a.impl) == (1, "c1", "ours")
    assert a.warmup >= 3 and a.steps > 0
    c = bench.workload(a)
    assert (c["H"], c["I"], c["E"], c["n_hot"], c["n_cold"], c["k"], c["T"]) == (4096, 3072, 384, 255, 129, 6, 1)
    assert c["routing"] == "uniform" and c["layers"] == 1
    assert c["no_res"] and not c["mirror"] and not c["zero_copy"]
    # the same line carries the skewed decode batches of 8 and 32 tokens
    assert [(T, n) for T, n in bench.PER_BATCH] == [(8, "c2"), (32, "c2")]
    cb = bench.workload(a, config="c2", batch=32)
    assert (cb["T"], cb["routing"], cb["s"], cb["n_hot"], cb["n_cold"]) == (32, "zipf", 1.1, 255, 129)
    assert cb["no_res"]


def test_workload_shapes_of_the_other_configs():
    c = bench.workload(_args("--config", "c2", "--batch", "32", "--skew", "1.5"))
    assert (c["T"], c["routing"], c["s"], c["E"], c["n_hot"]) == (32, "zipf", 1.5, 384, 255)
    a = _args("--config", "c3")
    c = bench.workload(a)
    assert c["layers"] == 20 and c["swap_every"] == 16 and not c["no_res"]
    assert (c["swap_every_steps"], c["max_swaps"], c["hysteresis"]) == (16, 8, 3.0)
    assert not c["mirror"]  # 20 layers keep the in-place exchange
    c = bench.workload(_args("--config", "c4"))
    assert (c["T"], c["n_hot"], c["n_cold"], c["prefill"]) == (8192, 384, 0, "fp4")
    assert bench.workload(_args("--config", "c4", "--prefill", "f16"))["prefill"] == "f16"
    c = bench.workload(_args("--config", "v1"))
    assert (c["T"], c["routing"]) == (6, "verify")


def test_prefill_targets_on_the_8192_token_layer():
    """At 8192 tokens x top-6 over 384 experts of H=4096, I=3072: 3.71 TFLOP on
    7.70 GB of weights, 67 MB of x in and 805 MB of per-pick fp32 outputs, about
    433 flop/B; at the measured 6751.7 GB/s that caps any kernel near 2.92 PFLOP/s."""
    flops = 2.0 * 3 * 4096 * 3072 * 8192 * 6
    algo = 384 * 20054016 + 8192 * 4096 * 2 + 8192 * 6 * 4096 * 4
    t = bench.prefill_targets(flops, algo, 1.5, 12000.0, "probe", 6751.7)
    assert abs(flops - 3.71e12) < 0.01e12
    assert abs(t["flop_per_byte"] - 433) < 2
    assert abs(t["hbm_bound_cap_tflops"] - 2924) < 20
    assert abs(t["achieved_tflops"] - 2473.9) < 1
    assert t["mxfp4_peak_tflops"] == 12000.0 and t["mxfp4_peak_kind"] == "probe"
    assert abs(t["frac_of_mxfp4_peak"] - 2473.9 / 12000.0) < 1e-4
    assert abs(t["cap_frac_of_mxfp4_peak"] - t["hbm_bound_cap_tflops"] / 12000.0) < 1e-12


def test_skew_share_statistic():
    import numpy as np

    ident = np.arange(100)[None, :]
    # 100 experts: picks only on experts 0..72, ranked first by the generator -> all on the top 73%
    c = np.zeros((3, 1, 100), np.int32)
    c[:, :, :73] = 1
    assert bench.skew_share(c, ident) == 1.0
    # uniform picks -> 73%
    assert abs(bench.skew_share(np.ones((5, 1, 100), np.int32), ident) - 0.73) < 1e-12
    # the generator's ranking decides, not the sample: a few picks on low-ranked experts
    # count as off the top even though they are the only experts picked
    c = np.zeros((1, 1, 100), np.int32)
    c[0, 0, 90:96] = 1
    assert bench.skew_share(c, ident) == 0.0
    # per layer, each layer's own ranking (layer 1 ranks experts in reverse)
    c = np.zeros((1, 2, 100), np.int32)
    c[0, 0, :73] = 2
    c[0, 1, 27:] = 2
    rank = np.stack([np.arange(100), np.arange(100)[::-1]])
    assert bench.skew_share(c, rank) == 1.0


def test_repetition_split_and_spread():
    assert bench.repetition_bounds(8000) == [0, 1600, 3200, 4800, 6400, 8000]
    assert bench.repetition_bounds(7) == [0, 1, 3, 4, 6, 7]
    assert bench.repetition_bounds(3) == [0, 1, 2, 3]
    assert bench.repetition_bounds(1) == [0, 1]
    b = bench.repetition_bounds(10)
    r = bench.repetition_spread(b, [2.0, 2.0, 4.0, 1.0, 2.0], 4)  # 2 steps x 4 tokens each
    assert r["tokens_per_s"] == [4000.0, 4000.0, 2000.0, 8000.0, 4000.0]
    assert (r["median"], r["min"], r["max"], r["n"]) == (4000.0, 2000.0, 8000.0, 5)


def test_step_launches_follow_the_library_paths():
    """The launch count the bench claims per layer-step: route, remap and the two
    copy launches, the FFN's prep and phases on the kernels the library picks, the
    combine."""
    import bench

    c1 = dict(T=1, n_cold=129, decode_kind=1)  # GEMV: prep, (gate/up + h prescale + down) x 2 classes
    assert bench.ffn_terms(c1) == 0
    assert bench.step_launches(c1) == 1 + 3 + (1 + 2 * 3) + 1
    assert bench.ffn_terms(dict(T=1, n_cold=129)) == 4  # the default at one token
    c2 = dict(T=32, n_cold=129)            # block-scaled 4-term: prep, 2 phases x 2 classes
    assert bench.ffn_terms(c2) == 4
    assert bench.step_launches(c2) == 1 + 3 + 5 + 1
    assert bench.ffn_terms(dict(T=32, n_cold=129, decode_kind=1)) == 0
    assert bench.ffn_terms(dict(T=32, n_cold=129, zero_copy=True)) == 0
    zc = dict(T=1, n_cold=129, zero_copy=True)  # GEMV, no copy launches
    assert bench.step_launches(zc) == 1 + 1 + (1 + 2 * 3) + 1
    c4 = dict(T=8192, n_cold=0, prefill="fp4")  # route in two kernels, no copy, one class
    assert bench.ffn_terms(c4) == 1
    assert bench.step_launches(c4) == 2 + 1 + 3 + 1
    c4f = dict(T=8192, n_cold=0, prefill="f16")  # three decode ranges + tcgen05 per phase
    assert bench.step_launches(c4f) == 2 + 1 + (1 + 1 * (2 * 4 + 1)) + 1
    assert bench.decode_arithmetic(c2).startswith("block-scaled")
    assert bench.decode_arithmetic(c1).startswith("dequant")
