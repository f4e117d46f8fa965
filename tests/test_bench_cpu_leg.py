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
