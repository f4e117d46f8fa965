"""Properties of the seeded input generators (no GPU): the routing shapes the
workloads claim."""
import numpy as np

import oracle
import synth


def _distinct_per_window(logits, k, window):
    _, ids, *_ = oracle.route(logits, k)
    return [len(np.unique(ids[w:w + window])) for w in range(0, ids.shape[0], window)]


def test_verify_window_picks_3_7x_the_experts_of_one_token():
    """Verify windows of 6 tokens (the k + 1 a speculative step checks) pick about
    3.7 times the distinct experts of one token, the multiplier "Milo and James Try
    Inference Engineering" measured for the verify window (section on expert
    prefetch from draft tokens)."""
    E, k, W = 384, 6, synth.VERIFY_WINDOW
    logits = synth.gen_logits_verify(W * 400, E, seed=123)
    ratio = np.mean(_distinct_per_window(logits, k, W)) / k
    assert 3.55 <= ratio <= 3.85, ratio


def test_verify_windows_are_independent():
    """Routing is correlated within a window only: with the shared component off the
    windows pick as independent tokens do, and tokens of different windows share
    experts no more than independent tokens."""
    E, k, W = 384, 6, synth.VERIFY_WINDOW
    ind = synth.gen_logits_verify(W * 300, E, seed=5, beta=0.0)
    r0 = np.mean(_distinct_per_window(ind, k, W)) / k
    expected = E * (1.0 - (1.0 - k / E) ** W) / k  # distinct of W independent uniform top-k draws
    assert abs(r0 - expected) < 0.15, (r0, expected)
    corr = synth.gen_logits_verify(W * 300, E, seed=6)
    _, ids, *_ = oracle.route(corr, k)
    # pairs of tokens from neighbouring windows overlap like independent tokens
    cross = [len(np.intersect1d(ids[w * W], ids[(w + 1) * W])) for w in range(299)]
    assert np.mean(cross) < 0.3, np.mean(cross)


def test_zipf_skew_matches_the_pages_share():
    """s = 1.5 puts ~98.7% of picks on 73% of the experts (the pages' routing skew);
    s = 1.1 is milder."""
    E, k = 384, 6
    perm = synth.zipf_permutation(E, 1)
    for s, lo, hi in ((1.5, 0.975, 0.995), (1.1, 0.93, 0.975)):
        _, ids, *_ = oracle.route(synth.gen_logits_zipf(2000, E, s, perm, seed=2), k)
        cnt = np.sort(np.bincount(ids.ravel(), minlength=E))[::-1]
        share = cnt[:int(0.73 * E)].sum() / cnt.sum()
        assert lo <= share <= hi, (s, share)
