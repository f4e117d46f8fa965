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


def test_weight_codes_follow_rounded_normal():
    """Nibble codes are draws of E2M1 round-to-nearest of N(0,1) (saturating at
    +-6): the frequencies match the normal probabilities of each code's rounding
    interval (scipy's normal CDF), every code occurs, scale bytes are 127 - U{0..8}."""
    import pytest

    stats = pytest.importorskip("scipy.stats")
    H, I = 256, 512
    blob = synth.gen_blobs(1, H, I, seed=5)[0].numpy()
    sec = synth.blob_sections(H, I)
    nib = np.concatenate([blob[sec["w13n"][0]:sec["w13n"][0] + sec["w13n"][1]],
                          blob[sec["w2n"][0]:sec["w2n"][0] + sec["w2n"][1]]])
    codes = np.concatenate([nib & 15, nib >> 4])
    freq = np.bincount(codes, minlength=16) / codes.size
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    mid = [(a + b) / 2 for a, b in zip(mags[:-1], mags[1:])]
    edges = np.array([0.0] + mid + [np.inf])
    half = np.diff(stats.norm.cdf(edges))  # P(|z| in the rounding interval of each magnitude) / 2
    want = np.concatenate([half, half])  # + and - codes
    n = codes.size
    assert np.all(np.bincount(codes, minlength=16) > 0)
    sigma = np.sqrt(np.maximum(want, 1.0 / n) * (1 - want) / n)
    assert np.all(np.abs(freq - want) < 6 * sigma + 2.0 ** -16)
    sc = np.concatenate([blob[sec["w13s"][0]:sec["w13s"][0] + sec["w13s"][1]],
                         blob[sec["w2s"][0]:sec["w2s"][0] + sec["w2s"][1]]])
    assert sc.min() == 119 and sc.max() == 127
    cnt = np.bincount(sc - 119, minlength=9) / sc.size
    assert np.all(np.abs(cnt - 1 / 9) < 6 * np.sqrt((1 / 9) * (8 / 9) / sc.size))


def test_zipf_first_pick_is_the_zipf_law():
    """logits = log p(rank) + Gumbel(0,1): the top pick is a draw from p (the
    Gumbel-max property), with rank 1 the first expert of the permutation."""
    E, s, T = 16, 1.1, 60000
    perm = synth.zipf_permutation(E, 3)
    l = synth.gen_logits_zipf(T, E, s, perm, seed=4)
    top = np.argmax(l, axis=1)
    freq = np.bincount(top, minlength=E) / T
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** -s / np.sum(r ** -s)
    want = np.empty(E)
    want[perm] = p
    assert np.all(np.abs(freq - want) < 6 * np.sqrt(want * (1 - want) / T))


def test_activations_are_bf16_standard_normal():
    import torch

    x = synth.gen_x(64, 4096, seed=9)
    assert x.dtype == torch.bfloat16 and tuple(x.shape) == (64, 4096)
    v = x.float().numpy().ravel()
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01
    assert np.array_equal(synth.gen_x(64, 4096, seed=9).float().numpy(), x.float().numpy())  # seeded


def test_starting_maps_are_placements():
    E, n_hot = 384, 255
    assert np.array_equal(synth.loc_identity(E, n_hot), np.arange(E))
    hot = synth.zipf_permutation(E, 1)[:n_hot]
    loc = synth.loc_from_hot_set(E, n_hot, hot)
    assert np.array_equal(np.sort(loc), np.arange(E))  # a bijection
    assert np.all(loc[hot] < n_hot)
    assert np.array_equal(np.sort(hot), np.argsort(np.where(loc < n_hot, loc, E + loc))[:n_hot])
