"""Pins of the CPU oracle against facts that do not come from the oracle itself:
hand-worked MXFP4 decodes and layout bytes (tests/golden), brute-force routing,
closed forms of the softmax and of structured expert FFNs, exact power-of-two
invariants, hand-derived residency swap lists and published FNV-1a vectors."""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _num(s):
    s = s.strip()
    if s.lower() == "nan":
        return float("nan")
    if s.lstrip("-").startswith("0x"):
        return float.fromhex(s)
    return float(s)


def _same(a, b):
    if math.isnan(b):
        return math.isnan(a)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


# ---------------------------------------------------------------- MXFP4 decode

def test_e2m1_table_matches_hand_values():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_codes.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 16
    for code, val in rows:
        assert _same(oracle.e2m1(int(code)), _num(val)), code


def test_mxfp4_bytes_hand_worked():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "mxfp4_bytes.txt")) if l.strip() and not l.startswith("#")]
    for b, s, lo, hi in rows:
        b, s = int(b, 16), int(s)
        # a 128-element row whose first byte is b and whose first block scale is s
        nib = np.zeros(64, np.uint8)
        nib[0] = b
        sc = np.full(4, 127, np.uint8)
        sc[0] = s
        out = oracle.decode_row(nib, sc, 128)
        assert _same(out[0], _num(lo)), (hex(b), s)
        assert _same(out[1], _num(hi)), (hex(b), s)


def test_e8m0_all_exponents():
    for e in range(255):
        assert oracle.e8m0(e) == 2.0 ** (e - 127)
    assert math.isnan(oracle.e8m0(255))


def test_layout_row_hand_worked():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "layout_row.txt")) if l.strip() and not l.startswith("#")]
    K = None
    scales = None
    nib = None
    expect = {}
    for f in lines:
        if f[0] == "K":
            K = int(f[1])
            nib = np.zeros(K // 2, np.uint8)
        elif f[0] == "scales":
            scales = np.array([int(v) for v in f[1:]], np.uint8)
        elif f[0] == "byte":
            nib[int(f[1])] = int(f[2], 16)
        elif f[0] == "value":
            expect[int(f[1])] = _num(f[2])
    out = oracle.decode_row(nib, scales, K)
    for k in range(K):
        want = expect.get(k, 0.0)
        assert out[k] == want, (k, out[k], want)


def test_layout_is_a_bijection():
    # every (byte, nibble) of a 2-group row holds exactly one logical element
    K = 256
    seen = set()
    for k in range(K):
        nib = np.zeros(K // 2, np.uint8)
        sc = np.full(K // 32, 127, np.uint8)
        # find which byte/nibble k reads by probing each position with code 2 (1.0)
        hits = []
        for byte in range(K // 2):
            for shift in (0, 4):
                nib[:] = 0
                nib[byte] = 2 << shift
                if oracle.decode_row(nib, sc, K)[k] == 1.0:
                    hits.append((byte, shift))
        assert len(hits) == 1, (k, hits)
        seen.add(hits[0])
    assert len(seen) == K


def test_scale_applies_to_its_own_32_block_only():
    K = 256
    rng = np.random.default_rng(1)
    nib = rng.integers(0, 256, K // 2, dtype=np.uint8)
    sc = np.full(K // 32, 127, np.uint8)
    base = oracle.decode_row(nib, sc, K)
    for b in range(K // 32):
        sc2 = sc.copy()
        sc2[b] = 128
        out = oracle.decode_row(nib, sc2, K)
        blk = np.arange(32 * b, 32 * b + 32)
        other = np.setdiff1d(np.arange(K), blk)
        assert np.array_equal(out[blk], 2.0 * base[blk])
        assert np.array_equal(out[other], base[other])


# ---------------------------------------------------------------- router

def _brute_topk(l, k):
    """Max-sum k-subset (exact rational sums), lexicographically smallest ids."""
    E = len(l)
    best = None
    for sub in itertools.combinations(range(E), k):
        s = sum(Fraction(float(l[i])) for i in sub)
        if best is None or s > best[0] or (s == best[0] and sub < best[1]):
            best = (s, sub)
    return set(best[1])


@pytest.mark.parametrize("case", ["random", "ties", "zeros", "equal", "int"])
def test_route_matches_brute_force_E16_k2(case):
    rng = np.random.default_rng(7)
    E, k = 16, 2
    for trial in range(40):
        if case == "random":
            l = rng.standard_normal(E).astype(np.float32)
        elif case == "ties":
            l = rng.integers(-3, 4, E).astype(np.float32)
        elif case == "zeros":
            l = rng.choice(np.array([0.0, -0.0, -1.0, 1.0], np.float32), E)
        elif case == "equal":
            l = np.full(E, 0.25, np.float32)
        else:
            l = rng.integers(0, 3, E).astype(np.float32) * np.float32(0.5)
        rc, ids, w, counts, offsets, entries = oracle.route(l[None, :], k)
        assert rc == 0
        got = list(ids[0])
        assert set(got) == _brute_topk(l, k)
        a, b = got
        assert l[a] > l[b] or (l[a] == l[b] and a < b)


def test_route_pos_neg_zero_tie_goes_to_lower_index():
    l = np.array([[-0.0, 0.0, -1.0, -2.0]], np.float32)
    rc, ids, *_ = oracle.route(l, 1)
    assert ids[0, 0] == 0
    l = np.array([[0.0, -0.0, -1.0, -2.0]], np.float32)
    rc, ids, *_ = oracle.route(l, 1)
    assert ids[0, 0] == 0


def test_route_selection_on_logits_not_probabilities():
    # two distinct logits whose softmax probabilities round to the same double
    a = np.float32(-200.0)
    b = np.nextafter(a, np.float32(0.0))
    l = np.array([[a, b, np.float32(0.0)]], np.float32)
    rc, ids, w, *_ = oracle.route(l, 2)
    assert list(ids[0]) == [2, 1]


def test_softmax_two_expert_closed_form():
    for a, b in [(0.5, -0.25), (3.0, 3.0), (-7.0, 2.0), (20.0, -20.0)]:
        l = np.array([[a, b]], np.float32)
        rc, ids, w, *_ = oracle.route(l, 2)
        p_a = 1.0 / (1.0 + math.exp(float(np.float32(b)) - float(np.float32(a))))
        wa = w[0][list(ids[0]).index(0)]
        wb = w[0][list(ids[0]).index(1)]
        assert wa == pytest.approx(p_a, rel=1e-15, abs=1e-300)
        p_b = 1.0 / (1.0 + math.exp(float(np.float32(a)) - float(np.float32(b))))
        assert wb == pytest.approx(p_b, rel=1e-15, abs=1e-300)


def test_softmax_equal_logits_and_shift_invariance():
    E = 16
    l = np.zeros((1, E), np.float32)
    rc, ids, w, *_ = oracle.route(l, 4)
    assert np.all(w == 1.0 / 16)
    rng = np.random.default_rng(3)
    l = rng.standard_normal((3, E)).astype(np.float32)
    _, ids1, w1, *_ = oracle.route(l, 3)
    _, ids2, w2, *_ = oracle.route(l + np.float32(8.0), 3)
    assert np.array_equal(ids1, ids2)
    np.testing.assert_allclose(w1, w2, rtol=1e-6)


def test_softmax_sums_to_one():
    rng = np.random.default_rng(4)
    l = rng.standard_normal((5, 16)).astype(np.float32)
    _, _, w, *_ = oracle.route(l, 16, renorm=0)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    _, _, w, *_ = oracle.route(l, 3, renorm=1)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)


def test_route_nonfinite_rejected():
    for bad in (np.nan, np.inf, -np.inf):
        l = np.zeros((2, 8), np.float32)
        l[1, 3] = bad
        rc, *_ = oracle.route(l, 2)
        assert rc == oracle.ERR_NONFINITE


def test_bucketing_invariants():
    rng = np.random.default_rng(5)
    T, E, k = 37, 16, 3
    l = rng.standard_normal((T, E)).astype(np.float32)
    rc, ids, w, counts, offsets, entries = oracle.route(l, k)
    assert counts.sum() == T * k
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert np.all(np.diff(offsets) == counts)
    for e in range(E):
        seg = entries[offsets[e]:offsets[e + 1]]
        assert np.all(ids.ravel()[seg] == e)
        assert np.all(np.diff(seg) > 0)
    assert sorted(entries.tolist()) == list(range(T * k))


# ---------------------------------------------------------------- placement

def test_remap_hand_built():
    # E=8, n_hot=4: experts 1,3,4,6 hot; 0,2,5,7 cold in that order
    loc = np.array([4, 0, 5, 1, 2, 6, 3, 7], np.int32)
    ids = np.array([[6, 0], [5, 0], [3, 7]], np.int32)
    phys, cold = oracle.remap(ids, loc, 4, 4)
    assert phys.tolist() == [[3, 4], [6, 4], [1, 7]]
    assert cold.tolist() == [0, 2, 3]


# ---------------------------------------------------------------- expert FFN

def _pack_matrix(W_codes, W_scales):
    """Test-side packer: codes [R, K] (0..15), scale bytes [R, K//32] -> (nibble bytes, scale bytes)."""
    R, K = W_codes.shape
    nib = np.zeros((R, K // 2), np.uint8)
    for r in range(R):
        for k in range(K):
            if k % 2 == 0:
                nib[r, k // 2] |= W_codes[r, k]
            else:
                nib[r, k // 2] |= W_codes[r, k] << 4
    return nib, np.asarray(W_scales, np.uint8)


def _blob(H, I, w13_codes, w13_sc, w2_codes, w2_sc):
    n13, s13 = _pack_matrix(w13_codes, w13_sc)
    n2, s2 = _pack_matrix(w2_codes, w2_sc)
    return np.concatenate([n13.ravel(), s13.ravel(), n2.ravel(), s2.ravel()])


def test_blob_size_matches_hand_computed_bytes():
    # 3*H*I nibbles plus one scale byte per 32 elements
    assert oracle.blob_offsets(256, 512)["total"] == 208896
    assert oracle.blob_offsets(4096, 3072)["total"] == 20054016
    assert synth.blob_sections(4096, 3072)["total"] == 20054016


def test_ffn_zero_weights_give_zero():
    H, I = 128, 256
    blob = np.zeros(oracle.blob_offsets(H, I)["total"], np.uint8)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, H))
    assert np.all(oracle.expert_ffn(blob, H, I, x) == 0.0)


def test_ffn_structured_closed_form():
    # gate row r reads x[(r) % H] with weight 1.0; up row r reads x[(r+5) % H] with
    # weight 2.0 (code 4); w2 row r reads h[(3r) % I] with weight 1.0.
    H, I = 128, 256
    w13 = np.zeros((2 * I, H), np.uint8)
    for r in range(I):
        w13[r, r % H] = 2              # 1.0
        w13[I + r, (r + 5) % H] = 4    # 2.0
    w2 = np.zeros((H, I), np.uint8)
    for r in range(H):
        w2[r, (3 * r) % I] = 2
    blob = _blob(H, I, w13, np.full((2 * I, H // 32), 127), w2, np.full((H, I // 32), 127))
    rng = np.random.default_rng(11)
    x = rng.standard_normal((2, H))
    y = oracle.expert_ffn(blob, H, I, x)
    for t in range(2):
        for r in range(H):
            c = (3 * r) % I
            g = x[t, c % H]
            u = 2.0 * x[t, (c + 5) % H]
            want = g / (1.0 + math.exp(-g)) * u
            assert y[t, r] == pytest.approx(want, rel=1e-15, abs=1e-300)


def test_ffn_power_of_two_scale_invariants():
    H, I = 128, 256
    sec = oracle.blob_offsets(H, I)
    blob = synth.gen_blobs(1, H, I, seed=3)[0].numpy()
    rng = np.random.default_rng(12)
    x = rng.standard_normal((2, H))
    y = oracle.expert_ffn(blob, H, I, x)
    # every w2 scale byte +1 doubles y exactly
    b2 = blob.copy()
    b2[sec["w2s"]:] += 1
    assert np.array_equal(oracle.expert_ffn(b2, H, I, x), 2.0 * y)
    # every up-row scale byte +1 doubles h, hence y, exactly
    b3 = blob.copy()
    up0 = sec["w13s"] + I * (H // 32)
    b3[up0:sec["w2n"]] += 1
    assert np.array_equal(oracle.expert_ffn(b3, H, I, x), 2.0 * y)


def test_ffn_matches_dense_numpy_reference():
    H, I = 128, 256
    blob = synth.gen_blobs(1, H, I, seed=9)[0].numpy()
    W13 = oracle.decode_matrix(blob, H, I, "w13")
    W2 = oracle.decode_matrix(blob, H, I, "w2")
    rng = np.random.default_rng(13)
    x = rng.standard_normal((3, H))
    gu = x @ W13.T
    g, u = gu[:, :I], gu[:, I:]
    h = g * (1.0 / (1.0 + np.exp(-g))) * u
    want = h @ W2.T
    got = oracle.expert_ffn(blob, H, I, x)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-10 * np.abs(want).max())


def test_combine_identical_experts():
    H, I, E, k = 128, 256, 8, 3
    blob = synth.gen_blobs(1, H, I, seed=21)[0].numpy()
    rng = np.random.default_rng(14)
    logits = rng.standard_normal((2, E)).astype(np.float32)
    x = synth.gen_x(2, H, seed=5)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    rc, ids, w, out = oracle.layer(logits, bits, k, 0, H, I, [blob] * E)
    y = oracle.expert_ffn(blob, H, I, oracle.bf16_bits_to_f64(bits))
    for t in range(2):
        np.testing.assert_allclose(out[t], w[t].sum() * y[t], rtol=1e-12, atol=1e-12 * np.abs(y).max())


@pytest.mark.parametrize("renorm,act4", [(0, False), (1, False), (0, True)])
def test_layer_distinct_experts_tagged_by_powers_of_two(renorm, act4):
    """Expert e is one base expert with every down-projection scale byte raised by
    e, so its output is exactly 2^e times the base output: the layer's result then
    names which experts each token used and with which weights. Picks come from a
    descending stable sort of the logits, weights from the softmax closed form."""
    H, I, E, k, T = 128, 256, 8, 3, 5
    sec = oracle.blob_offsets(H, I)
    base = synth.gen_blobs(1, H, I, seed=31)[0].numpy()
    blobs = []
    for e in range(E):
        b = base.copy()
        b[sec["w2s"]:] += e
        blobs.append(b)
    rng = np.random.default_rng(15)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = synth.gen_x(T, H, seed=6)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    y = oracle.expert_ffn(base, H, I, oracle.bf16_bits_to_f64(bits), act4=act4)
    rc, ids, w, out = oracle.layer(logits, bits, k, renorm, H, I, blobs, act4=act4)
    assert rc == 0
    want_ids = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, want_ids)
    l64 = logits.astype(np.float64)
    p = np.exp(l64 - l64.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    want_w = np.take_along_axis(p, want_ids, axis=1)
    if renorm:
        want_w /= want_w.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w, want_w, rtol=1e-13)
    tag = np.exp2(want_ids.astype(np.float64))
    want = (want_w * tag).sum(axis=1, keepdims=True) * y
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


# ---------------------------------------------------------------- MXFP4 activations (all-FP4 mode)

_E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # E2M1 magnitudes of codes 0..7 (pinned above)


def _golden_quant():
    for line in open(os.path.join(GOLDEN, "mxfp4_quant.txt")):
        if line.startswith("#") or not line.strip():
            continue
        sb, codes, vals = line.split("|")
        v = [_num(x) for x in vals.split(",")]
        v += [0.0] * (32 - len(v))
        yield int(sb), [int(ch, 16) for ch in codes.strip()], np.array(v, np.float64)


def _codes(nib, K):
    return [int((int(nib[i // 2]) >> (4 * (i % 2))) & 15) for i in range(K)]


def _brute_quant_block(v):
    """The OCP conversion of one 32-block restated with exact rationals: the
    exponent bracketed by exact powers of two, every E2M1 magnitude tried."""
    amax = max(abs(float(x)) for x in v)
    if amax == 0.0:
        X = -127
    else:
        e = math.frexp(amax)[1] - 1
        assert Fraction(2) ** e <= Fraction(amax) < Fraction(2) ** (e + 1)
        X = min(127, max(-127, e - 2))
    codes = []
    for x in v:
        r = Fraction(abs(float(x))) / Fraction(2) ** X
        best = min(range(8), key=lambda c: (abs(Fraction(_E2M1_MAG[c]) - r), c % 2))
        codes.append(best | (8 if math.copysign(1.0, float(x)) < 0 else 0))
    return X + 127, codes


def _brute_quant_dequant(row):
    out = np.empty(row.size)
    for b in range(row.size // 32):
        sb, codes = _brute_quant_block(row[32 * b: 32 * b + 32])
        for i, c in enumerate(codes):
            mag = _E2M1_MAG[c & 7] * 2.0 ** (sb - 127)
            out[32 * b + i] = -mag if c & 8 else mag
    return out


def test_quant_mxfp4_hand_worked():
    n = 0
    for sb, codes, v in _golden_quant():
        nib, sc = oracle.quant_mxfp4(v)
        assert sc.tolist() == [sb]
        assert _codes(nib, 32) == codes
        n += 1
    assert n == 8


def test_quant_mxfp4_matches_brute_force():
    rng = np.random.default_rng(41)
    blocks = []
    for _ in range(150):
        blocks.append(rng.standard_normal(32) * 2.0 ** rng.integers(-20, 21))
    for _ in range(50):  # ties and near-ties of the E2M1 grid at scale 2^0
        v = rng.choice([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 3.0], 32) * rng.choice([-1.0, 1.0], 32)
        v[0] = 4.0
        v[1:4] += rng.choice([0.0, 2.0 ** -40, -(2.0 ** -40)], 3)
        blocks.append(v)
    for _ in range(20):  # E8M0 clamps at both ends, sparse blocks
        v = np.where(rng.random(32) < 0.3, rng.standard_normal(32), 0.0)
        blocks.append(v * 2.0 ** rng.choice([-140, -128, 128, 140]))
    K = 32 * len(blocks)
    row = np.concatenate(blocks)
    nib, sc = oracle.quant_mxfp4(row)
    got = _codes(nib, K)
    for b, v in enumerate(blocks):
        sb, codes = _brute_quant_block(v)
        assert int(sc[b]) == sb, b
        assert got[32 * b: 32 * b + 32] == codes, b


def test_quant_mxfp4_scaling_and_sign():
    rng = np.random.default_rng(42)
    v = rng.standard_normal(256)
    nib, sc = oracle.quant_mxfp4(v)
    for k in (-5, 1, 7):
        n2, s2 = oracle.quant_mxfp4(v * 2.0 ** k)
        assert np.array_equal(n2, nib) and np.array_equal(s2.astype(int), sc.astype(int) + k)
    n3, s3 = oracle.quant_mxfp4(-v)
    assert np.array_equal(s3, sc) and np.array_equal(n3, nib ^ 0x88)


def test_ffn_act4_structured_closed_form():
    """Gate row r reads x[r % H] (weight 1), up row r reads x[(r+5) % H] (weight 2),
    down row r reads h[3r % I] (weight 1): with x and h quantised as the
    all-FP4 mode prescribes, y[r] = hq[3r % I] exactly."""
    H, I = 128, 256
    w13 = np.zeros((2 * I, H), np.uint8)
    for r in range(I):
        w13[r, r % H] = 2
        w13[I + r, (r + 5) % H] = 4
    w2 = np.zeros((H, I), np.uint8)
    for r in range(H):
        w2[r, (3 * r) % I] = 2
    blob = _blob(H, I, w13, np.full((2 * I, H // 32), 127), w2, np.full((H, I // 32), 127))
    rng = np.random.default_rng(43)
    x = rng.standard_normal((2, H)) * 3.0
    y = oracle.expert_ffn(blob, H, I, x, act4=True)
    for t in range(2):
        xq = _brute_quant_dequant(x[t])
        h = np.empty(I)
        for r in range(I):
            g, u = xq[r % H], 2.0 * xq[(r + 5) % H]
            h[r] = g / (1.0 + math.exp(-g)) * u
        hq = _brute_quant_dequant(h)
        want = np.array([hq[(3 * r) % I] for r in range(H)])
        assert np.array_equal(y[t], want)


# ---------------------------------------------------------------- residency

def test_residency_hand_derived():
    loc = np.arange(8, dtype=np.int32)  # 0..3 hot, 4..7 cold slots 0..3
    counts = np.array([5, 0, 2, 9, 7, 1, 0, 30], np.int32)
    new, pro, dem = oracle.residency(counts, loc, 4, 8, 3.0)
    assert pro.tolist() == [7, 4] and dem.tolist() == [1, 2]
    assert new.tolist() == [0, 7, 4, 3, 2, 5, 6, 1]


def test_residency_hysteresis_boundary_is_strict():
    loc = np.arange(4, dtype=np.int32)  # 0,1 hot; 2,3 cold
    counts = np.array([2, 5, 6, 0], np.int32)
    new, pro, dem = oracle.residency(counts, loc, 2, 8, 3.0)
    assert pro.size == 0 and new.tolist() == [0, 1, 2, 3]
    counts = np.array([2, 5, 7, 0], np.int32)
    new, pro, dem = oracle.residency(counts, loc, 2, 8, 3.0)
    assert pro.tolist() == [2] and dem.tolist() == [0]
    assert new.tolist() == [2, 1, 0, 3]


def test_residency_ties_and_limit():
    loc = np.arange(8, dtype=np.int32)
    counts = np.array([1, 1, 3, 3, 0, 4, 4, 0], np.int32)
    new, pro, dem = oracle.residency(counts, loc, 4, 8, 3.0)
    assert pro.tolist() == [5, 6] and dem.tolist() == [0, 1]
    new, pro, dem = oracle.residency(counts, loc, 4, 1, 3.0)
    assert pro.tolist() == [5] and dem.tolist() == [0]
    # unpicked cold experts never move, even against idle hot ones
    counts = np.zeros(8, np.int32)
    new, pro, dem = oracle.residency(counts, loc, 4, 8, 3.0)
    assert pro.size == 0


def test_residency_keeps_loc_a_bijection():
    rng = np.random.default_rng(15)
    E, n_hot = 64, 40
    loc = rng.permutation(E).astype(np.int32)
    for _ in range(50):
        counts = rng.integers(0, 12, E).astype(np.int32)
        loc, pro, dem = oracle.residency(counts, loc, n_hot, 8, 3.0)
        assert sorted(loc.tolist()) == list(range(E))


# ---------------------------------------------------------------- audit

def test_fnv1a64_published_vectors():
    assert oracle.fnv1a64(np.frombuffer(b"", np.uint8)) == 0xCBF29CE484222325
    assert oracle.fnv1a64(np.frombuffer(b"a", np.uint8)) == 0xAF63DC4C8601EC8C
    assert oracle.fnv1a64(np.frombuffer(b"foobar", np.uint8)) == 0x85944171F73967E8
