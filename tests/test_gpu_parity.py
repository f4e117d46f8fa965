"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Bar: routing ids, counts/offsets/entries, phys ids, cold lists and gathered
bytes bit-exact; router weights within rtol 2e-6 of the fp64 oracle (fp32
softmax over E <= 1024 terms: expf error, argument rounding and a log2(E)-deep
sum stay under 1.3e-6 relative); expert outputs and the layer output within
relative L2 5e-3 of the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import LayerFixture, bf16_bits, rel_l2

pytestmark = pytest.mark.gpu

W_RTOL = 2e-6
OUT_TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    oracle.build()


def _route_layer(E, k, renorm=0):
    """Minimal all-hot layer (H = I = 128, zero weights) for routing tests."""
    return LayerFixture(H=128, I=128, E=E, n_hot=E, n_cold=0, k=k, seed=1, renorm=renorm)


def _check_route(fx, logits_np, renorm=0):
    import moe_decode_host_gb300 as m

    T, E = logits_np.shape
    k = fx.k
    buf = m.StepBuffers(fx.layer, T)
    m.moe_route(fx.layer, torch.from_numpy(logits_np).cuda(), T, buf.topk_ids, buf.topk_w, buf.counts, buf.offsets,
                buf.entries)
    torch.cuda.synchronize()
    rc, ids, w, counts, offsets, entries = oracle.route(logits_np, k, renorm)
    assert rc == 0
    if T > 0:
        assert np.array_equal(buf.topk_ids.cpu().numpy()[:T], ids)
        np.testing.assert_allclose(buf.topk_w.cpu().numpy()[:T], w, rtol=W_RTOL, atol=0)
        assert np.array_equal(buf.entries.cpu().numpy()[:T * k], entries)
    assert np.array_equal(buf.counts.cpu().numpy(), counts)
    assert np.array_equal(buf.offsets.cpu().numpy(), offsets)
    return buf, counts


def test_e2m1_pair_conversion_lane_layout():
    out = torch.zeros(256, dtype=torch.int32, device="cuda")
    import moe_decode_host_gb300 as m

    m.debug_e2m1_pairs(out)
    v = out.cpu().numpy().view(np.uint32)
    lo = (v & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    hi = (v >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
    for b in range(256):
        assert lo[b] == oracle.e2m1(b & 15) and np.signbit(lo[b]) == np.signbit(oracle.e2m1(b & 15)), b
        assert hi[b] == oracle.e2m1(b >> 4) and np.signbit(hi[b]) == np.signbit(oracle.e2m1(b >> 4)), b


@pytest.mark.parametrize("E,k,T,renorm,dist", [
    (16, 2, 4, 0, "uniform"),      # c0
    (384, 6, 1, 0, "uniform"),     # c1
    (384, 6, 8, 0, "zipf1.1"),     # c2
    (384, 6, 32, 0, "zipf1.5"),    # c2, page-faithful skew
    (384, 6, 64, 1, "uniform"),    # largest single-CTA batch, renorm
    (384, 6, 65, 0, "uniform"),    # first two-kernel batch
    (384, 6, 1000, 1, "zipf1.1"),  # ragged multi-CTA, split bucketing (6000 picks)
    (96, 7, 700, 0, "zipf1.5"),    # split bucketing, 4900 picks (ragged per warp)
    (1024, 32, 200, 0, "uniform"), # split bucketing at maximum E and k
    (40, 5, 13, 1, "ties"),
    (1024, 32, 7, 0, "uniform"),   # maximum E and k
    (8, 8, 3, 0, "uniform"),       # k == E
    (33, 1, 5, 0, "ties"),
])
def test_route_parity(E, k, T, renorm, dist):
    fx = _route_layer(E, k, renorm)
    if dist == "uniform":
        logits = synth.gen_logits_uniform(T, E, seed=E * 1000 + T)
    elif dist == "ties":
        logits = np.random.default_rng(T).integers(-2, 3, (T, E)).astype(np.float32)
        logits[:, ::3] = -0.0
    else:
        s = float(dist[4:])
        logits = synth.gen_logits_zipf(T, E, s, synth.zipf_permutation(E, 5), seed=T)
    buf, counts = _check_route(fx, logits, renorm)
    # the window counters of the layer saw exactly these picks
    assert np.array_equal(fx.layer.get_counts(), counts)
    assert fx.layer.status() == 0


def test_route_c4_batch_8192():
    fx = _route_layer(384, 6)
    logits = synth.gen_logits_uniform(8192, 384, seed=synth.sub_seed("c4", "logits"))
    _check_route(fx, logits)


def test_route_empty_batch():
    import moe_decode_host_gb300 as m

    fx = _route_layer(16, 2)
    buf = m.StepBuffers(fx.layer, 0)
    buf.counts.fill_(7)
    buf.offsets.fill_(7)
    m.moe_route(fx.layer, None, 0, None, None, buf.counts, buf.offsets, None)
    torch.cuda.synchronize()
    assert buf.counts.abs().sum().item() == 0 and buf.offsets.abs().sum().item() == 0


def test_route_nonfinite_sets_status():
    import moe_decode_host_gb300 as m

    fx = _route_layer(16, 2)
    logits = synth.gen_logits_uniform(3, 16, seed=9)
    logits[1, 5] = np.nan
    buf = m.StepBuffers(fx.layer, 3)
    m.moe_route(fx.layer, torch.from_numpy(logits).cuda(), 3, buf.topk_ids, buf.topk_w, buf.counts, buf.offsets,
                buf.entries)
    torch.cuda.synchronize()
    assert fx.layer.status() == m.MOE_ERR_NONFINITE
    ids = buf.topk_ids.cpu().numpy()
    assert ids[1].tolist() == [0, 1] and buf.topk_w.cpu().numpy()[1].tolist() == [0.0, 0.0]
    _, ids0, *_ = oracle.route(logits[[0, 2]], 2)
    assert np.array_equal(ids[[0, 2]], ids0)
    fx.layer.clear_status()
    assert fx.layer.status() == 0


# ------------------------------------------------------------------ gather

def _gather_check(fx, logits, T):
    import moe_decode_host_gb300 as m

    buf = m.StepBuffers(fx.layer, T)
    fx.slots.fill_(0xAB)
    loc = fx.layer.get_loc()
    m.moe_route(fx.layer, torch.from_numpy(logits).cuda(), T, buf.topk_ids, buf.topk_w, buf.counts, buf.offsets,
                buf.entries)
    m.cold_gather(fx.layer, buf.topk_ids, T, buf.phys_ids, buf.cold_list, buf.n_cold_picked)
    m.moe_gather_join(fx.layer)
    torch.cuda.synchronize()
    ids = buf.topk_ids.cpu().numpy()[:T]
    phys, cold = oracle.remap(ids, loc, fx.n_hot, fx.n_cold)
    assert np.array_equal(buf.phys_ids.cpu().numpy()[:T * fx.k].reshape(T, fx.k), phys)
    n = int(buf.n_cold_picked.item())
    assert n == cold.size
    assert np.array_equal(buf.cold_list.cpu().numpy()[:n], cold)
    slots = fx.slots.cpu().numpy()
    for c in range(fx.n_cold):
        if c in set(cold.tolist()):
            assert np.array_equal(slots[c], fx.cold[c].numpy()), c
        else:
            assert np.all(slots[c] == 0xAB), c
    return buf


def test_cold_gather_c0():
    c = synth.CONFIGS["c0"]
    for loc in (synth.loc_identity(16, 12), np.random.default_rng(3).permutation(16).astype(np.int32)):
        fx = LayerFixture(H=c["H"], I=c["I"], E=16, n_hot=12, n_cold=4, k=2, seed=2, loc=loc)
        for T in (1, 4, 9):
            _gather_check(fx, synth.gen_logits_uniform(T, 16, seed=T), T)


def test_cold_gather_many_picks():
    """12,000 picks over 64 experts (16 cold, permuted placement): the remap takes
    several rounds of four picks per thread."""
    loc = np.random.default_rng(11).permutation(64).astype(np.int32)
    fx = LayerFixture(H=128, I=128, E=64, n_hot=48, n_cold=16, k=6, seed=6, loc=loc)
    T = 2000
    _gather_check(fx, synth.gen_logits_uniform(T, 64, seed=17), T)


def test_cold_gather_bad_expert_ids():
    import moe_decode_host_gb300 as m

    fx = LayerFixture(H=256, I=512, E=16, n_hot=12, n_cold=4, k=2, seed=2)
    ids = torch.tensor([[3, 13], [-1, 16]], dtype=torch.int32, device="cuda")
    buf = m.StepBuffers(fx.layer, 2)
    m.cold_gather(fx.layer, ids, 2, buf.phys_ids, buf.cold_list, buf.n_cold_picked)
    m.moe_gather_join(fx.layer)
    torch.cuda.synchronize()
    assert buf.phys_ids.cpu().numpy()[:4].tolist() == [3, 13, -1, -1]
    assert int(buf.n_cold_picked.item()) == 1 and int(buf.cold_list[0].item()) == 1
    assert fx.layer.status() == m.MOE_ERR_BAD_EXPERT
    assert np.array_equal(fx.slots[1].cpu().numpy(), fx.cold[1].numpy())


# ------------------------------------------------------------------ whole layer

def _run_layer(fx, logits, x, out_fp32):
    import moe_decode_host_gb300 as m

    T = logits.shape[0]
    buf = m.StepBuffers(fx.layer, T, out_fp32=out_fp32)
    m.run_step(fx.layer, buf, torch.from_numpy(logits).cuda(), x.cuda(), residency=False)
    torch.cuda.synchronize()
    assert fx.layer.status() == 0, fx.layer.diag().tolist()
    return buf


def _oracle_rows(fx, blobs, x_bits, ids, tokens):
    """Oracle y rows and layer outputs for the given tokens only."""
    xs = oracle.bf16_bits_to_f64(x_bits)
    y = {}
    by_expert = {}
    for t in tokens:
        for j in range(fx.k):
            by_expert.setdefault(int(ids[t, j]), []).append((t, j))
    for e, tj in by_expert.items():
        yy = oracle.expert_ffn(blobs[e], fx.H, fx.I, np.stack([xs[t] for t, _ in tj]))
        for (t, j), row in zip(tj, yy):
            y[(t, j)] = row
    return y


def _compare_layer(fx, buf, logits, x, tokens, out_fp32):
    T = logits.shape[0]
    rc, ids, w, *_ = oracle.route(logits, fx.k)
    assert np.array_equal(buf.topk_ids.cpu().numpy()[:T], ids)
    blobs = {e: fx.expert_bytes_now(int(e)) for e in np.unique(ids[tokens])}
    y = _oracle_rows(fx, blobs, bf16_bits(x), ids, tokens)
    ygpu = buf.y.cpu().numpy()
    out = buf.out.float().cpu().numpy()
    worst_y = 0.0
    for t in tokens:
        want = np.zeros(fx.H)
        for j in range(fx.k):
            worst_y = max(worst_y, rel_l2(ygpu[t * fx.k + j], y[(t, j)]))
            want += w[t, j] * y[(t, j)]
        r = rel_l2(out[t], want)
        assert r <= OUT_TOL, (t, r)
    assert worst_y <= OUT_TOL, worst_y
    return worst_y


@pytest.mark.parametrize("T,dist", [(1, "uniform"), (8, "zipf1.1"), (33, "zipf1.5"), (64, "uniform")])
def test_layer_zero_copy_matches_copy_path(T, dist):
    """Zero copy: the cold experts' weights are read in place from host memory and
    their slots stay untouched; the outputs match the copy path's on the same
    dequant-GEMV kernel to rounding (the same arithmetic in the same order; the two
    kernel variants are compiled separately, so the compiler's fused multiply-adds
    may differ in the last bit), and the oracle within the bar; the copy path on the
    block-scaled decode kernels matches the oracle too."""
    H, I, E, n_hot, k = 1024, 768, 32, 24, 6
    loc = np.random.default_rng(T).permutation(E).astype(np.int32)
    if dist == "uniform":
        logits = synth.gen_logits_uniform(T, E, seed=40 + T)
    else:
        logits = synth.gen_logits_zipf(T, E, float(dist[4:]), synth.zipf_permutation(E, 3), seed=40 + T)
    x = synth.gen_x(T, H, seed=41 + T)
    outs = []
    for zc in (False, True):
        fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=E - n_hot, k=k, seed=77, loc=loc, zero_copy=zc)
        fx.layer.set_decode_kind(1)  # the copy path on the same kernel as the zero-copy path
        fx.slots.fill_(0xAB)
        buf = _run_layer(fx, logits, x, True)
        outs.append((buf.y.cpu().clone(), buf.out.cpu().clone()))
        if zc:
            assert bool((fx.slots == 0xAB).all()), "zero copy wrote a scratch slot"
            _compare_layer(fx, buf, logits, x, list(range(0, T, max(1, T // 8))), True)
            assert int(buf.n_cold_picked.item()) > 0
        fx.layer.close()
    assert rel_l2(outs[1][0].numpy(), outs[0][0].numpy()) <= 1e-6
    assert rel_l2(outs[1][1].numpy(), outs[0][1].numpy()) <= 1e-6
    # the default decode kernels on the copy path
    fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=E - n_hot, k=k, seed=77, loc=loc)
    buf = _run_layer(fx, logits, x, True)
    _compare_layer(fx, buf, logits, x, list(range(0, T, max(1, T // 8))), True)
    fx.layer.close()


def test_layer_zero_copy_large_call_copies():
    """Zero copy applies to calls of at most 64 tokens; a 200-token call copies its
    cold experts (the tensor-core kernel reads the scratch) and matches the oracle."""
    H, I, E, n_hot, k, T = 256, 512, 8, 6, 2, 200
    fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=E - n_hot, k=k, seed=5, zero_copy=True)
    logits = synth.gen_logits_uniform(T, E, seed=8)
    x = synth.gen_x(T, H, seed=9)
    buf = _run_layer(fx, logits, x, True)
    rc, ids, w, want = oracle.layer(logits, bf16_bits(x), k, 0, H, I, fx.all_blobs_now())
    assert rc == 0
    assert rel_l2(buf.out.cpu().numpy(), want) <= OUT_TOL
    fx.layer.close()


@pytest.mark.parametrize("out_fp32", [False, True])
def test_layer_c0(out_fp32):
    c = synth.CONFIGS["c0"]
    fx = LayerFixture(H=c["H"], I=c["I"], E=c["E"], n_hot=c["n_hot"], n_cold=c["n_cold"], k=c["k"],
                      seed=synth.sub_seed("c0", "blobs"))
    logits = synth.gen_logits_uniform(c["T"], c["E"], seed=0)
    x = synth.gen_x(c["T"], c["H"], seed=synth.sub_seed("c0", "x"))
    buf = _run_layer(fx, logits, x, out_fp32)
    # whole-layer oracle on all tokens
    rc, ids, w, want = oracle.layer(logits, bf16_bits(x), c["k"], 0, c["H"], c["I"], fx.all_blobs_now())
    assert rc == 0
    got = buf.out.float().cpu().numpy()
    assert rel_l2(got, want) <= OUT_TOL
    _compare_layer(fx, buf, logits, x, list(range(c["T"])), out_fp32)


@pytest.mark.parametrize("decode_kind", [0, 1, 2])
@pytest.mark.parametrize("H,I,E,n_hot,k,T,dist", [
    (384, 640, 40, 30, 5, 13, "uniform"),   # uneven split of the reduction over warps; K stages of 128
    (128, 128, 8, 5, 8, 3, "uniform"),      # k == E, a single 128-group per row
    (512, 256, 64, 48, 6, 40, "zipf1.5"),   # buckets above 8, 16, 32 and 48 tokens (two column passes)
    (256, 512, 16, 0, 2, 17, "uniform"),    # everything cold
    (256, 512, 16, 8, 4, 1, "uniform"),     # one token
    (384, 640, 40, 30, 5, 2, "uniform"),    # two tokens
])
def test_layer_ragged_shapes(H, I, E, n_hot, k, T, dist, decode_kind):
    """Decode-sized calls on both decode kernels: the dequant-GEMV kernel (kind 1),
    block-scaled tensor cores with four-term activations (kind 2) and the default
    (kind 0)."""
    n_cold = E - n_hot
    loc = np.random.default_rng(E).permutation(E).astype(np.int32)
    fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=n_cold, k=k, seed=E + T, loc=loc)
    fx.layer.set_decode_kind(decode_kind)
    if dist == "uniform":
        logits = synth.gen_logits_uniform(T, E, seed=T)
    else:
        logits = synth.gen_logits_zipf(T, E, 1.5, synth.zipf_permutation(E, 1), seed=T)
    x = synth.gen_x(T, H, seed=T + 1)
    buf = _run_layer(fx, logits, x, True)
    rc, ids, w, want = oracle.layer(logits, bf16_bits(x), k, 0, H, I, fx.all_blobs_now())
    assert rel_l2(buf.out.cpu().numpy(), want) <= OUT_TOL
    if dist != "uniform":
        assert np.bincount(ids.ravel(), minlength=E).max() > 32


# ------------------------------------------------------------------ prefill-sized buckets

def _assigned_logits(counts, E, seed):
    """k=1 logits giving expert e exactly counts[e] tokens (tokens in shuffled order)."""
    rng = np.random.default_rng(seed)
    owner = rng.permutation(np.repeat(np.arange(E), counts))
    l = rng.standard_normal((owner.size, E)).astype(np.float32)
    l[np.arange(owner.size), owner] += 12.0
    return l


@pytest.mark.parametrize("H,I,E,n_hot,k,T,dist", [
    (256, 512, 16, 12, 2, 1024, "uniform"),  # ~128 tokens per expert, four of them cold
    (256, 256, 4, 4, 2, 600, "uniform"),     # ~300 per expert: two column passes (192 + rest)
    (384, 640, 40, 30, 5, 600, "zipf1.5"),   # buckets on both sides of 64, uneven K
    (512, 1536, 16, 12, 2, 1024, "uniform"),  # 16-byte scale rows: one group of 4 chunks, then three
])
def test_layer_prefill_buckets(H, I, E, n_hot, k, T, dist):
    n_cold = E - n_hot
    loc = np.random.default_rng(E + 1).permutation(E).astype(np.int32)
    fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=n_cold, k=k, seed=E + T, loc=loc)
    if dist == "uniform":
        logits = synth.gen_logits_uniform(T, E, seed=T)
    else:
        logits = synth.gen_logits_zipf(T, E, 1.5, synth.zipf_permutation(E, 2), seed=T)
    x = synth.gen_x(T, H, seed=T + 1)
    buf = _run_layer(fx, logits, x, True)
    rc, ids, w, want = oracle.layer(logits, bf16_bits(x), k, 0, H, I, fx.all_blobs_now())
    assert rc == 0
    cnt = np.bincount(ids.ravel(), minlength=E)
    assert cnt.max() > 64
    assert rel_l2(buf.out.cpu().numpy(), want) <= OUT_TOL
    _compare_layer(fx, buf, logits, x, list(range(0, T, 7)), True)
    fx.layer.close()


@pytest.mark.parametrize("counts", [[65, 64, 193, 0, 1, 128, 129, 70], [160, 161, 320, 0, 2, 337, 96, 112]])
def test_layer_prefill_bucket_edges(counts):
    """Buckets of exactly 64 (decode kernel) and 65 (tensor cores), one token, full
    column passes of 160 tokens with and without a padded tail, two and three
    passes, and an empty expert; cold ones included."""
    E, H, I = 8, 256, 512
    loc = np.array([6, 0, 7, 1, 2, 3, 4, 5], np.int32)  # experts 0 and 2 are cold
    fx = LayerFixture(H=H, I=I, E=E, n_hot=6, n_cold=2, k=1, seed=99, loc=loc)
    logits = _assigned_logits(counts, E, seed=3)
    T = logits.shape[0]
    x = synth.gen_x(T, H, seed=4)
    buf = _run_layer(fx, logits, x, True)
    rc, ids, w, want = oracle.layer(logits, bf16_bits(x), 1, 0, H, I, fx.all_blobs_now())
    assert rc == 0
    assert np.array_equal(np.bincount(ids.ravel(), minlength=E), counts)
    got = buf.out.cpu().numpy()
    assert rel_l2(got, want) <= OUT_TOL
    for e in range(E):  # every bucket on its own
        rows = np.nonzero(ids[:, 0] == e)[0]
        if rows.size:
            assert rel_l2(got[rows], want[rows]) <= OUT_TOL, e
    fx.layer.close()


def test_layer_prefill_full_size_with_cold_experts():
    """H=4096, I=3072 with 16 experts (4 cold) and 320 tokens of top-6: ~120 tokens
    per expert, so the hot and the cold experts both run on the tensor cores."""
    H, I, E, n_hot, k, T = 4096, 3072, 16, 12, 6, 320
    fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=E - n_hot, k=k, seed=123)
    logits = synth.gen_logits_uniform(T, E, seed=5)
    x = synth.gen_x(T, H, seed=6)
    buf = _run_layer(fx, logits, x, False)
    ids = buf.topk_ids.cpu().numpy()
    assert np.bincount(ids.ravel(), minlength=E).min() > 64
    _compare_layer(fx, buf, logits, x, [0, 1, 130, T - 1], False)
    fx.layer.close()


# ------------------------------------------------------------------ full sizes

@pytest.fixture(scope="module")
def c1_layer():
    c = synth.CONFIGS["c1"]
    fx = LayerFixture(H=c["H"], I=c["I"], E=c["E"], n_hot=c["n_hot"], n_cold=c["n_cold"], k=c["k"],
                      seed=synth.sub_seed("c1", "blobs"))
    yield fx
    fx.layer.close()


def test_layer_c1_batch1(c1_layer):
    c = synth.CONFIGS["c1"]
    fx = c1_layer
    for step in range(3):
        logits = synth.gen_logits_uniform(1, c["E"], seed=synth.sub_seed("c1", "logits", step))
        x = synth.gen_x(1, c["H"], seed=synth.sub_seed("c1", "x", step))
        buf = _run_layer(fx, logits, x, False)
        _compare_layer(fx, buf, logits, x, [0], False)
        _gather_check(fx, logits, 1)


@pytest.mark.parametrize("T", [6, 12])
def test_layer_verify_window(c1_layer, T):
    """Verify windows (6 tokens of one sequence with correlated routing) on the c1
    layer: one and two windows, cold experts included."""
    c = synth.CONFIGS["v1"]
    fx = c1_layer
    logits = synth.gen_logits_verify(T, c["E"], seed=synth.sub_seed("v1", "logits", T))
    x = synth.gen_x(T, c["H"], seed=synth.sub_seed("v1", "x", T))
    buf = _run_layer(fx, logits, x, False)
    _compare_layer(fx, buf, logits, x, list(range(0, T, 3)), False)
    _gather_check(fx, logits, T)


# ------------------------------------------------------------------ residency

def _skewed_logits(T, E, step, hot_first):
    """Logits that favour the experts listed in hot_first (so cold ones get picked)."""
    rng = np.random.default_rng(step)
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[:, hot_first] += 2.5
    return l


def paced_landing(n: int, swap_every: int) -> list:
    """Deferred residency: the call (counted from the one after the window closes)
    at which each of a plan's n pairs lands -- pair i at floor(i * span / n), span
    the calls before the next window closes (at least 1)."""
    span = max(1, swap_every - 1)
    return [i * span // n for i in range(n)]


@pytest.mark.parametrize("defer", [True, False])
@pytest.mark.parametrize("host_mirror", [False, True])
def test_residency_matches_oracle_and_keeps_bytes(host_mirror, defer):
    """Maps equal the oracle's rule on every window's counts.  Synchronous mode: the
    whole plan lands at the call that closes the window.  Deferred mode: the plan is
    made at the next call and its pairs land in plan order, paced over the calls
    before the next window closes.  Every expert keeps its bytes and the outputs
    equal a frozen layer's."""
    import moe_decode_host_gb300 as m

    H, I, E, n_hot, n_cold, k, T = 256, 512, 16, 12, 4, 2, 4
    swap_every, max_swaps, steps = 4, 3, 16
    seed = synth.sub_seed("residency")
    fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=n_cold, k=k, seed=seed, swap_every=swap_every,
                      max_swaps=max_swaps, host_mirror=host_mirror, residency_defer=defer)
    frozen = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=n_cold, k=k, seed=seed, swap_every=0)
    fp0 = [oracle.fnv1a64(b) for b in fx.all_blobs_now()]
    host0 = [oracle.fnv1a64(fx.cold[i].numpy()) for i in range(fx.cold.shape[0])]
    loc_o = fx.loc0.copy()      # the oracle's placement after every plan so far
    loc_now = fx.loc0.copy()    # the placement the layer should hold now
    landing = {}                # step -> pairs (promoted, demoted) landing then
    window = np.zeros(E, np.int64)
    total_swaps, spread = 0, 0
    for step in range(steps):
        favoured = [12, 13, 14, 15] if step < steps // 2 else [0, 1, 2, 3]
        logits = _skewed_logits(T, E, step, favoured)
        x = synth.gen_x(T, H, seed=step)
        buf = m.StepBuffers(fx.layer, T, out_fp32=True)
        bufz = m.StepBuffers(frozen.layer, T, out_fp32=True)
        lg = torch.from_numpy(logits).cuda()
        nsw = m.run_step(fx.layer, buf, lg, x.cuda(), residency=True)
        m.run_step(frozen.layer, bufz, lg, x.cuda(), residency=True)
        torch.cuda.synchronize()
        # same routing, same bytes: outputs identical whatever the placement
        assert torch.equal(buf.out, bufz.out), step
        rc, ids, w, counts, _, _ = oracle.route(logits, k)
        window += counts
        if (step + 1) % swap_every == 0:
            loc_o, pro, dem = oracle.residency(window.astype(np.int32), loc_o, n_hot, max_swaps, 3.0)
            window[:] = 0
            when = paced_landing(pro.size, swap_every) if defer else [None] * pro.size
            spread += len(set(when)) > 1
            for i, j in enumerate(when):
                landing.setdefault(step if j is None else step + 1 + j, []).append((int(pro[i]), int(dem[i])))
        pairs = landing.pop(step, [])
        assert nsw == len(pairs), step
        if pairs:
            for a, b in pairs:
                loc_now[a], loc_now[b] = loc_now[b], loc_now[a]
            total_swaps += nsw
            # byte audit: every expert, wherever it now lives
            fp = [oracle.fnv1a64(b) for b in fx.all_blobs_now()]
            assert fp == fp0, step
        assert np.array_equal(fx.layer.get_loc(), loc_now), step
        assert np.array_equal(fx.layer.get_counts(), window.astype(np.int32)), step
        rc, ids, w, want = oracle.layer(logits, bf16_bits(x), k, 0, H, I, fx.all_blobs_now())
        assert rel_l2(buf.out.cpu().numpy(), want) <= OUT_TOL
    assert total_swaps > 0
    if defer:
        assert spread > 0  # some plan landed over several calls
    # at the end the placement is the oracle's but for pairs still to land
    for a, b in sum(landing.values(), []):
        loc_now[a], loc_now[b] = loc_now[b], loc_now[a]
    assert np.array_equal(loc_now, loc_o)
    assert sorted(fx.layer.get_loc().tolist()) == list(range(E))
    if host_mirror:
        # with host copies nothing is ever written to host memory
        assert [oracle.fnv1a64(fx.cold[i].numpy()) for i in range(E)] == host0


@pytest.mark.parametrize("defer", [True, False])
def test_residency_injected_fault_leaves_map(defer):
    import moe_decode_host_gb300 as m

    fx = LayerFixture(H=256, I=512, E=16, n_hot=12, n_cold=4, k=2, seed=4, swap_every=1, residency_defer=defer)
    logits = _skewed_logits(4, 16, 0, [12, 13])
    buf = m.StepBuffers(fx.layer, 4)
    m.moe_route(fx.layer, torch.from_numpy(logits).cuda(), 4, buf.topk_ids, buf.topk_w, buf.counts, buf.offsets,
                buf.entries)
    loc_before = fx.layer.get_loc()
    fx.layer.inject_fault(1)
    with pytest.raises(m.MoeError) as ei:
        m.residency_update(fx.layer)
    assert ei.value.code == m.MOE_ERR_INJECTED
    assert np.array_equal(fx.layer.get_loc(), loc_before)
    if defer:
        # the next call closes the window (its plan lands at the call after)
        assert m.residency_update(fx.layer) == 0
        assert np.array_equal(fx.layer.get_loc(), loc_before)
    assert m.residency_update(fx.layer) > 0
    assert not np.array_equal(fx.layer.get_loc(), loc_before)


@pytest.mark.parametrize("defer", [True, False])
@pytest.mark.parametrize("host_mirror", [False, True])
def test_shared_scratch_across_layers(host_mirror, defer):
    """Several layers share one slot scratch and run one after another (the c3
    structure at c0 size), swapping every other step: each layer's output still
    matches the oracle and every expert keeps its bytes (with host copies a
    promotion may read a scratch slot only while it holds that layer's copy)."""
    import moe_decode_host_gb300 as m

    H, I, E, n_hot, n_cold, k, T = 256, 512, 16, 12, 4, 2, 4
    eb = m.expert_bytes(H, I)
    slots = torch.empty((n_cold, eb), dtype=torch.uint8, device="cuda")
    scratch = m.Scratch(n_cold, eb, slots)
    layers = []
    for L in range(3):
        loc = synth.loc_from_hot_set(E, n_hot, np.random.default_rng(L).permutation(E)[:n_hot])
        layers.append(LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=n_cold, k=k, seed=100 + L, loc=loc,
                                   scratch=scratch, slots=slots, swap_every=2, max_swaps=2, hysteresis=0.5,
                                   host_mirror=host_mirror, residency_defer=defer))
    fp0 = [[oracle.fnv1a64(b) for b in fx.all_blobs_now()] for fx in layers]
    x = synth.gen_x(T, H, seed=5).cuda()
    swaps = 0
    for step in range(6):
        bufs = []
        for L, fx in enumerate(layers):
            logits = synth.gen_logits_uniform(T, E, seed=step * 10 + L)
            buf = m.StepBuffers(fx.layer, T, out_fp32=True)
            swaps += m.run_step(fx.layer, buf, torch.from_numpy(logits).cuda(), x, residency=True)
            bufs.append((fx, logits, buf))
        torch.cuda.synchronize()
        # compare each layer's output with the oracle on the bytes it used (the maps only
        # change at the end of a step, after every layer ran)
        for fx, logits, buf in bufs:
            blobs = fx.all_blobs_now()
            rc, ids, w, want = oracle.layer(logits, bf16_bits(x), k, 0, H, I, blobs)
            assert rel_l2(buf.out.cpu().numpy(), want) <= OUT_TOL
    assert swaps > 0
    for fx, f0 in zip(layers, fp0):
        assert [oracle.fnv1a64(b) for b in fx.all_blobs_now()] == f0
        assert fx.layer.status() == 0


def test_invalid_arguments_launch_nothing():
    import moe_decode_host_gb300 as m

    fx = LayerFixture(H=256, I=512, E=16, n_hot=12, n_cold=4, k=2, seed=4)
    buf = m.StepBuffers(fx.layer, 4)
    with pytest.raises(m.MoeError) as ei:
        m.moe_grouped_ffn(fx.layer, torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda"), 4, buf.phys_ids,
                          buf.counts, buf.offsets, buf.entries, buf.y, buf.workspace, workspace_bytes=16)
    assert ei.value.code == m.MOE_ERR_INVALID_ARG
    # cold blobs must be pinned host memory, hot blobs device memory
    with pytest.raises(m.MoeError):
        m.Layer(E=16, k=2, H=256, I=512, n_hot=12, n_cold=4, scratch=fx.scratch,
                hot_ptrs=[fx.hot[h] for h in range(12)], cold_ptrs=[fx.slots[c] for c in range(4)],
                init_loc=np.arange(16))
    with pytest.raises(m.MoeError):
        m.Layer(E=16, k=2, H=256, I=512, n_hot=12, n_cold=4, scratch=fx.scratch,
                hot_ptrs=[fx.cold[0] for h in range(12)], cold_ptrs=[fx.cold[c] for c in range(4)],
                init_loc=np.arange(16))
