"""GPU parity of the block-scaled (all-FP4) prefill path -- tcgen05 kind::mxf4 with x
and h converted to MXFP4 -- against the oracle's all-FP4 mode, through the C ABI.

The oracle's all-FP4 mode quantises each token's x row and each pick's h row with
the OCP Microscaling rule for E2M1 and multiplies the dequantised values in fp64.
The GPU decides x's codes exactly as the oracle does (x is bf16, so the scaling by
a power of two is exact in both); h is quantised from the fp32 values the tensor
cores accumulate, so a code can differ where h lies within fp32 rounding of a
decision point.  Bars: routing bit-exact; every compared output row within
relative L2 5e-3 of the oracle's all-FP4 result."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import LayerFixture, bf16_bits, oracle_pick_rows, rel_l2

pytestmark = pytest.mark.gpu

OUT_TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    oracle.build()


def _run(fx, logits, x, out_fp32=True):
    import moe_decode_host_gb300 as m

    fx.layer.set_prefill_kind(1)
    T = logits.shape[0]
    buf = m.StepBuffers(fx.layer, T, out_fp32=out_fp32)
    m.run_step(fx.layer, buf, torch.from_numpy(logits).cuda(), x.cuda(), residency=False)
    torch.cuda.synchronize()
    assert fx.layer.status() == 0, fx.layer.diag().tolist()
    return buf


def _assigned_logits(counts, E, seed):
    """k=1 logits giving expert e exactly counts[e] tokens (tokens in shuffled order)."""
    rng = np.random.default_rng(seed)
    owner = rng.permutation(np.repeat(np.arange(E), counts))
    l = rng.standard_normal((owner.size, E)).astype(np.float32)
    l[np.arange(owner.size), owner] += 12.0
    return l


@pytest.mark.parametrize("H,I,E,n_hot,k,T,dist", [
    (256, 512, 16, 12, 2, 1024, "uniform"),   # ~128 tokens per expert, four experts cold
    (384, 640, 40, 30, 5, 600, "zipf1.5"),    # K of 1.5 and 2.5 stages; buckets from 1 token up
    (512, 1536, 16, 12, 2, 1024, "uniform"),  # several K stages per pass
    (256, 256, 4, 4, 2, 600, "uniform"),      # ~300 tokens per expert: two column passes
])
def test_mx_layer_matches_oracle_fp4_mode(H, I, E, n_hot, k, T, dist):
    loc = np.random.default_rng(E + 1).permutation(E).astype(np.int32)
    fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=E - n_hot, k=k, seed=E + T, loc=loc)
    if dist == "uniform":
        logits = synth.gen_logits_uniform(T, E, seed=T)
    else:
        logits = synth.gen_logits_zipf(T, E, 1.5, synth.zipf_permutation(E, 2), seed=T)
    x = synth.gen_x(T, H, seed=T + 1)
    buf = _run(fx, logits, x)
    rc, ids, w, want = oracle.layer(logits, bf16_bits(x), k, 0, H, I, fx.all_blobs_now(), act4=True)
    assert rc == 0
    assert np.array_equal(buf.topk_ids.cpu().numpy()[:T], ids)
    got = buf.out.cpu().numpy()
    assert rel_l2(got, want) <= OUT_TOL
    worst = max(rel_l2(got[t], want[t]) for t in range(T))
    assert worst <= OUT_TOL, worst
    # and the quantisation is really on: the unquantised layer is far away
    _, _, _, plain = oracle.layer(logits, bf16_bits(x), k, 0, H, I, fx.all_blobs_now())
    assert rel_l2(got, plain) > 0.05
    fx.layer.close()


@pytest.mark.parametrize("counts", [[65, 64, 193, 0, 1, 128, 129, 70], [160, 161, 320, 0, 2, 385, 96, 17]])
def test_mx_bucket_edges(counts):
    """One-token and small buckets, a bucket of exactly one pass (192 would be the
    pass width), two and three passes with ragged tails, an empty expert; cold
    experts included."""
    E, H, I = 8, 256, 512
    loc = np.array([6, 0, 7, 1, 2, 3, 4, 5], np.int32)  # experts 0 and 2 are cold
    fx = LayerFixture(H=H, I=I, E=E, n_hot=6, n_cold=2, k=1, seed=99, loc=loc)
    logits = _assigned_logits(counts, E, seed=3)
    T = logits.shape[0]
    x = synth.gen_x(T, H, seed=4)
    buf = _run(fx, logits, x)
    rc, ids, w, want = oracle.layer(logits, bf16_bits(x), 1, 0, H, I, fx.all_blobs_now(), act4=True)
    assert rc == 0
    assert np.array_equal(np.bincount(ids.ravel(), minlength=E), counts)
    got = buf.out.cpu().numpy()
    for e in range(E):  # every bucket on its own
        rows = np.nonzero(ids[:, 0] == e)[0]
        if rows.size:
            assert rel_l2(got[rows], want[rows]) <= OUT_TOL, e
    fx.layer.close()


def test_mx_decode_sized_calls_stay_unquantised():
    """Calls of at most 64 tokens run the decode kernel on unquantised activations
    whatever the prefill kind."""
    H, I, E, k, T = 256, 512, 16, 2, 40
    fx = LayerFixture(H=H, I=I, E=E, n_hot=12, n_cold=4, k=k, seed=8)
    logits = synth.gen_logits_uniform(T, E, seed=2)
    x = synth.gen_x(T, H, seed=3)
    buf = _run(fx, logits, x)
    rc, ids, w, want = oracle.layer(logits, bf16_bits(x), k, 0, H, I, fx.all_blobs_now())
    assert rel_l2(buf.out.cpu().numpy(), want) <= OUT_TOL
    fx.layer.close()


def _pass_positions(cnt, width=192, tile=16):
    pos = set()
    for s in range(0, cnt, width):
        e = min(cnt, s + width)
        pos.update({s, min(s + tile - 1, e - 1), max(s, e - tile), e - 1})
    return sorted(pos)


def test_mx_prefill_8192_every_bucket():
    """The 8192-token layer of 384 experts (H=4096, I=3072, top-6, all in HBM) on the
    block-scaled path: the first and last token of the first and last 16-token tile
    of every column pass of every expert bucket against the oracle's all-FP4 mode."""
    c = synth.CONFIGS["c4"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    fx = LayerFixture(H=H, I=I, E=E, n_hot=E, n_cold=0, k=k, seed=synth.sub_seed("c4", "blobs"))
    logits = synth.gen_logits_uniform(T, E, seed=synth.sub_seed("c4", "logits"))
    x = synth.gen_x(T, H, seed=synth.sub_seed("c4", "x"))
    buf = _run(fx, logits, x, out_fp32=False)
    rc, ids, w, counts, offsets, entries = oracle.route(logits, k)
    assert np.array_equal(buf.topk_ids.cpu().numpy()[:T], ids)
    picks = {}
    for e in range(E):
        for p in _pass_positions(int(counts[e])):
            i = int(entries[offsets[e] + p])
            picks[(i // k, i % k)] = e
    assert len(set(picks.values())) == E
    xs = oracle.bf16_bits_to_f64(bf16_bits(x))
    loc = fx.layer.get_loc()
    y = oracle_pick_rows(lambda e: fx.expert_bytes_now(e, loc), H, I, xs, picks, act4=True)
    ygpu = buf.y.cpu().numpy()
    worst = max(rel_l2(ygpu[t * k + j], y[(t, j)]) for (t, j) in picks)
    assert worst <= OUT_TOL, worst
    # whole tokens through the combine
    out = buf.out.float().cpu().numpy()
    for t in (0, 4097, T - 1):
        tj = {(t, j): int(ids[t, j]) for j in range(k)}
        yt = oracle_pick_rows(lambda e: fx.expert_bytes_now(e, loc), H, I, xs, tj, act4=True)
        want = sum(w[t, j] * yt[(t, j)] for j in range(k))
        assert rel_l2(out[t], want) <= OUT_TOL, t
    fx.layer.close()
