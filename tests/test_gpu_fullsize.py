"""Full-size GPU parity of the stacked-layer structure and of the large batches,
through the C ABI, against the CPU oracle.

- Three layers of the 384-expert shape (H=4096, I=3072, 255 in HBM, 129 cold)
  share one 129-slot scratch ("DeepSeek-V4.1-Flash on One GB300 Without the Second
  GPU", section 1: every layer uses the same scratch because layers run one after
  another), with skewed routing over starting hot sets drawn from a different
  permutation, so the residency manager swaps within the test.  After every step:
  routing, physical ids, cold lists and gathered slot bytes bit-exact; the
  placement map equal to the oracle's residency rule after every update (in the
  deferred mode one step after each window closes, in the synchronous mode at
  once); the
  fingerprint of every moved expert and of 64 random ones per layer unchanged
  wherever the expert now lives (same page, section 4: the byte audit); every
  token's output within the relative-L2 bar.
- The 8192-token prefill layer: the first and last token of the first and last
  16-token tile of every column pass of every expert bucket, against the oracle.
- The skewed decode batches of 8 and 32 tokens: every token.

Bars as in the other parity tests: ids, maps and bytes bit-exact; outputs within
relative L2 5e-3 of the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import LayerFixture, bf16_bits, fingerprints, oracle_pick_rows, rel_l2

pytestmark = pytest.mark.gpu

OUT_TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    oracle.build()


def _check_outputs(fx, buf, ids, w, x, tokens, loc):
    """Every pick's y row of the listed tokens and their combined outputs against
    the oracle (bytes read wherever `loc` places each expert)."""
    k = fx.k
    xs = oracle.bf16_bits_to_f64(bf16_bits(x))
    picks = {(t, j): int(ids[t, j]) for t in tokens for j in range(k)}
    y = oracle_pick_rows(lambda e: fx.expert_bytes_now(e, loc), fx.H, fx.I, xs, picks)
    ygpu = buf.y.cpu().numpy()
    out = buf.out.float().cpu().numpy()
    for t in tokens:
        want = np.zeros(fx.H)
        for j in range(k):
            r = rel_l2(ygpu[t * k + j], y[(t, j)])
            assert r <= OUT_TOL, (t, j, r)
            want += w[t, j] * y[(t, j)]
        r = rel_l2(out[t], want)
        assert r <= OUT_TOL, (t, r)


# ------------------------------------------------------------------ stacked layers

@pytest.mark.parametrize("host_mirror,defer", [(False, True), (True, True), (False, False)])
def test_shared_scratch_full_shape(host_mirror, defer):
    import moe_decode_host_gb300 as m

    c = synth.CONFIGS["c3"]
    H, I, E, n_hot, n_cold, k = c["H"], c["I"], c["E"], c["n_hot"], c["n_cold"], c["k"]
    NL, T, steps, swap_every, max_swaps, hyst = 3, 4, 8, 2, 8, 3.0
    eb = m.expert_bytes(H, I)
    slots = torch.empty((n_cold, eb), dtype=torch.uint8, device="cuda")
    scratch = m.Scratch(n_cold, eb, slots)
    layers = []
    for li in range(NL):
        perm = synth.zipf_permutation(E, synth.sub_seed("c3", "perm", li))
        other = synth.zipf_permutation(E, synth.sub_seed("c3", "hotset", li))
        loc = synth.loc_from_hot_set(E, n_hot, other[:n_hot])
        fx = LayerFixture(H=H, I=I, E=E, n_hot=n_hot, n_cold=n_cold, k=k, seed=synth.sub_seed("c3", "blobs", li),
                          loc=loc, scratch=scratch, slots=slots, swap_every=swap_every, max_swaps=max_swaps,
                          hysteresis=hyst, host_mirror=host_mirror, residency_defer=defer)
        fx.perm = perm
        fx.loc_o = loc.copy()    # the oracle's placement after every plan so far
        fx.loc_now = loc.copy()  # the placement the layer should hold now
        fx.pending = None        # deferred: (placement, promoted, demoted) of a closed window
        fx.window = np.zeros(E, np.int64)
        fx.fp0 = fingerprints(lambda e, fx=fx, l0=loc: fx.expert_bytes_now(e, l0), list(range(E)))
        layers.append(fx)
    rng = np.random.default_rng(3)
    total_swaps = 0
    for step in range(steps):
        for li, fx in enumerate(layers):
            logits = synth.gen_logits_zipf(T, E, c["s"], fx.perm, seed=synth.sub_seed("c3", "logits", li, step))
            x = synth.gen_x(T, H, seed=synth.sub_seed("c3", "x", li, step))
            loc = fx.layer.get_loc()
            assert np.array_equal(loc, fx.loc_now)
            buf = m.StepBuffers(fx.layer, T, out_fp32=True)
            m.moe_route(fx.layer, torch.from_numpy(logits).cuda(), T, buf.topk_ids, buf.topk_w, buf.counts,
                        buf.offsets, buf.entries)
            m.cold_gather(fx.layer, buf.topk_ids, T, buf.phys_ids, buf.cold_list, buf.n_cold_picked)
            m.moe_gather_join(fx.layer)
            torch.cuda.synchronize()
            # routing, remap and the gathered bytes, before the next layer reuses the slots
            rc, ids, w, counts, offsets, entries = oracle.route(logits, k)
            assert rc == 0
            assert np.array_equal(buf.topk_ids.cpu().numpy()[:T], ids)
            assert np.array_equal(buf.counts.cpu().numpy(), counts)
            assert np.array_equal(buf.entries.cpu().numpy()[:T * k], entries)
            phys, cold = oracle.remap(ids, loc, n_hot, n_cold)
            assert np.array_equal(buf.phys_ids.cpu().numpy()[:T * k].reshape(T, k), phys)
            n = int(buf.n_cold_picked.item())
            assert n == cold.size and np.array_equal(buf.cold_list.cpu().numpy()[:n], cold)
            owner = {int(loc[e]) - n_hot: e for e in range(E) if loc[e] >= n_hot}
            for cs in cold.tolist():
                assert np.array_equal(slots[cs].cpu().numpy(), fx.expert_bytes_now(owner[cs], loc)), (step, li, cs)
            m.moe_grouped_ffn(fx.layer, x.cuda(), T, buf.phys_ids, buf.counts, buf.offsets, buf.entries, buf.y,
                              buf.workspace)
            m.moe_combine(buf.y, buf.topk_w, T, k, H, buf.out, True)
            nsw = m.residency_update(fx.layer)
            torch.cuda.synchronize()
            assert fx.layer.status() == 0, fx.layer.diag().tolist()
            fx.window += counts
            landed = None
            if defer and fx.pending is not None:
                landed, fx.pending = fx.pending, None
            if (step + 1) % swap_every == 0:
                fx.loc_o, pro, dem = oracle.residency(fx.window.astype(np.int32), fx.loc_o, n_hot, max_swaps, hyst)
                fx.window[:] = 0
                if defer:
                    fx.pending = (fx.loc_o.copy(), pro, dem)
                else:
                    landed = (fx.loc_o.copy(), pro, dem)
            now = fx.layer.get_loc()
            if landed is not None:
                fx.loc_now, pro, dem = landed
                assert nsw == pro.size, (step, li)
                total_swaps += nsw
                assert np.array_equal(now, fx.loc_now), (step, li)
                audit = sorted(set(pro.tolist()) | set(dem.tolist()) | set(rng.choice(E, 64, replace=False).tolist()))
                fp = fingerprints(lambda e, fx=fx, l1=now: fx.expert_bytes_now(e, l1), audit)
                assert all(fp[e] == fx.fp0[e] for e in audit), (step, li)
            else:
                assert nsw == 0
                assert np.array_equal(now, fx.loc_now), (step, li)
            # outputs: the bytes each expert had when the FFN ran are its bytes now
            _check_outputs(fx, buf, ids, w, x, list(range(T)), fx.layer.get_loc())
    assert total_swaps > 0
    for fx in layers:
        now = fx.layer.get_loc()
        assert sorted(now.tolist()) == list(range(E))
        fp = fingerprints(lambda e, fx=fx, l1=now: fx.expert_bytes_now(e, l1), list(range(E)))
        assert fp == fx.fp0
        fx.layer.close()


# ------------------------------------------------------------------ large batches

def _run(fx, logits, x, out_fp32):
    import moe_decode_host_gb300 as m

    T = logits.shape[0]
    buf = m.StepBuffers(fx.layer, T, out_fp32=out_fp32)
    m.run_step(fx.layer, buf, torch.from_numpy(logits).cuda(), x.cuda(), residency=False)
    torch.cuda.synchronize()
    assert fx.layer.status() == 0, fx.layer.diag().tolist()
    return buf


def _pass_positions(cnt, width=160, tile=16):
    """Bucket positions that sample every column pass of `width` tokens: the first
    and last token of its first and last 16-token tile."""
    pos = set()
    for s in range(0, cnt, width):
        e = min(cnt, s + width)
        pos.update({s, min(s + tile - 1, e - 1), max(s, e - tile), e - 1})
    return sorted(pos)


def test_prefill_8192_every_bucket():
    c = synth.CONFIGS["c4"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    fx = LayerFixture(H=H, I=I, E=E, n_hot=E, n_cold=0, k=k, seed=synth.sub_seed("c4", "blobs"))
    logits = synth.gen_logits_uniform(T, E, seed=synth.sub_seed("c4", "logits"))
    x = synth.gen_x(T, H, seed=synth.sub_seed("c4", "x"))
    buf = _run(fx, logits, x, False)
    rc, ids, w, counts, offsets, entries = oracle.route(logits, k)
    assert np.array_equal(buf.topk_ids.cpu().numpy()[:T], ids)
    assert counts.min() > 64  # every bucket on the tensor cores (two-pass buckets: the bucket-edge test)
    picks = {}
    for e in range(E):
        for p in _pass_positions(int(counts[e])):
            i = int(entries[offsets[e] + p])
            picks[(i // k, i % k)] = e
    assert len(set(picks.values())) == E
    xs = oracle.bf16_bits_to_f64(bf16_bits(x))
    loc = fx.layer.get_loc()
    y = oracle_pick_rows(lambda e: fx.expert_bytes_now(e, loc), H, I, xs, picks)
    ygpu = buf.y.cpu().numpy()
    worst = max(rel_l2(ygpu[t * k + j], y[(t, j)]) for (t, j) in picks)
    assert worst <= OUT_TOL, worst
    # and whole tokens through the combine: the first, a middle and the last
    _check_outputs(fx, buf, ids, w, x, [0, 4097, T - 1], loc)
    fx.layer.close()


@pytest.mark.parametrize("T,s", [(8, 1.1), (32, 1.1), (32, 1.5)])
def test_skewed_decode_batches_every_token(T, s):
    c = synth.CONFIGS["c2"]
    perm = synth.zipf_permutation(c["E"], synth.sub_seed("c2", "perm"))
    loc = synth.loc_from_hot_set(c["E"], c["n_hot"], perm[:c["n_hot"]])
    fx = LayerFixture(H=c["H"], I=c["I"], E=c["E"], n_hot=c["n_hot"], n_cold=c["n_cold"], k=c["k"],
                      seed=synth.sub_seed("c2", "blobs"), loc=loc)
    logits = synth.gen_logits_zipf(T, c["E"], s, perm, seed=synth.sub_seed("c2", "logits", T, s))
    x = synth.gen_x(T, c["H"], seed=synth.sub_seed("c2", "x", T))
    buf = _run(fx, logits, x, False)
    rc, ids, w, *_ = oracle.route(logits, c["k"])
    assert np.array_equal(buf.topk_ids.cpu().numpy()[:T], ids)
    _check_outputs(fx, buf, ids, w, x, list(range(T)), fx.layer.get_loc())
    fx.layer.close()
