"""Benchmark of the MoE decode layer with host-resident cold experts on GB300.

One step = one pass of the whole path over one batch: moe_route -> cold_gather ->
moe_grouped_ffn -> moe_combine -> residency_update (acting every 16 steps with
hysteresis 3.0 and at most 8 swaps).  Default workload: one layer with H=4096,
I=3072, 384 experts (255 in HBM, 129 in pinned host memory), top-6, one decode
token per step, router logits N(0,1).  Steps cycle over a pool of 64 distinct
routings; the 7.7 GB weight pool is far larger than L2, so no L2 flush is used.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

HBM_NOMINAL_GBS = 8000.0


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per unit of work,
# from the ncu captures summarised under profiles/ (a smaller layer of the same
# expert shape; traffic scales with the experts processed).  An entry is set to
# None whenever its kernel changes after the capture.
NCU_TRAFFIC = {
    # per cold expert copied: the slot writes stay in L2 during the launch
    "cold_copy": {"bytes_per_expert": (11520 + 15616) / 2,
                  "source": "profiles/cold_copy_kernel_c1_small.md"},
    # per distinct expert through the decode kernels (gate/up + down launches)
    "ffn_decode": {"bytes_per_expert": (66931968 + 642560 + 33490432) / 5,
                   "source": "profiles/ffn_decode_kernel_c1_small.md"},
    # per expert through the tcgen05 kernels at about 128 tokens per expert: the
    # capture (935596288 + 92993792 + 483277568 + 112975360 bytes over 64 experts)
    # predates the converters' scale-word prefetch, so no figure is reported
    "ffn_tc": {"bytes_per_expert": None,
               "source": "profiles/ffn_tc_kernel_c4_small.md (counters of the previous kernel build)"},
}


def _traffic(kind, experts_per_call):
    t = NCU_TRAFFIC.get(kind)
    if not t:
        return None, None
    if t.get("bytes_per_expert") is None:
        return None, t.get("source")
    return float(t["bytes_per_expert"] * experts_per_call), t["source"]


def _tensor_peak():
    """Dense f16/bf16 tensor peak: the measured sustained cuBLAS bf16 rate (the
    kernel is timed inside a long step loop); kind::f16 with f16 operands runs at
    the bf16 rate."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured (bf16_tflops_sustained; f16 runs at the bf16 rate)"
    except Exception:
        return 1700.0, "fallback (sustained bf16)"


FP4_OVER_BF16 = 6.0  # nominal dense tensor rates per GPU: 13.5 PFLOP/s MXFP4 over 2.25 bf16


def prefill_targets(flops: float, algo_bytes: float, ms: float, tc_peak_tflops: float, hbm_gbs: float) -> dict:
    """The prefill config against its own target, a fraction of the dense MXFP4
    tensor peak: that peak is not measured here, so it is the measured bf16 peak
    times the nominal FP4/bf16 ratio. The workload's irreducible bytes (each
    picked expert's weights once, x in and the output out) cap what any kernel can
    reach: flops / (bytes / HBM peak)."""
    achieved = flops / (ms * 1e-3) / 1e12
    mxfp4_peak = tc_peak_tflops * FP4_OVER_BF16
    cap = flops / (algo_bytes / (hbm_gbs * 1e9)) / 1e12
    return {"achieved_tflops": achieved, "mxfp4_peak_tflops": mxfp4_peak,
            "mxfp4_peak_kind": "measured bf16 x 6 (nominal dense FP4/bf16 ratio)",
            "frac_of_mxfp4_peak": achieved / mxfp4_peak,
            "hbm_bound_cap_tflops": cap, "frac_of_hbm_bound_cap": achieved / cap,
            "flop_per_byte": flops / algo_bytes}


def repetition_bounds(K: int, n: int = 5) -> list:
    """Step indices splitting K timed steps into n repetitions of (nearly) equal
    length: [0, ..., K]; fewer repetitions when K < n (one step each)."""
    n = max(1, min(n, K))
    return [round(K * j / n) for j in range(n + 1)]


def repetition_spread(bounds: list, rep_ms: list, tokens_per_step: int) -> dict:
    """Throughput of each repetition (this rank's clock) and their median, min and
    max, in the line's unit."""
    vals = [tokens_per_step * (bounds[j + 1] - bounds[j]) / (ms * 1e-3) for j, ms in enumerate(rep_ms)]
    return {"n": len(vals), "steps_each": [bounds[j + 1] - bounds[j] for j in range(len(vals))],
            "tokens_per_s": vals, "median": float(np.median(vals)), "min": float(min(vals)),
            "max": float(max(vals)), "note": "the timed region split at event marks; rank 0's clock"}


def skew_share(counts, frac_experts: float = 0.73) -> float:
    """Share of the picks that land on the most-picked `frac_experts` of the
    experts (the skew statistic the pages quote: 98.7% of picks on 73% of
    experts), per layer over all timed steps, pooled over layers.
    counts: int [steps, layers, E] picks per expert."""
    per_layer = np.asarray(counts, dtype=np.int64).sum(axis=0)  # [layers, E]
    n_top = int(round(frac_experts * per_layer.shape[1]))
    top = np.sort(per_layer, axis=1)[:, ::-1][:, :n_top].sum()
    return float(top / max(1, per_layer.sum()))


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8000)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c1", choices=["c1", "c2", "c3", "c4", "v1"])
    ap.add_argument("--batch", type=int, default=None, help="tokens per step (c2/c3: 8 or 32)")
    ap.add_argument("--skew", type=float, default=None, help="Zipf exponent for skewed routing")
    ap.add_argument("--layers", type=int, default=None, help="layers for c3")
    ap.add_argument("--pool", type=int, default=64)
    ap.add_argument("--residency", dest="no_residency", action="store_false", default=None,
                    help="run the residency manager (default: only where the workload specifies it, the "
                         "20-layer stack)")
    ap.add_argument("--no-residency", dest="no_residency", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--experts", type=int, default=None, help="override E (profiling on a smaller layer)")
    ap.add_argument("--hot", type=int, default=None, help="override n_hot (with --experts)")
    ap.add_argument("--no-link-probe", action="store_true")
    ap.add_argument("--copy-ctas", type=int, default=0, help="CTAs of the cold copy kernel (0 = library default)")
    ap.add_argument("--mirror", dest="mirror", action="store_true", default=None,
                    help="keep a pinned host copy of every expert (residency moves bytes one way only); "
                         "default on for single-layer workloads")
    ap.add_argument("--no-mirror", dest="mirror", action="store_false")
    ap.add_argument("--hysteresis", type=float, default=3.0, help="residency threshold ratio")
    ap.add_argument("--swap-every", type=int, default=16, help="residency update interval in steps")
    ap.add_argument("--max-swaps", type=int, default=8, help="swaps per residency update")
    ap.add_argument("--n-hot", type=int, default=None, help="HBM-resident experts per layer (rest cold)")
    ap.add_argument("--zero-copy", action="store_true",
                    help="the FFN reads picked cold experts in place from host memory (no slot copy)")
    return ap.parse_args()


def workload(args):
    import synth

    c = dict(synth.CONFIGS[args.config])
    if args.no_residency is None:
        # residency only where the workload asks for it (the stacked-layer config)
        args.no_residency = "swap_every" not in c
    if args.batch is not None:
        c["T"] = args.batch
    if args.skew is not None:
        c["s"] = args.skew
    if args.layers is not None:
        c["layers"] = args.layers
    if args.experts is not None:
        c["E"] = args.experts
        c["n_hot"] = args.hot if args.hot is not None else min(c["n_hot"], args.experts)
        c["n_cold"] = c["E"] - c["n_hot"]
    c["name"] = args.config
    # host copies of every expert: default for one layer (7.7 GB pinned); a 20-layer
    # stack would need 154 GB of pinned host memory, so it keeps the in-place exchange
    c["mirror"] = args.mirror if args.mirror is not None else (
        c.get("layers", 1) == 1 and c["n_cold"] > 0 and not args.no_residency)
    c["zero_copy"] = bool(args.zero_copy)
    if args.n_hot is not None and args.experts is None:
        c["n_hot"] = min(args.n_hot, c["E"])
        c["n_cold"] = c["E"] - c["n_hot"]
    c["hysteresis"], c["swap_every_steps"], c["max_swaps"] = args.hysteresis, args.swap_every, args.max_swaps
    return c


def _rank_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(dist, value: float, device) -> float:
    """The largest of every rank's value (the slowest replica's elapsed time); the
    value itself on a single process."""
    if not dist:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, steps: int, tokens_per_step: int, elapsed_ms: float) -> float:
    """Whole-job tokens/s: every replica processes its own steps, timed by the
    slowest replica."""
    return world * steps * tokens_per_step / (elapsed_ms * 1e-3)


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ reference arm (CPU oracle)

ORACLE_TOKENS_PER_CALL = 8  # one oracle token of the 384-expert layer takes about two seconds


def oracle_tokens_per_s(c, seconds: float, seed_tag="cpu"):
    """Times the CPU oracle on a bounded sample of the workload: whole tokens of
    the layer (route + every pick's expert FFN + combine), expert bytes drawn by the
    seeded generator on the CPU.  The oracle runs every pick on its own token, so
    its time per token does not depend on the batch: each call takes the first
    ORACLE_TOKENS_PER_CALL tokens of a seeded step of the workload (routing is per
    token, so they route as they do in the whole step).  Returns (tokens/s, tokens,
    seconds, sample text)."""
    import torch

    import oracle
    import synth

    H, I, E, k = c["H"], c["I"], c["E"], c["k"]
    T_step = max(1, c["T"])
    T = min(T_step, ORACLE_TOKENS_PER_CALL)
    oracle.build()
    tok = 0
    t_total = 0.0
    blob_cache = {}
    step = 0
    while t_total < seconds or tok == 0:
        if c.get("routing") == "zipf":
            perm = synth.zipf_permutation(E, synth.sub_seed(c["name"], "perm"))
            logits = synth.gen_logits_zipf(T_step, E, c.get("s", 1.1), perm, seed=synth.sub_seed(seed_tag, step))
        elif c.get("routing") == "verify":
            logits = synth.gen_logits_verify(T_step, E, seed=synth.sub_seed(seed_tag, step))
        else:
            logits = synth.gen_logits_uniform(T_step, E, seed=synth.sub_seed(seed_tag, step))
        x = synth.gen_x(T_step, H, seed=synth.sub_seed(seed_tag, "x", step))
        logits = np.ascontiguousarray(logits[:T])
        bits = np.ascontiguousarray(x[:T].view(torch.int16).numpy().view(np.uint16))
        # expert bytes are generated outside the timed region (they are inputs)
        _, ids, _, _, _, _ = oracle.route(logits, k)
        blobs = []
        picked = set(ids.ravel().tolist())
        for e in range(E):
            if e in picked:
                if e not in blob_cache:
                    blob_cache[e] = synth.gen_blobs(1, H, I, seed=synth.sub_seed(seed_tag, "blob", e))[0].numpy()
                blobs.append(blob_cache[e])
            else:
                blobs.append(blob_cache.get(e, np.zeros(1, np.uint8)))
        t0 = time.perf_counter()
        rc, _, _, out = oracle.layer(logits, bits, k, 0, H, I, blobs)
        t_total += time.perf_counter() - t0
        assert rc == 0
        tok += T
        step += 1
        if len(blob_cache) > 64:
            blob_cache.clear()
    sample = (f"{tok} token(s) of the {c['name']} layer (the first {T} of a {T_step}-token step, {step} "
              f"step(s)): route, {k} expert FFNs per token, combine; single-threaded C oracle, fp64")
    return tok / t_total, tok, t_total, sample


def run_reference(args, budget_s: float = 150.0):
    """The CPU oracle as the reference arm, on this arm's workload and metric.  Each
    step is one batch of the workload's tokens through the whole oracle layer; the
    number of timed steps is capped so the run ends within a few minutes (one
    oracle token of the 384-expert layer takes seconds)."""
    rank, world, _ = _rank_env()
    if rank != 0:
        return
    c = workload(args)
    oracle_tokens_per_s(c, 0.0, seed_tag="ref-warm") if args.warmup > 0 else None
    t_steps = []
    tok_total = 0
    sample = ""
    for s in range(max(1, args.steps)):
        v, tok, secs, sample = oracle_tokens_per_s(c, 0.0, seed_tag=f"ref{s}")
        t_steps.append(secs)
        tok_total += tok
        if sum(t_steps) + secs > budget_s:
            break
    total = sum(t_steps)
    value = tok_total / total
    n = len(t_steps)
    sample = (f"{n} step(s) of {min(max(1, c['T']), ORACLE_TOKENS_PER_CALL)} token(s) (the first of each "
              f"{c['T']}-token step) of the {c['name']} layer (of {args.steps} requested; capped "
              f"at {budget_s:.0f} s of oracle time): route, {c['k']} expert FFNs per token, combine; "
              f"single-threaded C oracle, fp64")
    line = {"impl": "reference", "metric": "MoE layer tokens/s (decode)", "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": n, "steps_requested": args.steps, "warmup": min(args.warmup, 1),
            "ms_per_step": 1000.0 * total / n, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config_json(c, args),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _config_json(c, args):
    return {"workload": f"{c['name']}: MoE layer H={c['H']} I={c['I']} E={c['E']} ({c['n_hot']} HBM / "
                        f"{c['n_cold']} pinned host) top-{c['k']}, {c['T']} token(s)/step, "
                        f"{'Zipf s=%.2f' % c.get('s', 1.1) if c.get('routing') == 'zipf' else ('verify-window (6 tokens of one sequence, correlated)' if c.get('routing') == 'verify' else 'uniform')} routing"
                        + (f", {c['layers']} layers sharing one slot scratch" if c.get("layers", 1) > 1 else ""),
            "tokens_per_step": c["T"], "layers": c.get("layers", 1),
            "residency": "off" if args.no_residency else (
                "every %d steps, hysteresis %g, <=%d swaps, " % (c["swap_every_steps"], c["hysteresis"], c["max_swaps"]) + (
                "host copy of every expert" if c.get("mirror") else "in-place HBM/host exchange")),
            "step_pool": (min(max(args.pool, args.steps + args.warmup), 2048)
                          if (not args.no_residency and c["n_cold"] > 0) else args.pool),
            "l2": "inputs larger than L2 (7.7 GB expert pool per layer), no flush",
            "cold_experts": ("read in place from pinned host memory by the FFN (zero copy)"
                             if c.get("zero_copy") and c["T"] <= 64 else "copied into the HBM slot scratch"),
            "parallelism": "replicas" if args.gpus > 1 else "single GPU"}


# ------------------------------------------------------------------ our arm

def build_layers(c, dev, seed_tag="bench"):
    import torch

    import moe_decode_host_gb300 as m
    import synth

    H, I, E, k, n_hot, n_cold = c["H"], c["I"], c["E"], c["k"], c["n_hot"], c["n_cold"]
    eb = m.expert_bytes(H, I)
    L = c.get("layers", 1)
    slots = torch.empty((max(1, n_cold), eb), dtype=torch.uint8, device=dev)
    scratch = m.Scratch(n_cold, eb, slots) if n_cold > 0 else None
    layers = []
    for li in range(L):
        if c["name"] in ("c2",):
            perm = synth.zipf_permutation(E, synth.sub_seed(c["name"], "perm", li))
            loc = synth.loc_from_hot_set(E, n_hot, perm[:n_hot])
        elif c["name"] == "c3":
            perm = synth.zipf_permutation(E, synth.sub_seed(c["name"], "perm", li))
            other = synth.zipf_permutation(E, synth.sub_seed(c["name"], "hotset", li))
            loc = synth.loc_from_hot_set(E, n_hot, other[:n_hot])
        else:
            perm = None
            loc = synth.loc_identity(E, n_hot)
        hot = torch.empty((max(1, n_hot), eb), dtype=torch.uint8, device=dev)
        mirror = bool(c.get("mirror"))
        if mirror:
            # a pinned host copy of every expert (indexed by expert id)
            cold = torch.empty((E, eb), dtype=torch.uint8, pin_memory=True)
            synth.fill_layer(hot, None, loc, H, I, synth.sub_seed(seed_tag, c["name"], li), device=dev, mirror=cold)
        else:
            cold = torch.empty((max(1, n_cold), eb), dtype=torch.uint8, pin_memory=True)
            synth.fill_layer(hot, cold, loc, H, I, synth.sub_seed(seed_tag, c["name"], li), device=dev)
        n_host = E if mirror else n_cold
        layer = m.Layer(E=E, k=k, H=H, I=I, n_hot=n_hot, n_cold=n_cold, scratch=scratch,
                        hot_ptrs=[hot[h] for h in range(n_hot)], cold_ptrs=[cold[i] for i in range(n_host)],
                        init_loc=loc, swap_every=0 if c.get("no_res") else c["swap_every_steps"],
                        max_swaps=c["max_swaps"], hysteresis=c["hysteresis"],
                        host_mirror=mirror, zero_copy=bool(c.get("zero_copy")))
        layers.append(dict(layer=layer, hot=hot, cold=cold, perm=perm))
    return layers, scratch, slots


def gen_pool(c, layers, P, PL, dev):
    """Inputs of PL distinct steps: entry i holds, per layer, the logits of step i and
    the activations of step i % P.  Routing never repeats within PL steps, so with
    PL large the residency manager sees the workload's picking frequencies rather
    than a short loop it could learn."""
    import torch

    import synth

    T, E, H = c["T"], c["E"], c["H"]
    xs = [[synth.gen_x(T, H, seed=synth.sub_seed(c["name"], "x", li, p)).to(dev) for li in range(len(layers))]
          for p in range(min(P, PL))]
    pool = []
    for p in range(PL):
        per_layer = []
        for li, L in enumerate(layers):
            if c.get("routing") == "zipf":
                lg = synth.gen_logits_zipf(T, E, c.get("s", 1.1), L["perm"],
                                           seed=synth.sub_seed(c["name"], "logits", li, p))
            elif c.get("routing") == "verify":
                lg = synth.gen_logits_verify(T, E, seed=synth.sub_seed(c["name"], "logits", li, p))
            else:
                lg = synth.gen_logits_uniform(T, E, seed=synth.sub_seed(c["name"], "logits", li, p))
            per_layer.append((torch.from_numpy(lg).to(dev), xs[p % len(xs)][li], lg))
        pool.append(per_layer)
    return pool


def measure_link_peak(dev):
    """Host-link read peak: max of a pinned H2D cudaMemcpyAsync and the zero-copy
    16-byte-load probe kernel (the same loop as cold_gather), 1 GiB each."""
    import torch

    import moe_decode_host_gb300 as m

    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8).pin_memory()
    src.fill_(1)
    dst = torch.empty(n, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream()
    res = {}
    for name in ("memcpy", "zero_copy"):
        best = 0.0
        for _ in range(4):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(st)
            if name == "memcpy":
                dst.copy_(src, non_blocking=True)
            else:
                m.link_probe(src, dst, n, 0, st)
            e1.record(st)
            e1.synchronize()
            best = max(best, n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
        res[name] = best
    del src, dst
    return max(res.values()), res


def run_ours(args):
    import torch

    import moe_decode_host_gb300 as m

    rank, world, local = _rank_env()
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist = dist_mod
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    c = workload(args)
    c["no_res"] = args.no_residency
    hbm_peak, peak_kind = _peaks()
    if args.no_link_probe:
        link_peak, link_detail = None, {"skipped": True}
    else:
        link_peak, link_detail = measure_link_peak(dev)
    layers, scratch, slots = build_layers(c, dev)
    # with residency on, routing comes from up to 2048 distinct steps (no short loop)
    resid = not args.no_residency and c["n_cold"] > 0
    P = min(max(args.pool, args.steps + args.warmup), 2048) if resid else args.pool
    pool = gen_pool(c, layers, args.pool, P, dev)
    T, k, H, E = c["T"], c["k"], c["H"], c["E"]
    eb = m.expert_bytes(H, c["I"])
    NL = len(layers)
    bufs = [m.StepBuffers(L["layer"], T) for L in layers]
    for L in layers:
        L["layer"].set_copy_ctas(args.copy_ctas)
    K, W = args.steps, args.warmup
    counts_log = torch.zeros((K, NL, E), dtype=torch.int32, device=dev)
    ncold_log = torch.zeros((K, NL), dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()
    nev = 6

    def step(i, timed, ev=None):
        swaps = 0
        launches = 0
        for li, L in enumerate(layers):
            lg, x, _ = pool[i % P][li]
            b = bufs[li]
            layer = L["layer"]
            counts = counts_log[i, li] if timed else b.counts
            ncold = ncold_log[i, li] if timed else b.n_cold_picked
            if ev is not None:
                ev[li][0].record(st)
            m.moe_route(layer, lg, T, b.topk_ids, b.topk_w, counts, b.offsets, b.entries, st)
            if ev is not None:
                ev[li][1].record(st)
            m.cold_gather(layer, b.topk_ids, T, b.phys_ids, b.cold_list, ncold, st)
            if ev is not None:
                ev[li][2].record(st)
            m.moe_grouped_ffn(layer, x, T, b.phys_ids, counts, b.offsets, b.entries, b.y, b.workspace, stream=st)
            if ev is not None:
                ev[li][3].record(st)
            m.moe_combine(b.y, b.topk_w, T, k, H, b.out, False, st)
            if ev is not None:
                ev[li][4].record(st)
            n = m.residency_update(layer, st)
            if ev is not None:
                ev[li][5].record(st)
            swaps += n
            launches += step_launches(T, c["n_cold"]) + (1 if n > 0 else 0)
        return swaps, launches

    for i in range(W):
        step(i, False)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    # per-call events go in a separate pass after the timed region (below); inside it
    # only the library's own events around the cold copy and the FFN kernels run
    Kb = min(K, 256)
    events = [[[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(NL)] for _ in range(Kb)]
    for L in layers:
        L["layer"].profile(K)  # events around each cold copy, on the layer's copy stream
    clocks = Clocks(local)
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # the timed steps also fall into five repetitions, marked by an event at each
    # inner boundary (four records in the whole region), for the spread
    bounds = repetition_bounds(K)
    marks = {b: torch.cuda.Event(enable_timing=True) for b in bounds[1:-1]}
    torch.cuda.synchronize()
    t_start.record(st)
    total_swaps = 0
    launches = 0
    for i in range(K):
        s, n = step(i, True)
        total_swaps += s
        launches += n
        if i + 1 in marks:
            marks[i + 1].record(st)
    t_end.record(st)
    torch.cuda.synchronize()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(dist, t_start.elapsed_time(t_end), dev)
    try:
        evs = [t_start] + [marks[b] for b in bounds[1:-1]] + [t_end]
        rep_ms = [evs[j].elapsed_time(evs[j + 1]) for j in range(len(evs) - 1)]
        repetitions = repetition_spread(bounds, rep_ms, T * world)
    except Exception as exc:  # the spread is an addition; it never costs the line
        repetitions = {"error": str(exc)[:200]}
    if dist:
        dist.barrier()
    copy_ms = [L["layer"].profile_read(K) for L in layers]
    ffn_kern_ms = np.array([L["layer"].profile_read_ffn(K) for L in layers]).T  # [K, NL]
    for L in layers:
        L["layer"].profile(0)
    # per-call durations: Kb further steps with events around every call
    for i in range(Kb):
        step(K + i, False, events[i])
    torch.cuda.synchronize()
    names = ["moe_route", "cold_gather", "moe_grouped_ffn", "moe_combine", "residency_update"]
    per = {n: [] for n in names}
    for i in range(Kb):
        for li in range(NL):
            ev = events[i][li]
            for j, n in enumerate(names):
                per[n].append(ev[j].elapsed_time(ev[j + 1]))
    counts_h = counts_log.cpu().numpy()
    ncold_h = ncold_log.cpu().numpy()
    distinct = (counts_h > 0).sum(axis=2)  # [K, NL]
    act_bytes = T * H * 2 + T * k * (H * 4 + c["I"] * 4 * 2) + T * H * 2  # x, y, h write+read, x16
    ffn_bytes = distinct * eb + act_bytes
    gather_bytes = ncold_h * eb
    hot_bytes = (distinct - ncold_h) * eb
    # FFN kernel time without the wait for the cold copy (recorded by the library)
    ffn_k_tot_ms = float(ffn_kern_ms.sum())
    ffn_gbs = float(ffn_bytes.sum() / (ffn_k_tot_ms * 1e-3) / 1e9)
    ffn_flops = 2.0 * 3.0 * H * c["I"] * T * k * K * NL
    ffn_tflops = ffn_flops / (ffn_k_tot_ms * 1e-3) / 1e12
    # the copy runs on the layer's copy stream, overlapped with the FFN: its duration
    # comes from the events the library records around it on that stream
    copy_tot_ms = float(sum(float(np.sum(c)) for c in copy_ms))
    n_copies = int(sum(len(c) for c in copy_ms))
    gather_gbs = float(gather_bytes.sum() / (copy_tot_ms * 1e-3) / 1e9) if copy_tot_ms > 0 else 0.0
    lp = link_peak if link_peak else float("inf")
    tstar_nom = np.maximum(hot_bytes / (HBM_NOMINAL_GBS * 1e9), gather_bytes / (lp * 1e9))
    tstar_meas = np.maximum(hot_bytes / (hbm_peak * 1e9), gather_bytes / (lp * 1e9))
    step_ms = elapsed_ms / K
    value = job_rate(world, K, T, elapsed_ms)
    # dominant kernel: the one with the most GPU time over the timed region, the cold
    # copy (on the copy stream) or the FFN call's kernels (wait for the copy excluded)
    tot = {n: float(np.sum(per[n])) for n in names}
    dom = "cold_gather" if copy_tot_ms > ffn_k_tot_ms else "moe_grouped_ffn"
    mean_distinct = float(distinct.mean())
    mean_cold = float(ncold_h.mean())
    if dom == "moe_grouped_ffn" and T > 64:
        tc_peak, tc_kind = _tensor_peak()
        tr, src = _traffic("ffn_tc", mean_distinct)
        roof = {"kernel": "moe_grouped_ffn (tcgen05 kind::f16 grouped GEMM for buckets > 64 tokens)",
                "bound": "tensor", "achieved": ffn_tflops, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": ffn_tflops / tc_peak, "traffic": tr, "traffic_source": src,
                "algorithmic_bytes_per_call": float(ffn_bytes.sum() / (K * NL)),
                "ms_mean": ffn_k_tot_ms / (K * NL), "flops_per_call": ffn_flops / (K * NL), "peak_kind": tc_kind,
                "hbm_gbs_same_calls": ffn_gbs,
                "prefill_target": prefill_targets(ffn_flops, float((distinct * eb).sum()) + K * NL * 2.0 * T * H * 2,
                                                  ffn_k_tot_ms, tc_peak, hbm_peak)}
    elif dom == "moe_grouped_ffn":
        tr, src = _traffic("ffn_decode", mean_distinct)
        roof = {"kernel": "moe_grouped_ffn (decode dequant-GEMV)", "bound": "hbm", "achieved": ffn_gbs,
                "peak": hbm_peak, "unit": "GB/s", "frac": ffn_gbs / hbm_peak, "traffic": tr,
                "traffic_source": src, "algorithmic_bytes_per_call": float(ffn_bytes.sum() / (K * NL)),
                "ms_mean": ffn_k_tot_ms / (K * NL), "peak_kind": peak_kind}
    else:
        tr, src = _traffic("cold_copy", mean_cold)
        roof = {"kernel": "cold_copy_kernel (cold_gather's zero-copy host reads)", "bound": "link",
                "achieved": gather_gbs, "launches": n_copies, "ms_mean": copy_tot_ms / max(1, n_copies),
                "peak": link_peak, "unit": "GB/s", "frac": gather_gbs / link_peak if link_peak else None,
                "traffic": tr, "traffic_source": src,
                "traffic_note": "DRAM bytes only: the copy reads host memory over the C2C link and its slot "
                                "writes stay in L2 during the launch",
                "algorithmic_bytes_per_launch": float(gather_bytes.sum() / max(1, n_copies)),
                "peak_kind": "measured in this run (max of pinned cudaMemcpyAsync and zero-copy probe)"}
    line = {"metric": "MoE layer tokens/s (decode)", "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e2m1xf16->f32", "data": "synthetic", "config": _config_json(c, args),
            "roofline": roof,
            "kernels": {n: {"ms_mean": float(np.mean(per[n])), "share": tot[n] / max(1e-9, sum(tot.values()))}
                        for n in names},
            "kernels_note": "per-call CUDA events over %d further steps run after the timed region" % Kb,
            "step_roofline": {"tstar_ms_nominal_hbm": float(1e3 * tstar_nom.sum() / K),
                              "frac_nominal": float(1e3 * tstar_nom.sum() / K / step_ms),
                              "tstar_ms_measured_hbm": float(1e3 * tstar_meas.sum() / K),
                              "frac_measured": float(1e3 * tstar_meas.sum() / K / step_ms),
                              "hbm_peak_gbs": hbm_peak, "link_peak_gbs": link_peak, "link_probe": link_detail},
            "ffn_hbm_gbs": ffn_gbs, "ffn_kernel_ms_mean": ffn_k_tot_ms / (K * NL), "gather_link_gbs": gather_gbs,
            "distinct_experts_per_layer_step": float(distinct.mean()),
            "picks_on_top_73pct_experts": skew_share(counts_h),
            "repetitions": repetitions,
            "cold_experts_per_layer_step": float(ncold_h.mean()), "swaps": int(total_swaps),
            "clocks": clk, "gpu_launches": int(launches),
            "device_status": [int(L["layer"].status()) for L in layers]}
    if not args.no_e2e:
        line["e2e"] = run_e2e(args, c, layers, pool, bufs, dev, dist, world)
    if rank == 0 and not args.no_cpu:
        v, tok, secs, sample = oracle_tokens_per_s(c, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def step_launches(T, n_cold):
    """Kernels one layer-step launches (residency swap kernel excluded)."""
    route = 1 if T <= 64 else 2                      # one-CTA route, or top-k + bucketing
    gather = 1 + (1 if n_cold > 0 else 0)            # remap, byte copy on the copy stream
    calls = 4 if n_cold > 0 else 2                   # FFN phases: (gate/up, down) x (hot, cold)
    per_call = 1 + (1 if T > 8 else 0) + (1 if T > 16 else 0) + (2 if T > 64 else 0)  # decode ranges, gather + tcgen05
    ffn = 1 + calls * per_call + calls // 2          # activation prep, phases, h prescale per down phase
    return route + gather + ffn + 1                  # + combine


def run_e2e(args, c, layers, pool, bufs, dev, dist, world):
    """Same steps through the public API with host buffers: pinned host logits and x
    copied in, the layer output copied back, every step, inside the timed region."""
    import torch

    import moe_decode_host_gb300 as m

    T, k, H, E = c["T"], c["k"], c["H"], c["E"]
    P = len(pool)
    NL = len(layers)
    host_in = [[(torch.from_numpy(pool[p][li][2]).pin_memory(), pool[p][li][1].cpu().pin_memory())
                for li in range(NL)] for p in range(P)]
    d_lg = [torch.empty((T, E), dtype=torch.float32, device=dev) for _ in range(NL)]
    d_x = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(NL)]
    host_out = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(NL)]
    st = torch.cuda.current_stream()
    K = max(1, args.steps)

    def step(i):
        for li, L in enumerate(layers):
            lg_h, x_h = host_in[i % P][li]
            d_lg[li].copy_(lg_h, non_blocking=True)
            d_x[li].copy_(x_h, non_blocking=True)
            m.run_step(L["layer"], bufs[li], d_lg[li], d_x[li], st, residency=not args.no_residency)
            host_out[li].copy_(bufs[li].out[:T], non_blocking=True)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(K):
        step(i)
    e1.record(st)
    torch.cuda.synchronize()
    ms = max_over_ranks(dist, e0.elapsed_time(e1), dev)
    return {"value": job_rate(world, K, T, ms), "unit": "tokens/s",
            "h2d_bytes_per_step": NL * (T * E * 4 + T * H * 2), "d2h_bytes_per_step": NL * T * H * 2}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
