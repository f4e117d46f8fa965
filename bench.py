"""Benchmark of the MoE decode layer with host-resident cold experts on GB300.

One step = one pass of the whole path over one batch: moe_route -> cold_gather ->
moe_grouped_ffn -> moe_combine -> residency_update (acting every 16 steps with
hysteresis 3.0 and at most 8 swaps where the workload runs the residency manager).
Default workload: one layer with H=4096, I=3072, 384 experts (255 in HBM, 129 in
pinned host memory), top-6, one decode token per step, router logits N(0,1); the
same line also carries the layer at decode batches of 8 and 32 tokens with Zipf
s=1.1 routing (`per_batch`).  Steps draw their routing from a pool of distinct
steps; the 7.7 GB weight pool is far larger than L2, so no L2 flush is used.

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

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per unit of work, from
# ncu captures of a smaller layer of the same expert shape (traffic scales with the
# experts processed).  None once the kernel has changed since its capture.
NCU_TRAFFIC = {
    "cold_copy": (11776 + 11776) / 1,                       # per cold expert copied (both launches)
    "ffn_decode": (66932992 + 728576 + 33495040) / 5,      # dequant-GEMV, per distinct expert, both phases
    "ffn_mx_decode": (536729344 + 3894528 + 268741632 + 4389120) / 40,  # 4-term block-scaled, per distinct expert
    "ffn_mx": (891086080 + 6049792 + 472940544 + 79744768) / 64,       # all-FP4 prefill, per expert at ~128 tokens
    "ffn_tc": (934021120 + 93158656 + 482610432 + 114407680) / 64,     # f16 prefill, per expert at ~128 tokens
}


def _traffic(kind, units):
    b = NCU_TRAFFIC.get(kind)
    return None if b is None else float(b * units)


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


def prefill_targets(flops: float, algo_bytes: float, ms: float, mxfp4_peak_tflops: float, mxfp4_kind: str,
                    hbm_gbs: float) -> dict:
    """The prefill config against its own target, a fraction of the dense MXFP4
    tensor peak. The workload's irreducible bytes (each picked expert's weights
    once, x in and the per-pick outputs out) cap what any kernel can reach:
    flops / (bytes / HBM peak)."""
    achieved = flops / (ms * 1e-3) / 1e12
    cap = flops / (algo_bytes / (hbm_gbs * 1e9)) / 1e12
    return {"achieved_tflops": achieved, "mxfp4_peak_tflops": mxfp4_peak_tflops, "mxfp4_peak_kind": mxfp4_kind,
            "frac_of_mxfp4_peak": achieved / mxfp4_peak_tflops,
            "hbm_bound_cap_tflops": cap, "frac_of_hbm_bound_cap": achieved / cap,
            "cap_frac_of_mxfp4_peak": cap / mxfp4_peak_tflops,
            "flop_per_byte": flops / algo_bytes}


def measure_mxfp4_peak(dev, iters: int = 4096, reps: int = 5):
    """Dense block-scaled FP4 rate of this GPU from the library's probe (one CTA per
    SM issuing kind::mxf4 MMAs on shared-memory operands): best of `reps` launches,
    TFLOP/s."""
    import torch

    import moe_decode_host_gb300 as m

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    st = torch.cuda.current_stream()
    m.mxf4_peak_probe(64, status, 0, st)  # warm-up
    best = 0.0
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        m.mxf4_peak_probe(iters, status, 0, st)
        e1.record(st)
        e1.synchronize()
        flops = sms * iters * 2.0 * 128 * 256 * 64
        best = max(best, flops / (e0.elapsed_time(e1) * 1e-3) / 1e12)
    assert int(status.item()) == 0
    return best


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


def skew_share(counts, ranking, frac_experts: float = 0.73) -> float:
    """Share of the picks that land on the `frac_experts` most popular experts of
    the routing generator (the skew statistic the pages quote: 98.7% of picks on 73%
    of experts), pooled over layers.  The popularity order is the generator's own
    (the Zipf permutation; expert order for uniform routing, where every expert is
    equally popular), not the order observed in the sample, so a short sample of
    uniform routing reads about 0.73.
    counts: int [steps, layers, E] picks per expert; ranking: int [layers, E], most
    popular expert first."""
    per_layer = np.asarray(counts, dtype=np.int64).sum(axis=0)  # [layers, E]
    ranking = np.asarray(ranking, dtype=np.int64)
    n_top = int(round(frac_experts * per_layer.shape[1]))
    top = sum(int(per_layer[li, ranking[li, :n_top]].sum()) for li in range(per_layer.shape[0]))
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
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c1", choices=["c1", "c2", "c3", "c4", "v1"])
    ap.add_argument("--batch", type=int, default=None, help="tokens per step (c2/c3: 8 or 32)")
    ap.add_argument("--skew", type=float, default=None, help="Zipf exponent for skewed routing")
    ap.add_argument("--layers", type=int, default=None, help="layers for c3")
    ap.add_argument("--pool", type=int, default=64, help="distinct steps of routing (at least)")
    ap.add_argument("--residency", dest="no_residency", action="store_false", default=None,
                    help="run the residency manager (default: only where the workload specifies it, the "
                         "20-layer stack)")
    ap.add_argument("--no-residency", dest="no_residency", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-per-batch", action="store_true",
                    help="skip the decode batches of 8 and 32 tokens that the default line carries")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle time of each CPU baseline leg")
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
    ap.add_argument("--residency-sync", action="store_true",
                    help="synchronous residency (plan and move at the closing call, draining the stream) "
                         "instead of the default deferred mode")
    ap.add_argument("--n-hot", type=int, default=None, help="HBM-resident experts per layer (rest cold)")
    ap.add_argument("--prefill", default=None, choices=["f16", "fp4"],
                    help="arithmetic of calls above 64 tokens: exact-weight f16 tensor cores, or block-scaled "
                         "FP4 with x and h in MXFP4 (default for the 8192-token config)")
    ap.add_argument("--decode-kind", type=int, default=0, choices=[0, 1, 2],
                    help="arithmetic of calls of at most 64 tokens: 1 the dequant-GEMV kernel, 2 block-scaled "
                         "tensor cores with 4-term MXFP4 activations, 0 (default) the library's choice (2)")
    ap.add_argument("--zero-copy", action="store_true",
                    help="the FFN reads picked cold experts in place from host memory (no slot copy)")
    return ap.parse_args()


def workload(args, config=None, batch=None):
    import synth

    name = config or args.config
    c = dict(synth.CONFIGS[name])
    no_res = args.no_residency
    if no_res is None:
        # residency only where the workload asks for it (the stacked-layer config)
        no_res = "swap_every" not in c
    c["no_res"] = no_res
    if config is None:
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
    if batch is not None:
        c["T"] = batch
    c["name"] = name
    # host copies of every expert: default for one layer (7.7 GB pinned); a 20-layer
    # stack would need 154 GB of pinned host memory, so it keeps the in-place exchange
    c["mirror"] = args.mirror if args.mirror is not None else (
        c.get("layers", 1) == 1 and c["n_cold"] > 0 and not no_res)
    c["zero_copy"] = bool(args.zero_copy)
    c["prefill"] = args.prefill or ("fp4" if c["T"] > 64 else "f16")
    c["decode_kind"] = args.decode_kind
    if args.n_hot is not None and args.experts is None:
        c["n_hot"] = min(args.n_hot, c["E"])
        c["n_cold"] = c["E"] - c["n_hot"]
    c["hysteresis"], c["swap_every_steps"], c["max_swaps"] = args.hysteresis, args.swap_every, args.max_swaps
    c["residency_sync"] = bool(args.residency_sync)
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


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


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


# ------------------------------------------------------------------ CPU oracle timing

ORACLE_TOKENS_PER_CALL = 8  # one oracle token of the 384-expert layer takes about two seconds
ORACLE_BLOB_POOL = 16       # distinct expert blobs the timed oracle calls read
_BLOB_POOLS: dict = {}


def _blob_pool(H, I, n):
    """n seeded expert blobs of shape (H, I), drawn once per process."""
    import synth

    key = (H, I, n)
    if key not in _BLOB_POOLS:
        b = synth.gen_blobs(n, H, I, seed=synth.sub_seed("oracle-timing", "blobs", H, I))
        _BLOB_POOLS[key] = [b[i].numpy() for i in range(n)]
    return _BLOB_POOLS[key]


def _oracle_jobs(c, seed_tag, n_jobs):
    """Inputs of n_jobs oracle calls: each the first ORACLE_TOKENS_PER_CALL tokens of
    a seeded step of the workload (logits, x bits)."""
    import torch

    import synth

    E, H = c["E"], c["H"]
    T_step = max(1, c["T"])
    T = min(T_step, ORACLE_TOKENS_PER_CALL)
    jobs = []
    for step in range(n_jobs):
        if c.get("routing") == "zipf":
            perm = synth.zipf_permutation(E, synth.sub_seed(c["name"], "perm"))
            logits = synth.gen_logits_zipf(T_step, E, c.get("s", 1.1), perm, seed=synth.sub_seed(seed_tag, step))
        elif c.get("routing") == "verify":
            logits = synth.gen_logits_verify(T_step, E, seed=synth.sub_seed(seed_tag, step))
        else:
            logits = synth.gen_logits_uniform(T_step, E, seed=synth.sub_seed(seed_tag, step))
        x = synth.gen_x(T_step, H, seed=synth.sub_seed(seed_tag, "x", step))
        jobs.append((np.ascontiguousarray(logits[:T]),
                     np.ascontiguousarray(x[:T].view(torch.int16).numpy().view(np.uint16))))
    return jobs, T, T_step


def oracle_tokens_per_s(c, seconds: float, seed_tag="cpu", threads: int = 1):
    """Times the CPU oracle on a bounded sample of the workload: whole tokens of the
    layer (route + every pick's expert FFN + combine), on `threads` host threads
    (the oracle's C calls run without the interpreter lock, each call on its own
    tokens).  The oracle runs every pick on its own token, so its time per token
    does not depend on the batch: each call takes the first ORACLE_TOKENS_PER_CALL
    tokens of a seeded step of the workload (routing is per token, so they route as
    they do in the whole step).  Expert e reads the bytes of blob e mod
    ORACLE_BLOB_POOL of a seeded pool (drawn outside the timed region; the oracle's
    time does not depend on the byte values).  Calls continue until `seconds` of
    wall time have passed (at least one per thread).  Returns (tokens/s, tokens,
    seconds, sample text)."""
    import concurrent.futures as cf

    import oracle
    import synth

    H, I, E, k = c["H"], c["I"], c["E"], c["k"]
    oracle.build()
    pool = _blob_pool(H, I, min(ORACLE_BLOB_POOL, E))
    blobs = [pool[e % len(pool)] for e in range(E)]
    batch = max(2, threads) * 2
    jobs, T, T_step = _oracle_jobs(c, seed_tag, batch)

    def call(j):
        logits, bits = jobs[j % len(jobs)]
        rc, _, _, _ = oracle.layer(logits, bits, k, 0, H, I, blobs)
        assert rc == 0
        return logits.shape[0]

    tok = 0
    calls = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max(1, threads)) as ex:
        while True:
            done = list(ex.map(call, range(calls, calls + max(1, threads))))
            tok += sum(done)
            calls += len(done)
            if time.perf_counter() - t0 >= seconds:
                break
    secs = time.perf_counter() - t0
    who = "single-threaded" if threads == 1 else f"{threads} host threads, one call each at a time"
    sample = (f"{tok} token(s) of the {c['name']} layer (the first {T} of a {T_step}-token step, {calls} "
              f"call(s)): route, {k} expert FFNs per token, combine; C oracle, fp64, {who}; expert bytes from "
              f"a pool of {len(pool)} seeded blobs")
    return tok / secs, tok, secs, sample


def cpu_baseline(c, seconds: float, seed_tag="cpu") -> dict:
    """The oracle on every host core this process may use (the reported value) and
    on one core, each for about `seconds` of wall time."""
    cores = host_cores()
    v_all, tok_all, s_all, sample_all = oracle_tokens_per_s(c, seconds, seed_tag=seed_tag + "-all", threads=cores)
    v_one, tok_one, s_one, sample_one = oracle_tokens_per_s(c, seconds, seed_tag=seed_tag + "-one", threads=1)
    return {"value": v_all, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample_all,
            "single_thread": {"value": v_one, "unit": "tokens/s", "cores": 1, "sample": sample_one}}


def run_reference(args, budget_s: float = 120.0):
    """The CPU oracle as the reference arm, on this arm's workload and metric: each
    step is one batch of oracle calls on every host core this process may use (one
    call per core), each call on the first tokens of a seeded step of the workload;
    the number of timed steps is capped so the run ends within a few minutes."""
    rank, world, _ = _rank_env()
    if rank != 0:
        return
    c = workload(args)
    cores = host_cores()
    if args.warmup > 0:
        oracle_tokens_per_s(c, 0.0, seed_tag="ref-warm", threads=cores)
    t_steps = []
    tok_total = 0
    sample = ""
    for s in range(max(1, args.steps)):
        v, tok, secs, sample = oracle_tokens_per_s(c, 0.0, seed_tag=f"ref{s}", threads=cores)
        t_steps.append(secs)
        tok_total += tok
        if sum(t_steps) + secs > budget_s:
            break
    total = sum(t_steps)
    value = tok_total / total
    n = len(t_steps)
    sample = (f"{n} step(s) of {cores} oracle call(s) on {cores} host threads, each call the first "
              f"{min(max(1, c['T']), ORACLE_TOKENS_PER_CALL)} token(s) of a {c['T']}-token step of the "
              f"{c['name']} layer (of {args.steps} requested; capped at {budget_s:.0f} s of oracle time): route, "
              f"{c['k']} expert FFNs per token, combine; C oracle, fp64; expert bytes from a pool of "
              f"{ORACLE_BLOB_POOL} seeded blobs")
    line = {"impl": "reference", "metric": "MoE layer tokens/s (decode)", "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": n, "steps_requested": args.steps, "warmup": min(args.warmup, 1),
            "ms_per_step": 1000.0 * total / n, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config_json(c, args),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _routing_name(c):
    if c.get("routing") == "zipf":
        return "Zipf s=%.2f" % c.get("s", 1.1)
    if c.get("routing") == "verify":
        return "verify-window (6 tokens of one sequence, correlated)"
    return "uniform"


def _config_json(c, args, pool_steps=None):
    return {"workload": f"{c['name']}: MoE layer H={c['H']} I={c['I']} E={c['E']} ({c['n_hot']} HBM / "
                        f"{c['n_cold']} pinned host) top-{c['k']}, {c['T']} token(s)/step, {_routing_name(c)} routing"
                        + (f", {c['layers']} layers sharing one slot scratch" if c.get("layers", 1) > 1 else ""),
            "tokens_per_step": c["T"], "layers": c.get("layers", 1),
            "residency": "off" if c["no_res"] else (
                "every %d steps, hysteresis %g, <=%d swaps, %s, " % (
                    c["swap_every_steps"], c["hysteresis"], c["max_swaps"],
                    "synchronous" if c.get("residency_sync") else "deferred one step (no stream sync)") + (
                "host copy of every expert" if c.get("mirror") else "in-place HBM/host exchange")),
            "step_pool": pool_steps if pool_steps is not None else args.pool,
            "l2": "inputs larger than L2 (7.7 GB expert pool per layer), no flush",
            "cold_experts": ("read in place from pinned host memory by the FFN (zero copy)"
                             if c.get("zero_copy") and c["T"] <= 64 else "copied into the HBM slot scratch"),
            "decode_arithmetic": (None if c["T"] > 64 else decode_arithmetic(c)),
            "prefill_arithmetic": (None if c["T"] <= 64 else (
                "block-scaled FP4 tensor cores (tcgen05 kind::mxf4), x and h quantised to MXFP4"
                if c.get("prefill") == "fp4" else "f16 tensor cores (tcgen05 kind::f16), weights expanded exactly")),
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
        layer.set_prefill_kind(1 if c.get("prefill") == "fp4" else 0)
        layer.set_decode_kind(c.get("decode_kind", 0))
        layer.set_residency_defer(not c.get("residency_sync", False))
        layers.append(dict(layer=layer, hot=hot, cold=cold, perm=perm))
    return layers, scratch, slots


def popularity(c, layers):
    """Per layer, experts from most to least popular under the routing generator
    (expert order for uniform routing)."""
    E = c["E"]
    return np.stack([L["perm"] if (L["perm"] is not None and c.get("routing") == "zipf") else np.arange(E)
                     for L in layers])


def gen_pool(c, layers, P, PL, dev):
    """Inputs of PL distinct steps: entry i holds, per layer, the logits of step i and
    the activations of step i % P.  Routing never repeats within PL steps."""
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


def host_numa(dev_index: int) -> dict:
    """The NUMA nodes this process sees and the GPU's node (sysfs): pinned host
    memory lands on the node of the allocating thread, so with one node there is no
    placement to choose."""
    out = {}
    try:
        nodes = sorted(int(d[4:]) for d in os.listdir("/sys/devices/system/node")
                       if d.startswith("node") and d[4:].isdigit())
        out["nodes"] = nodes
    except Exception:
        out["nodes"] = None
    try:
        bus = subprocess.run(["nvidia-smi", "-i", str(dev_index), "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip().lower()
        path = f"/sys/bus/pci/devices/{bus[-12:]}/numa_node"
        out["gpu_node"] = int(open(path).read().strip())
    except Exception:
        out["gpu_node"] = None
    return out


def measure_link_peak(dev):
    """Host-link read peak: max of a pinned H2D cudaMemcpyAsync and the zero-copy
    16-byte-load probe kernel (the same loop as cold_gather), 1 GiB each."""
    import torch

    import moe_decode_host_gb300 as m

    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
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


def ffn_terms(c):
    """Activation terms of the library's block-scaled FFN for this workload's calls
    (0: the dequant-GEMV / f16 tensor-core kernels), by the library's rule."""
    T = c["T"]
    if T > 64:
        return 1 if c.get("prefill") == "fp4" else 0
    kind = c.get("decode_kind", 0)
    if kind == 1 or (c.get("zero_copy") and c.get("n_cold", 0) > 0):
        return 0
    return 4


def step_launches(c):
    """Kernels one layer-step launches (residency move kernels excluded)."""
    T, n_cold = c["T"], c["n_cold"]
    zc = bool(c.get("zero_copy")) and n_cold > 0 and T <= 64
    route = 1 if T <= 64 else 2                          # one-CTA route, or top-k + bucketing
    gather = 1 + (0 if (n_cold == 0 or zc) else 2)      # remap; gate/up planes, down planes
    classes = 2 if n_cold > 0 else 1                    # HBM-resident and cold experts
    if ffn_terms(c) > 0:
        ffn = 1 + 2 * classes                           # activation prep, gate/up and down per class
    else:
        per_phase = 1 + (T > 8) + (T > 16) + (T > 64)   # decode token ranges, tcgen05 kernel
        ffn = 1 + classes * (2 * per_phase + 1)         # activation prep, phases, h prescale per down phase
    return route + gather + ffn + 1                     # + combine


def decode_arithmetic(c):
    """What the FFN of a decode-sized call computes in, as the library picks it."""
    if ffn_terms(c) == 4:
        return "block-scaled FP4 tensor cores (tcgen05 kind::mxf4), activations as sums of 4 MXFP4 terms"
    return "dequant-GEMV (E2M1 -> f16 in registers, mma.sync)"


def measure(c, args, dev, dist, world, link_peak, link_detail, local, mx_peak=None):
    """Builds the workload's layers, runs W warm-up steps, times K steps on the
    device (events on the stream, max over ranks), then per-call breakdown steps and
    the end-to-end leg, all on distinct steps of routing.  Returns the measurement
    as a dict (the JSON line's fields) and frees the layers."""
    import torch

    import moe_decode_host_gb300 as m

    hbm_peak, peak_kind = _peaks()
    layers, scratch, slots = build_layers(c, dev)
    K, W = args.steps, args.warmup
    Kb = min(K, 64)
    Ke = 0 if args.no_e2e else K
    # every phase of the run reads its own steps of routing (up to 2048 distinct)
    P = min(max(args.pool, W + K + Kb + Ke), 2048)
    pool = gen_pool(c, layers, args.pool, P, dev)
    T, k, H, E = c["T"], c["k"], c["H"], c["E"]
    eb = m.expert_bytes(H, c["I"])
    NL = len(layers)
    bufs = [m.StepBuffers(L["layer"], T) for L in layers]
    for L in layers:
        L["layer"].set_copy_ctas(args.copy_ctas)
    counts_log = torch.zeros((K, NL, E), dtype=torch.int32, device=dev)
    ncold_log = torch.zeros((K, NL), dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()
    nev = 6

    def step(i, log=None, ev=None):
        swaps = 0
        launches = 0
        for li, L in enumerate(layers):
            lg, x, _ = pool[i % P][li]
            b = bufs[li]
            layer = L["layer"]
            counts = counts_log[log, li] if log is not None else b.counts
            ncold = ncold_log[log, li] if log is not None else b.n_cold_picked
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
            n = m.residency_update(layer, st) if not c["no_res"] else 0
            if ev is not None:
                ev[li][5].record(st)
            swaps += n
            launches += step_launches(c) + (1 if n > 0 else 0)
        return swaps, launches

    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    events = [[[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(NL)] for _ in range(Kb)]
    for L in layers:
        L["layer"].profile(K)  # events around each cold copy (copy stream) and each FFN call
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
        s, n = step(W + i, log=i)
        total_swaps += s
        launches += n
        if i + 1 in marks:
            marks[i + 1].record(st)
    # the timed work includes each layer's last residency move (deferred moves run on
    # the layers' copy streams)
    for L in layers:
        m.moe_gather_join(L["layer"], st)
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
        step(W + K + i, ev=events[i])
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
    act_bytes = T * H * 2 + T * k * H * 4  # x read (bf16), y written (fp32 per pick)
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
    copy_tot_ms = float(sum(float(np.sum(cm)) for cm in copy_ms))
    n_copies = int(sum(len(cm) for cm in copy_ms))
    gather_gbs = float(gather_bytes.sum() / (copy_tot_ms * 1e-3) / 1e9) if copy_tot_ms > 0 else 0.0
    lp = link_peak if link_peak else float("inf")
    tstar_nom = np.maximum(hot_bytes / (HBM_NOMINAL_GBS * 1e9), gather_bytes / (lp * 1e9))
    tstar_meas = np.maximum(hot_bytes / (hbm_peak * 1e9), gather_bytes / (lp * 1e9))
    step_ms = elapsed_ms / K
    value = job_rate(world, K, T, elapsed_ms)
    # the residency moves' own link reads (one expert per swap, host to HBM) on top of
    # the cold copies: the bound the policy's churn leaves
    tstar_res_ms = float(1e3 * tstar_meas.sum() / K) + (total_swaps * eb / (lp * 1e9) * 1e3 / K)
    # dominant kernel: the one with the most GPU time over the timed region, the cold
    # copy (on the copy stream) or the FFN call's kernels (wait for the copy excluded)
    tot = {n: float(np.sum(per[n])) for n in names}
    dom = "cold_gather" if copy_tot_ms > ffn_k_tot_ms else "moe_grouped_ffn"
    mean_distinct = float(distinct.mean())
    mean_cold = float(ncold_h.mean())
    if dom == "moe_grouped_ffn" and T > 64:
        fp4 = c.get("prefill") == "fp4"
        if fp4:
            tc_peak, tc_kind = mx_peak, "measured in this run (dense kind::mxf4 probe)"
            kern = "moe_grouped_ffn (tcgen05 kind::mxf4 block-scaled grouped GEMM, x and h in MXFP4)"
        else:
            tc_peak, tc_kind = _tensor_peak()
            kern = "moe_grouped_ffn (tcgen05 kind::f16 grouped GEMM for buckets > 64 tokens)"
        t_tensor = ffn_flops / (tc_peak * 1e12)
        t_hbm = float(ffn_bytes.sum()) / (hbm_peak * 1e9)
        roof = {"kernel": kern, "ms_mean": ffn_k_tot_ms / (K * NL), "flops_per_call": ffn_flops / (K * NL),
                "algorithmic_bytes_per_call": float(ffn_bytes.sum() / (K * NL)),
                "tensor_tflops": ffn_tflops, "tensor_peak_tflops": tc_peak, "tensor_peak_kind": tc_kind,
                "tensor_frac": ffn_tflops / tc_peak, "hbm_gbs": ffn_gbs, "hbm_frac": ffn_gbs / hbm_peak,
                "traffic": _traffic("ffn_mx" if fp4 else "ffn_tc", mean_distinct),
                "prefill_target": prefill_targets(ffn_flops, float(ffn_bytes.sum()), ffn_k_tot_ms, mx_peak,
                                                  "measured in this run (dense kind::mxf4 probe)", hbm_peak)}
        if t_hbm >= t_tensor:  # the call's bytes take longer than its flops at the kind's peak
            roof.update({"bound": "hbm", "achieved": ffn_gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": ffn_gbs / hbm_peak, "peak_kind": peak_kind})
        else:
            roof.update({"bound": "tensor", "achieved": ffn_tflops, "peak": tc_peak, "unit": "TFLOP/s",
                         "frac": ffn_tflops / tc_peak, "peak_kind": tc_kind})
    elif dom == "moe_grouped_ffn":
        arith = decode_arithmetic(c)
        roof = {"kernel": "moe_grouped_ffn (decode: %s)" % arith, "bound": "hbm", "achieved": ffn_gbs,
                "peak": hbm_peak, "unit": "GB/s", "frac": ffn_gbs / hbm_peak,
                "traffic": _traffic("ffn_decode" if arith.startswith("dequant") else "ffn_mx_decode", mean_distinct),
                "algorithmic_bytes_per_call": float(ffn_bytes.sum() / (K * NL)),
                "ms_mean": ffn_k_tot_ms / (K * NL), "peak_kind": peak_kind}
    else:
        roof = {"kernel": "cold_copy_kernel (cold_gather's zero-copy host reads)", "bound": "link",
                "achieved": gather_gbs, "launches": n_copies, "ms_mean": copy_tot_ms / max(1, n_copies),
                "peak": link_peak, "unit": "GB/s", "frac": gather_gbs / link_peak if link_peak else None,
                "traffic": _traffic("cold_copy", mean_cold),
                "traffic_note": "DRAM bytes only: the copy reads host memory over the C2C link and its slot "
                                "writes stay in L2 during the launch",
                "algorithmic_bytes_per_launch": float(gather_bytes.sum() / max(1, n_copies)),
                "peak_kind": "measured in this run (max of pinned cudaMemcpyAsync and zero-copy probe)"}
    res = {"value": value, "ms_per_step": step_ms, "roofline": roof,
           "kernels": {n: {"ms_mean": float(np.mean(per[n])), "share": tot[n] / max(1e-9, sum(tot.values()))}
                       for n in names},
           "kernels_note": "per-call CUDA events over %d further steps run after the timed region" % Kb,
           "step_roofline": {"tstar_ms_nominal_hbm": float(1e3 * tstar_nom.sum() / K),
                             "frac_nominal": float(1e3 * tstar_nom.sum() / K / step_ms),
                             "tstar_ms_measured_hbm": float(1e3 * tstar_meas.sum() / K),
                             "frac_measured": float(1e3 * tstar_meas.sum() / K / step_ms),
                             "tstar_ms_with_residency_moves": tstar_res_ms,
                             "frac_with_residency_moves": tstar_res_ms / step_ms,
                             "hbm_peak_gbs": hbm_peak, "link_peak_gbs": link_peak, "link_probe": link_detail},
           "ffn_hbm_gbs": ffn_gbs, "ffn_kernel_ms_mean": ffn_k_tot_ms / (K * NL), "gather_link_gbs": gather_gbs,
           "distinct_experts_per_layer_step": mean_distinct,
           "picks_on_top_73pct_experts": skew_share(counts_h, popularity(c, layers)),
           "picks_sampled": int(counts_h.sum()),
           "repetitions": repetitions,
           "cold_experts_per_layer_step": mean_cold, "swaps": int(total_swaps),
           "clocks": clk, "gpu_launches": int(launches),
           "device_status": [int(L["layer"].status()) for L in layers],
           "pool_steps": P}
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, c, layers, pool, bufs, dev, dist, world, first=W + K + Kb, K=Ke)
    for L in layers:
        L["layer"].close()
    if scratch is not None:
        scratch.close()
    del layers, scratch, slots, pool, bufs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_e2e(args, c, layers, pool, bufs, dev, dist, world, first, K):
    """Steps through the public API with host buffers, on routing steps the device-
    timed region did not use: every step copies its logits and x in from pinned
    host memory and the layer output back out, inside the timed region; timed with
    the host clock from the first call to the end of a final synchronize."""
    import torch

    import moe_decode_host_gb300 as m

    T, k, H, E = c["T"], c["k"], c["H"], c["E"]
    P = len(pool)
    NL = len(layers)
    ids = [(first + i) % P for i in range(K)]
    host_in = {p: [(torch.from_numpy(pool[p][li][2]).pin_memory(), pool[p][li][1].cpu().pin_memory())
                   for li in range(NL)] for p in sorted(set(ids))}
    d_lg = [torch.empty((T, E), dtype=torch.float32, device=dev) for _ in range(NL)]
    d_x = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(NL)]
    host_out = [torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True) for _ in range(NL)]
    st = torch.cuda.current_stream()

    def step(p):
        for li, L in enumerate(layers):
            lg_h, x_h = host_in[p][li]
            d_lg[li].copy_(lg_h, non_blocking=True)
            d_x[li].copy_(x_h, non_blocking=True)
            m.run_step(L["layer"], bufs[li], d_lg[li], d_x[li], st, residency=not c["no_res"])
            host_out[li].copy_(bufs[li].out[:T], non_blocking=True)

    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for p in ids:
        step(p)
    torch.cuda.synchronize()
    ms = max_over_ranks(dist, (time.perf_counter() - t0) * 1e3, dev)
    return {"value": job_rate(world, K, T, ms), "unit": "tokens/s",
            "h2d_bytes_per_step": NL * (T * E * 4 + T * H * 2), "d2h_bytes_per_step": NL * T * H * 2,
            "timing": "host clock around the steps, ending in a synchronize; routing steps disjoint from the "
                      "device-timed region's"}


PER_BATCH = ((8, "c2"), (32, "c2"))  # decode batches the default line also carries (Zipf s=1.1)


def run_ours(args):
    import torch

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
    if args.no_link_probe:
        link_peak, link_detail = None, {"skipped": True}
    else:
        link_peak, link_detail = measure_link_peak(dev)
        link_detail["numa"] = host_numa(local)
    mx_peak = measure_mxfp4_peak(dev) if c["T"] > 64 else None
    res = measure(c, args, dev, dist, world, link_peak, link_detail, local, mx_peak)
    pool_steps = res.pop("pool_steps")
    line = {"metric": "MoE layer tokens/s (decode)", "value": res.pop("value"), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": res.pop("ms_per_step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e2m1xe2m1->f32" if ffn_terms(c) > 0 else "e2m1xf16->f32",
            "data": "synthetic", "config": _config_json(c, args, pool_steps)}
    line.update(res)
    default_run = (args.config == "c1" and args.batch is None and args.experts is None and not args.zero_copy
                   and args.n_hot is None)
    if default_run and not args.no_per_batch:
        per_batch = {}
        for T, name in PER_BATCH:
            cb = workload(args, config=name, batch=T)
            r = measure(cb, args, dev, dist, world, link_peak, link_detail, local)
            ps = r.pop("pool_steps")
            per_batch[str(T)] = {"config": _config_json(cb, args, ps), "value": r["value"], "unit": "tokens/s",
                                 "ms_per_step": r["ms_per_step"], "roofline": r["roofline"],
                                 "step_roofline": {kk: v for kk, v in r["step_roofline"].items()
                                                   if kk != "link_probe"},
                                 "e2e": r.get("e2e"), "kernels": r["kernels"],
                                 "ffn_hbm_gbs": r["ffn_hbm_gbs"], "gather_link_gbs": r["gather_link_gbs"],
                                 "distinct_experts_per_layer_step": r["distinct_experts_per_layer_step"],
                                 "cold_experts_per_layer_step": r["cold_experts_per_layer_step"],
                                 "picks_on_top_73pct_experts": r["picks_on_top_73pct_experts"],
                                 "repetitions": r["repetitions"], "clocks": r["clocks"],
                                 "gpu_launches": r["gpu_launches"], "device_status": r["device_status"]}
        line["per_batch"] = per_batch
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(c, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
