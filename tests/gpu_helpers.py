"""Set-up helpers for the GPU tests: layers built from the seeded generator,
device buffers, and readers that fetch an expert's current bytes wherever the
placement map says it lives (so the oracle sees exactly what the GPU used)."""
from __future__ import annotations

import numpy as np
import torch

import synth


class LayerFixture:
    def __init__(self, *, H, I, E, n_hot, n_cold, k, seed, loc=None, swap_every=0, max_swaps=8,
                 hysteresis=3.0, renorm=0, scratch=None, slots=None, gen_device="cuda", host_mirror=False,
                 zero_copy=False, residency_defer=True):
        import moe_decode_host_gb300 as m

        self.m = m
        self.H, self.I, self.E, self.n_hot, self.n_cold, self.k = H, I, E, n_hot, n_cold, k
        self.eb = m.expert_bytes(H, I)
        dev = torch.device("cuda")
        self.loc0 = np.arange(E, dtype=np.int32) if loc is None else np.asarray(loc, np.int32)
        self.host_mirror = host_mirror
        self.hot = torch.empty((max(1, n_hot), self.eb), dtype=torch.uint8, device=dev)
        if host_mirror:
            # a host copy of every expert, indexed by expert id
            self.cold = torch.empty((E, self.eb), dtype=torch.uint8, pin_memory=True)
            synth.fill_layer(self.hot, None, self.loc0, H, I, seed, device=gen_device, mirror=self.cold)
        else:
            self.cold = torch.empty((max(1, n_cold), self.eb), dtype=torch.uint8, pin_memory=True)
            synth.fill_layer(self.hot, self.cold, self.loc0, H, I, seed, device=gen_device)
        n_host = E if host_mirror else n_cold
        if scratch is None:
            self.slots = torch.empty((max(1, n_cold), self.eb), dtype=torch.uint8, device=dev)
            self.scratch = m.Scratch(n_cold, self.eb, self.slots) if n_cold > 0 else None
        else:
            self.slots, self.scratch = slots, scratch
        self.layer = m.Layer(E=E, k=k, H=H, I=I, n_hot=n_hot, n_cold=n_cold, scratch=self.scratch,
                             hot_ptrs=[self.hot[h] for h in range(n_hot)],
                             cold_ptrs=[self.cold[c] for c in range(n_host)], init_loc=self.loc0,
                             renorm=renorm, swap_every=swap_every, max_swaps=max_swaps, hysteresis=hysteresis,
                             host_mirror=host_mirror, zero_copy=zero_copy)
        if not residency_defer:
            self.layer.set_residency_defer(False)

    def expert_bytes_now(self, e: int, loc=None) -> np.ndarray:
        """Current bytes of expert e (from its HBM slot or its host blob)."""
        loc = self.layer.get_loc() if loc is None else loc
        p = int(loc[e])
        if p < self.n_hot:
            return self.hot[p].cpu().numpy()
        if self.host_mirror:
            return self.cold[e].numpy().copy()
        return self.cold[p - self.n_hot].numpy().copy()

    def all_blobs_now(self) -> list:
        loc = self.layer.get_loc()
        return [self.expert_bytes_now(e, loc) for e in range(self.E)]


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.cpu().view(torch.int16).numpy().view(np.uint16)


def rel_l2(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def oracle_pick_rows(blob_of, H, I, x_f64, picks, act4=False):
    """Oracle expert outputs for the picks {(t, j): expert}: one oracle call per
    expert with its tokens batched, the experts spread over the host's cores (the
    oracle's expert FFN keeps no shared state, and ctypes releases the interpreter
    lock during the call).  blob_of(e) returns expert e's bytes; x_f64 [T, H]."""
    import concurrent.futures as cf
    import os

    import oracle

    by_e = {}
    for tj, e in picks.items():
        by_e.setdefault(int(e), []).append(tj)

    def one(e):
        tj = by_e[e]
        return e, oracle.expert_ffn(blob_of(e), H, I, np.stack([x_f64[t] for t, _ in tj]), act4=act4)

    out = {}
    workers = max(1, len(os.sched_getaffinity(0)))
    with cf.ThreadPoolExecutor(workers) as ex:
        for e, yy in ex.map(one, sorted(by_e)):
            for tj, row in zip(by_e[e], yy):
                out[tj] = row
    return out


def fingerprints(blob_of, experts):
    """FNV-1a-64 of each listed expert's current bytes (oracle), over host threads."""
    import concurrent.futures as cf
    import os

    import oracle

    workers = max(1, len(os.sched_getaffinity(0)))
    with cf.ThreadPoolExecutor(workers) as ex:
        return dict(zip(experts, ex.map(lambda e: oracle.fnv1a64(blob_of(e)), experts)))
