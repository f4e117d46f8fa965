"""Seeded synthetic inputs for the MoE decode layer with host-resident cold experts.

This module is shared by the tests, the bench and the oracle checks, and it holds
none of the layer's arithmetic: it only draws bytes, activations and router logits
with the shapes and distributions of the workloads, and writes the starting
placement maps.  Both the CUDA path and the oracle consume exactly the bytes made
here.

Workloads (from the pages' setting: 384 experts, top-6, 255 hot / 129 cold per
layer, MXFP4 expert weights; "DeepSeek-V4.1-Flash on One GB300 Without the Second
GPU", section 1; "Milo and James try inference engineering", the model paragraph):

  c0  H=256,  I=512,  E=16  (12 hot, 4 cold),  k=2, T=4,      uniform routing
  c1  H=4096, I=3072, E=384 (255 hot, 129 cold), k=6, T=1,    uniform routing
  c2  as c1, T=8 and T=32, Zipf-skewed routing (s=1.1; s=1.5 also offered)
  c3  20 layers of c1's shape, one shared 129-slot scratch, skewed routing,
      mismatched starting hot sets, residency every 16 steps
  c4  as c1, T=8192, uniform routing, all 384 experts resident in HBM

Weight bytes: every nibble is an independent draw from the distribution of
E2M1 codes obtained by rounding N(0,1) to nearest (ties to even) and saturating
at +-6, quantised to 1/65536.  Because nibbles are i.i.d., the physical byte order
inside a row does not change the distribution, so bytes are drawn directly.
Scale bytes are 127 - U{0..8} (scales 2^-8 .. 2^0).
"""
from __future__ import annotations

import hashlib
import math

import numpy as np
import torch

CONFIGS = {
    "c0": dict(H=256, I=512, E=16, n_hot=12, n_cold=4, k=2, T=4, routing="uniform", layers=1),
    "c1": dict(H=4096, I=3072, E=384, n_hot=255, n_cold=129, k=6, T=1, routing="uniform", layers=1),
    "c2": dict(H=4096, I=3072, E=384, n_hot=255, n_cold=129, k=6, T=8, routing="zipf", s=1.1, layers=1),
    "c3": dict(H=4096, I=3072, E=384, n_hot=255, n_cold=129, k=6, T=1, routing="zipf", s=1.1, layers=20,
               swap_every=16),
    "c4": dict(H=4096, I=3072, E=384, n_hot=384, n_cold=0, k=6, T=8192, routing="uniform", layers=1),
    # verify window: the k + 1 = 6 tokens a speculative step checks, from one
    # sequence, with routing correlated so that the window picks about 3.7 times the
    # distinct experts of one token
    "v1": dict(H=4096, I=3072, E=384, n_hot=255, n_cold=129, k=6, T=6, routing="verify", layers=1),
}

VERIFY_WINDOW = 6
# Strength of the shared per-sequence logit component: with E = 384 and k = 6 a
# window of 6 tokens then picks 3.7x the distinct experts of one token (Monte Carlo;
# 0 gives 5.8x, independent tokens).
VERIFY_BETA = 1.42


def sub_seed(*parts) -> int:
    """Stable 63-bit seed derived from a config name, a layer and a tensor name."""
    h = hashlib.blake2b(repr(parts).encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def blob_sections(H: int, I: int) -> dict:
    """Byte offsets of the four planes of one expert blob (the library's format:
    w13 nibbles [2I, H/2], w13 scales [2I, H/32], w2 nibbles [H, I/2], w2 scales [H, I/32])."""
    w13n = 2 * I * (H // 2)
    w13s = 2 * I * (H // 32)
    w2n = H * (I // 2)
    w2s = H * (I // 32)
    offs = {"w13n": (0, w13n), "w13s": (w13n, w13s), "w2n": (w13n + w13s, w2n),
            "w2s": (w13n + w13s + w2n, w2s)}
    offs["total"] = w13n + w13s + w2n + w2s
    return offs


def _code_probabilities() -> np.ndarray:
    """P(code) for the 16 E2M1 codes when N(0,1) is rounded to the nearest code."""
    # magnitude codes 0..7 stand for 0, .5, 1, 1.5, 2, 3, 4, 6; decision points are
    # the midpoints between neighbours
    edges = [0.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, math.inf]

    def phi(z):
        return 1.0 if math.isinf(z) else 0.5 * (1.0 + math.erf(z / math.sqrt(2.0)))

    pos = [phi(edges[i + 1]) - phi(edges[i]) for i in range(8)]
    p = np.array(pos + pos, dtype=np.float64)  # codes 8..15 carry the negative sign
    return p / p.sum()


def nibble_table() -> np.ndarray:
    """65536-entry table mapping a uniform 16-bit draw to a nibble code.

    Every code gets at least one entry so that all 16 codes (including -0 and +-6)
    occur in large draws."""
    p = _code_probabilities()
    n = 1 << 16
    raw = p * n
    cnt = np.maximum(np.floor(raw).astype(np.int64), 1)
    # largest remainder to fill up to exactly 65536 entries
    while cnt.sum() < n:
        i = int(np.argmax(raw - cnt))
        cnt[i] += 1
    while cnt.sum() > n:
        i = int(np.argmax(cnt))
        cnt[i] -= 1
    return np.repeat(np.arange(16, dtype=np.uint8), cnt)


_TABLE_CACHE: dict = {}


def _table_on(device) -> torch.Tensor:
    key = str(device)
    if key not in _TABLE_CACHE:
        _TABLE_CACHE[key] = torch.from_numpy(nibble_table()).to(device)
    return _TABLE_CACHE[key]


def _random_nibble_bytes(n_bytes: int, gen: torch.Generator, device) -> torch.Tensor:
    table = _table_on(device)
    u = torch.randint(0, 1 << 16, (2 * n_bytes,), generator=gen, device=device, dtype=torch.int32)
    codes = table[u]
    return codes[0::2] | (codes[1::2] << 4)


def _random_scale_bytes(n_bytes: int, gen: torch.Generator, device) -> torch.Tensor:
    d = torch.randint(0, 9, (n_bytes,), generator=gen, device=device, dtype=torch.int32)
    return (127 - d).to(torch.uint8)


def gen_blobs(n: int, H: int, I: int, seed: int, device="cpu", out: torch.Tensor | None = None) -> torch.Tensor:
    """n expert blobs of the library's format as a uint8 tensor [n, blob_bytes]."""
    sec = blob_sections(H, I)
    if out is None:
        out = torch.empty((n, sec["total"]), dtype=torch.uint8, device=device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    for i in range(n):
        for name in ("w13n", "w13s", "w2n", "w2s"):
            off, size = sec[name]
            if name.endswith("n"):
                out[i, off:off + size] = _random_nibble_bytes(size, gen, device)
            else:
                out[i, off:off + size] = _random_scale_bytes(size, gen, device)
    return out


def fill_layer(hot: torch.Tensor, cold: torch.Tensor, loc: np.ndarray, H: int, I: int, seed: int,
               device="cpu", mirror: torch.Tensor | None = None) -> None:
    """Draws every expert's blob (expert ids in ascending order, one generator) and
    writes it where the placement map puts it: hot[loc[e]] when loc[e] < n_hot,
    else cold[loc[e] - n_hot] (cold may be None when a mirror is given).  With
    `mirror` ([E, blob_bytes]) every expert's blob is also written to mirror[e].
    hot/cold/mirror may live on any device (cold and mirror are usually pinned host
    memory)."""
    n_hot = hot.shape[0]
    sec = blob_sections(H, I)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    tmp = torch.empty(sec["total"], dtype=torch.uint8, device=device)
    for e in range(len(loc)):
        for name in ("w13n", "w13s", "w2n", "w2s"):
            off, size = sec[name]
            if name.endswith("n"):
                tmp[off:off + size] = _random_nibble_bytes(size, gen, device)
            else:
                tmp[off:off + size] = _random_scale_bytes(size, gen, device)
        p = int(loc[e])
        if p < n_hot:
            hot[p].copy_(tmp)
        elif cold is not None:
            cold[p - n_hot].copy_(tmp)
        if mirror is not None:
            mirror[e].copy_(tmp)


def gen_x(T: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    """Activations bf16(N(0,1)) of shape [T, H]."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    return torch.randn((T, H), generator=gen, dtype=torch.float32).to(torch.bfloat16).to(device)


def gen_logits_uniform(T: int, E: int, seed: int) -> np.ndarray:
    """Router logits N(0,1) in fp32, shape [T, E] (uniform routing)."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((T, E)).astype(np.float32)


def zipf_permutation(E: int, seed: int) -> np.ndarray:
    """Experts listed from most to least popular."""
    return np.random.default_rng(seed).permutation(E)


def gen_logits_zipf(T: int, E: int, s: float, perm: np.ndarray, seed: int) -> np.ndarray:
    """Skewed logits l_e = log p(rank(e)) + Gumbel(0,1), p(r) proportional to r^-s.

    The top-k of these logits is a draw without replacement from the Zipf law over
    the permuted experts, so the routed picks follow the skew."""
    rng = np.random.default_rng(seed)
    ranks = np.empty(E, dtype=np.int64)
    ranks[perm] = np.arange(1, E + 1)
    logp = -s * np.log(ranks.astype(np.float64))
    logp -= np.log(np.sum(np.exp(logp)))
    u = rng.random((T, E))
    u = np.clip(u, 1e-300, 1.0 - 1e-16)
    g = -np.log(-np.log(u))
    return (logp[None, :] + g).astype(np.float32)


def gen_logits_verify(T: int, E: int, seed: int, window: int = VERIFY_WINDOW,
                      beta: float = VERIFY_BETA) -> np.ndarray:
    """Logits of verify windows: tokens t of window w = t // window get
    N(0,1) + beta * b_w, with b_w ~ N(0,1) per expert shared by the window, so the
    tokens of one sequence tend to pick the same experts."""
    rng = np.random.default_rng(seed)
    n_win = (T + window - 1) // window
    b = rng.standard_normal((n_win, E))
    z = rng.standard_normal((T, E))
    return (z + beta * b[np.arange(T) // window]).astype(np.float32)


def loc_identity(E: int, n_hot: int) -> np.ndarray:
    """Starting map: experts 0..n_hot-1 hot in order, the rest in cold slots in order."""
    return np.arange(E, dtype=np.int32)


def loc_from_hot_set(E: int, n_hot: int, hot: np.ndarray) -> np.ndarray:
    """Starting map from a hot set: hot experts take HBM slots in ascending id order,
    the others take cold slots in ascending id order.  loc[e] < n_hot is an HBM slot,
    loc[e] = n_hot + c is cold slot c."""
    hot = np.sort(np.asarray(hot, dtype=np.int64))
    assert hot.size == n_hot
    is_hot = np.zeros(E, dtype=bool)
    is_hot[hot] = True
    cold = np.nonzero(~is_hot)[0]
    loc = np.empty(E, dtype=np.int32)
    loc[hot] = np.arange(n_hot, dtype=np.int32)
    loc[cold] = n_hot + np.arange(cold.size, dtype=np.int32)
    return loc


def hit_fraction(picks: np.ndarray, E: int, frac_experts: float = 0.73) -> float:
    """Share of picks that land on the most-picked `frac_experts` of the experts
    (the skew statistic the pages quote: 98.7% of picks on 73% of experts)."""
    cnt = np.bincount(np.asarray(picks).ravel(), minlength=E)
    top = np.sort(cnt)[::-1][: int(round(frac_experts * E))]
    return float(top.sum() / max(1, cnt.sum()))
