"""CPU oracle for the MoE decode layer (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may
import this package.  It wraps ``moe_oracle.c`` (plain C, IEEE double, no code
shared with the CUDA path) through ctypes, plus numpy marshalling.  See the header
of ``moe_oracle.c`` for what each function restates and where it comes from.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERR_ARG = -1
ERR_NONFINITE = -3


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            Z = ctypes.c_size_t
            lib.or_e2m1.restype = D
            lib.or_e2m1.argtypes = [ctypes.c_uint]
            lib.or_e8m0.restype = D
            lib.or_e8m0.argtypes = [ctypes.c_uint]
            lib.or_nibble_at.restype = ctypes.c_uint
            lib.or_nibble_at.argtypes = [P, I]
            lib.or_decode_row.restype = None
            lib.or_decode_row.argtypes = [P, P, I, P]
            lib.or_route.restype = I
            lib.or_route.argtypes = [P, I, I, I, I, P, P, P, P, P]
            lib.or_remap.restype = I
            lib.or_remap.argtypes = [P, I, P, I, I, P, P]
            lib.or_expert_ffn.restype = None
            lib.or_expert_ffn.argtypes = [P, I, I, P, I, P]
            lib.or_expert_ffn_act4.restype = None
            lib.or_expert_ffn_act4.argtypes = [P, I, I, P, I, P]
            lib.or_quant_mxfp4.restype = None
            lib.or_quant_mxfp4.argtypes = [P, I, P, P]
            lib.or_combine.restype = None
            lib.or_combine.argtypes = [P, P, I, I, I, P]
            lib.or_layer.restype = I
            lib.or_layer.argtypes = [P, P, I, I, I, I, I, I, P, P, P, P]
            lib.or_layer_act4.restype = I
            lib.or_layer_act4.argtypes = [P, P, I, I, I, I, I, I, P, P, P, P]
            lib.or_residency.restype = I
            lib.or_residency.argtypes = [P, P, I, I, I, D, P, P]
            lib.or_fnv1a64.restype = ctypes.c_uint64
            lib.or_fnv1a64.argtypes = [P, Z]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def e2m1(code: int) -> float:
    return _load().or_e2m1(code)


def e8m0(e: int) -> float:
    return _load().or_e8m0(e)


def decode_row(nib_row: np.ndarray, scale_row: np.ndarray, K: int) -> np.ndarray:
    nib_row = _c(nib_row, np.uint8)
    scale_row = _c(scale_row, np.uint8)
    assert nib_row.size == K // 2 and scale_row.size == K // 32
    out = np.empty(K, dtype=np.float64)
    _load().or_decode_row(_p(nib_row), _p(scale_row), K, _p(out))
    return out


def blob_offsets(H: int, I: int) -> dict:
    w13n = 2 * I * (H // 2)
    w13s = 2 * I * (H // 32)
    w2n = H * (I // 2)
    return {"w13n": 0, "w13s": w13n, "w2n": w13n + w13s, "w2s": w13n + w13s + w2n,
            "total": w13n + w13s + w2n + H * (I // 32)}


def decode_matrix(blob: np.ndarray, H: int, I: int, which: str) -> np.ndarray:
    """Dense decode of 'w13' ([2I, H]) or 'w2' ([H, I]) from a blob (slow; small shapes)."""
    o = blob_offsets(H, I)
    blob = _c(blob, np.uint8)
    if which == "w13":
        R, K, n0, s0 = 2 * I, H, o["w13n"], o["w13s"]
    else:
        R, K, n0, s0 = H, I, o["w2n"], o["w2s"]
    out = np.empty((R, K), dtype=np.float64)
    for r in range(R):
        out[r] = decode_row(blob[n0 + r * (K // 2): n0 + (r + 1) * (K // 2)],
                            blob[s0 + r * (K // 32): s0 + (r + 1) * (K // 32)], K)
    return out


def route(logits: np.ndarray, k: int, renorm: int = 0):
    """Returns (rc, ids[T,k], w[T,k], counts[E], offsets[E+1], entries[T*k])."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float64)
    counts = np.zeros(E, dtype=np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    entries = np.zeros(max(1, T * k), dtype=np.int32)
    rc = _load().or_route(_p(logits), T, E, k, renorm, _p(ids), _p(w), _p(counts), _p(offsets), _p(entries))
    return rc, ids, w, counts, offsets, entries[: T * k]


def remap(ids: np.ndarray, loc: np.ndarray, n_hot: int, n_cold: int):
    """Returns (phys[same shape as ids], cold_list[n])."""
    ids = _c(ids, np.int32)
    loc = _c(loc, np.int32)
    phys = np.zeros_like(ids)
    cold = np.zeros(max(1, n_cold), dtype=np.int32)
    n = _load().or_remap(_p(ids), ids.size, _p(loc), n_hot, n_cold, _p(phys), _p(cold))
    return phys, cold[:n].copy()


def expert_ffn(blob: np.ndarray, H: int, I: int, x: np.ndarray, act4: bool = False) -> np.ndarray:
    """x: [n_tok, H] (any float dtype; converted to double).  Returns y [n_tok, H] double.
    act4: the all-FP4 mode (x and h quantised to MXFP4 per token, 32-element blocks)."""
    blob = _c(blob, np.uint8)
    x = _c(np.atleast_2d(x), np.float64)
    n = x.shape[0]
    y = np.zeros((n, H), dtype=np.float64)
    fn = _load().or_expert_ffn_act4 if act4 else _load().or_expert_ffn
    fn(_p(blob), H, I, _p(x), n, _p(y))
    return y


def quant_mxfp4(v: np.ndarray):
    """MXFP4 quantisation of a row of K values (K a multiple of 32) by the OCP rule:
    returns (nibble bytes [K/2] in the documented row layout, scale bytes [K/32])."""
    v = _c(np.ravel(v), np.float64)
    K = v.size
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    nib = np.zeros(K // 2, dtype=np.uint8)
    sc = np.zeros(K // 32, dtype=np.uint8)
    _load().or_quant_mxfp4(_p(v), K, _p(nib), _p(sc))
    return nib, sc


def combine(y: np.ndarray, w: np.ndarray, k: int) -> np.ndarray:
    y = _c(y, np.float64)
    w = _c(w, np.float64)
    T = w.shape[0]
    H = y.shape[1]
    out = np.zeros((T, H), dtype=np.float64)
    _load().or_combine(_p(y), _p(w), T, k, H, _p(out))
    return out


def layer(logits: np.ndarray, x_bf16_bits: np.ndarray, k: int, renorm: int, H: int, I: int, blobs: list,
          act4: bool = False):
    """Whole layer. blobs[e] = expert e's bytes (numpy uint8).  Returns (rc, ids, w, out).
    act4: the all-FP4 mode for every pick (see expert_ffn)."""
    logits = _c(logits, np.float32)
    x = _c(x_bf16_bits, np.uint16)
    T, E = logits.shape
    arrs = [_c(b, np.uint8) for b in blobs]
    ptrs = (ctypes.c_void_p * E)(*[a.ctypes.data for a in arrs])
    ids = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float64)
    out = np.zeros((T, H), dtype=np.float64)
    fn = _load().or_layer_act4 if act4 else _load().or_layer
    rc = fn(_p(logits), _p(x), T, E, k, renorm, H, I, ptrs, _p(ids), _p(w), _p(out))
    return rc, ids, w, out


def residency(counts: np.ndarray, loc: np.ndarray, n_hot: int, max_swaps: int, hysteresis: float):
    """Returns (new_loc, promoted[n], demoted[n])."""
    counts = _c(counts, np.int32)
    loc = _c(loc, np.int32).copy()
    E = counts.size
    pro = np.zeros(max(1, max_swaps), dtype=np.int32)
    dem = np.zeros(max(1, max_swaps), dtype=np.int32)
    n = _load().or_residency(_p(counts), _p(loc), E, n_hot, max_swaps, float(hysteresis), _p(pro), _p(dem))
    return loc, pro[:n].copy(), dem[:n].copy()


def fnv1a64(b: np.ndarray) -> int:
    b = _c(b, np.uint8)
    return int(_load().or_fnv1a64(_p(b), b.size))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) to float64, exactly."""
    u = (np.asarray(bits, dtype=np.uint32) << 16).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)
