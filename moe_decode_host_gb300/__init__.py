"""moe_decode_host_gb300: MoE decode layer with host-resident cold experts on GB300.

Thin Python binding of the C ABI in include/moehost.h (libmoehost.so).  The entry
points keep the C names -- moe_route, cold_gather, moe_grouped_ffn, moe_combine,
residency_update -- and only marshal arguments: torch (or raw) pointers in,
status codes out as MoeError.  PyTorch is used for device memory and streams.
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._lib import (LIB_PATH, MOE_ERR_BAD_EXPERT, MOE_ERR_CUDA, MOE_ERR_INJECTED, MOE_ERR_INVALID_ARG,
                   MOE_ERR_NOMEM, MOE_ERR_NONFINITE, MOE_ERR_SCRATCH_TOO_SMALL, MOE_ERR_TIMEOUT,
                   MOE_NOALLOC_SCRATCH_BYTES, MOE_OK, MoeError, check, lib, moe_params, ptr, stream_handle)

__all__ = ["LIB_PATH", "MoeError", "Scratch", "Layer", "StepBuffers", "expert_bytes", "moe_route", "cold_gather",
           "moe_grouped_ffn", "moe_combine", "residency_update", "moe_gather_join", "link_probe", "debug_e2m1_pairs", "debug_e2m1_round", "run_step",
           "MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_CUDA", "MOE_ERR_NONFINITE", "MOE_ERR_BAD_EXPERT",
           "MOE_ERR_TIMEOUT", "MOE_ERR_NOMEM", "MOE_ERR_INJECTED", "MOE_ERR_SCRATCH_TOO_SMALL",
           "moe_grouped_ffn_noalloc", "residency_plan", "quant_mxfp4", "mxf4_peak_probe"]


def expert_bytes(H: int, I: int) -> int:
    return int(lib.moe_expert_bytes(H, I))


class Scratch:
    """Shared cold-slot scratch over caller-owned device memory (slot c at c*expert_bytes)."""

    def __init__(self, n_slots: int, nbytes_per_expert: int, slot_dev):
        h = ctypes.c_void_p()
        check(lib.moe_scratch_create(n_slots, nbytes_per_expert, ptr(slot_dev), ctypes.byref(h)),
              "moe_scratch_create")
        self.handle = h
        self.memory = slot_dev

    def close(self):
        if self.handle:
            lib.moe_scratch_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Layer:
    """One MoE layer handle (moe_layer_create)."""

    def __init__(self, *, E, k, H, I, n_hot, n_cold, scratch, hot_ptrs, cold_ptrs, init_loc, renorm=0,
                 swap_every=16, max_swaps=8, hysteresis=3.0, host_mirror=False, zero_copy=False):
        """cold_ptrs: the n_cold cold slots' host blobs, or with host_mirror the host
        copies of all E experts indexed by expert id. zero_copy: the FFN reads picked
        cold experts in place from host memory (calls of at most 64 tokens)."""
        self.p = moe_params(E, k, H, I, n_hot, n_cold, renorm, swap_every, max_swaps, hysteresis,
                            1 if host_mirror else 0, 1 if zero_copy else 0)
        hot = (ctypes.c_void_p * max(1, n_hot))(*[ptr(x) for x in hot_ptrs])
        n_host = E if host_mirror else n_cold
        cold = (ctypes.c_void_p * max(1, n_host))(*[ptr(x) for x in cold_ptrs])
        loc = np.ascontiguousarray(init_loc, dtype=np.int32)
        h = ctypes.c_void_p()
        check(lib.moe_layer_create(ctypes.byref(self.p), scratch.handle if scratch else None,
                                   hot if n_hot else None, cold if n_host else None, loc.ctypes.data,
                                   ctypes.byref(h)), "moe_layer_create")
        self.handle = h
        self.scratch = scratch
        self.E, self.k, self.H, self.I = E, k, H, I
        self.n_hot, self.n_cold = n_hot, n_cold

    def close(self):
        if getattr(self, "handle", None):
            lib.moe_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def ffn_workspace_bytes(self, T: int) -> int:
        n = ctypes.c_size_t()
        check(lib.moe_ffn_workspace_bytes(self.handle, T, ctypes.byref(n)), "moe_ffn_workspace_bytes")
        return int(n.value)

    def get_loc(self) -> np.ndarray:
        out = np.zeros(self.E, np.int32)
        check(lib.moe_layer_get_loc(self.handle, out.ctypes.data), "moe_layer_get_loc")
        return out

    def get_counts(self) -> np.ndarray:
        out = np.zeros(self.E, np.int32)
        check(lib.moe_layer_get_counts(self.handle, out.ctypes.data), "moe_layer_get_counts")
        return out

    def status(self) -> int:
        s = ctypes.c_int()
        check(lib.moe_get_status(self.handle, ctypes.byref(s)), "moe_get_status")
        return int(s.value)

    def diag(self) -> np.ndarray:
        out = np.zeros(16, np.int32)
        check(lib.moe_get_diag(self.handle, out.ctypes.data), "moe_get_diag")
        return out

    def clear_status(self):
        check(lib.moe_clear_status(self.handle), "moe_clear_status")

    def set_prefill_kind(self, kind: int):
        """0: exact-weight f16 tensor-core path for calls of more than 64 tokens;
        1: all-FP4 block-scaled path (x and h quantised to MXFP4)."""
        check(lib.moe_layer_set_prefill_kind(self.handle, kind), "moe_layer_set_prefill_kind")

    def set_decode_kind(self, kind: int):
        """Arithmetic of calls of at most 64 tokens: 1 the dequant-GEMV kernel; 2
        block-scaled tensor cores with 4-term MXFP4 activations; 0 (default) the
        library's choice (kind 2)."""
        check(lib.moe_layer_set_decode_kind(self.handle, kind), "moe_layer_set_decode_kind")

    def set_residency_defer(self, defer: bool):
        """True (default): residency plans are made and applied one step after their
        window closes, with no stream synchronisation; False: at once, synchronously."""
        check(lib.moe_layer_set_residency_defer(self.handle, 1 if defer else 0), "moe_layer_set_residency_defer")

    def set_copy_ctas(self, ctas: int):
        check(lib.moe_layer_set_copy_ctas(self.handle, ctas), "moe_layer_set_copy_ctas")

    def profile(self, max_records: int):
        check(lib.moe_layer_profile(self.handle, max_records), "moe_layer_profile")

    def profile_read(self, max_records: int) -> np.ndarray:
        out = np.zeros(max(1, max_records), np.float32)
        n = ctypes.c_int()
        check(lib.moe_layer_profile_read(self.handle, out.ctypes.data, max_records, ctypes.byref(n)),
              "moe_layer_profile_read")
        return out[: n.value].copy()

    def profile_read_ffn(self, max_records: int) -> np.ndarray:
        out = np.zeros(max(1, max_records), np.float32)
        n = ctypes.c_int()
        check(lib.moe_layer_profile_read_ffn(self.handle, out.ctypes.data, max_records, ctypes.byref(n)),
              "moe_layer_profile_read_ffn")
        return out[: n.value].copy()

    def inject_fault(self, what: int):
        check(lib.moe_layer_inject_fault(self.handle, what), "moe_layer_inject_fault")


def moe_route(layer: Layer, logits, T, topk_ids, topk_w, counts, offsets, entries, stream=None):
    check(lib.moe_route(layer.handle, ptr(logits), T, ptr(topk_ids), ptr(topk_w), ptr(counts), ptr(offsets),
                        ptr(entries), stream_handle(stream)), "moe_route")


def cold_gather(layer: Layer, topk_ids, T, phys_ids, cold_list, n_cold_picked, stream=None):
    check(lib.cold_gather(layer.handle, ptr(topk_ids), T, ptr(phys_ids), ptr(cold_list), ptr(n_cold_picked),
                          stream_handle(stream)), "cold_gather")


def moe_gather_join(layer: Layer, stream=None):
    check(lib.moe_gather_join(layer.handle, stream_handle(stream)), "moe_gather_join")


def moe_grouped_ffn(layer: Layer, x, T, phys_ids, counts, offsets, entries, y, workspace, workspace_bytes=None,
                    stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    check(lib.moe_grouped_ffn(layer.handle, ptr(x), T, ptr(phys_ids), ptr(counts), ptr(offsets), ptr(entries),
                              ptr(y), ptr(workspace), workspace_bytes, stream_handle(stream)), "moe_grouped_ffn")


def moe_grouped_ffn_noalloc(layer: Layer, x, T, phys_ids, counts, offsets, entries, y, stream=None):
    """moe_grouped_ffn with the library's static workspace (no device allocation;
    for callers that cannot allocate)."""
    check(lib.moe_grouped_ffn_noalloc(layer.handle, ptr(x), T, ptr(phys_ids), ptr(counts), ptr(offsets),
                                      ptr(entries), ptr(y), stream_handle(stream)), "moe_grouped_ffn_noalloc")


def moe_combine(y, topk_w, T, k, H, out, out_fp32=False, stream=None):
    check(lib.moe_combine(ptr(y), ptr(topk_w), T, k, H, ptr(out), 1 if out_fp32 else 0, stream_handle(stream)),
          "moe_combine")


def residency_update(layer: Layer, stream=None) -> int:
    n = ctypes.c_int32()
    check(lib.residency_update(layer.handle, ctypes.byref(n), stream_handle(stream)), "residency_update")
    return int(n.value)


def residency_plan(counts, loc, n_hot: int, max_swaps: int, hysteresis: float):
    """The swaps one acting residency_update would make (host only, no GPU):
    returns (loc after the swaps, promoted experts, demoted experts)."""
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    loc = np.ascontiguousarray(loc, dtype=np.int32)
    E = int(counts.size)
    out = np.empty(E, np.int32)
    pro = np.empty(max(1, max_swaps), np.int32)
    dem = np.empty(max(1, max_swaps), np.int32)
    n = lib.moe_residency_plan(ptr(counts), ptr(loc), E, n_hot, max_swaps, float(hysteresis), ptr(out), ptr(pro),
                               ptr(dem))
    if n < 0:
        check(n, "moe_residency_plan")
    return out, pro[:n].copy(), dem[:n].copy()


def quant_mxfp4(x, rows: int, K: int, nib, scales, stream=None):
    """MXFP4 quantisation of bf16 rows x [rows, K] into nib [rows, K/2] and scales
    [rows, K/32] (device tensors), on the GPU."""
    check(lib.moe_quant_mxfp4(ptr(x), rows, K, ptr(nib), ptr(scales), stream_handle(stream)), "moe_quant_mxfp4")


def link_probe(src_host, dst_dev, nbytes, ctas=0, stream=None):
    check(lib.moe_link_probe(ptr(src_host), ptr(dst_dev), nbytes, ctas, stream_handle(stream)), "moe_link_probe")


def mxf4_peak_probe(iters, status_dev, ctas=0, stream=None):
    """Launches the dense block-scaled FP4 rate probe (time it on `stream`):
    ctas x iters MMAs of 2 * 128 * 256 * 64 flops each."""
    check(lib.moe_mxf4_peak_probe(iters, ctas, ptr(status_dev), stream_handle(stream)), "moe_mxf4_peak_probe")


def debug_e2m1_pairs(out_dev, stream=None):
    check(lib.moe_debug_e2m1_pairs(ptr(out_dev), stream_handle(stream)), "moe_debug_e2m1_pairs")


def debug_e2m1_round(v_dev, out_dev, stream=None):
    """Both E2M1 roundings of every value of fp32 tensor v_dev into uint32 out_dev [2n]."""
    check(lib.moe_debug_e2m1_round(ptr(v_dev), int(v_dev.numel()), ptr(out_dev), stream_handle(stream)),
          "moe_debug_e2m1_round")


class StepBuffers:
    """Device buffers of one decode step for T tokens (torch allocations)."""

    def __init__(self, layer: Layer, T: int, device="cuda", out_fp32=False):
        import torch
        k, E, H = layer.k, layer.E, layer.H
        n = max(1, T * k)
        i32 = dict(dtype=torch.int32, device=device)
        self.T = T
        self.topk_ids = torch.empty((max(1, T), k), **i32)
        self.topk_w = torch.empty((max(1, T), k), dtype=torch.float32, device=device)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.entries = torch.empty(n, **i32)
        self.phys_ids = torch.empty(n, **i32)
        self.cold_list = torch.empty(max(1, min(max(layer.n_cold, 1), n)), **i32)
        self.n_cold_picked = torch.zeros(1, **i32)
        self.y = torch.empty((n, H), dtype=torch.float32, device=device)
        ws = layer.ffn_workspace_bytes(T)
        self.workspace = torch.empty(max(256, ws), dtype=torch.uint8, device=device)
        self.out_fp32 = out_fp32
        self.out = torch.empty((max(1, T), H), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=device)


def run_step(layer: Layer, buf: StepBuffers, logits, x, stream=None, residency=True) -> int:
    """One pass of the layer: route, cold gather, grouped FFN, combine, then the
    residency step.  Returns the number of swaps made (0 on non-acting steps)."""
    T = buf.T
    moe_route(layer, logits, T, buf.topk_ids, buf.topk_w, buf.counts, buf.offsets, buf.entries, stream)
    cold_gather(layer, buf.topk_ids, T, buf.phys_ids, buf.cold_list, buf.n_cold_picked, stream)
    moe_grouped_ffn(layer, x, T, buf.phys_ids, buf.counts, buf.offsets, buf.entries, buf.y, buf.workspace,
                    stream=stream)
    moe_combine(buf.y, buf.topk_w, T, layer.k, layer.H, buf.out, buf.out_fp32, stream)
    return residency_update(layer, stream) if residency else 0
