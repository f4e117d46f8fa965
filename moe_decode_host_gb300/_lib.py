"""ctypes binding of libmoehost.so: same names as the C ABI in include/moehost.h.

Argument marshalling only: tensors are turned into raw pointers, streams into
cudaStream_t handles, and non-zero status codes into MoeError.  Every step of the
layer runs in the library's CUDA kernels; there is no Python or CPU fallback, and
importing this module fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoehost.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python moe_decode_host_gb300/build.py, or __graft_entry__.build())")

lib = ctypes.CDLL(LIB_PATH)

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_CUDA = -2
MOE_ERR_NONFINITE = -3
MOE_ERR_BAD_EXPERT = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_NOMEM = -6
MOE_ERR_INJECTED = -7
MOE_ERR_SCRATCH_TOO_SMALL = -8
MOE_NOALLOC_SCRATCH_BYTES = 8 << 20  # size of moe_grouped_ffn_noalloc's static workspace (moehost.h)


class moe_params(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("k", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("n_hot", ctypes.c_int), ("n_cold", ctypes.c_int), ("renorm", ctypes.c_int),
                ("swap_every", ctypes.c_int), ("max_swaps", ctypes.c_int), ("hysteresis", ctypes.c_float),
                ("host_mirror", ctypes.c_int), ("zero_copy", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t

_SIGS = {
    "moe_expert_bytes": (_Z, [_I, _I]),
    "moe_scratch_create": (_I, [_I, _Z, _P, ctypes.POINTER(_P)]),
    "moe_scratch_destroy": (_I, [_P]),
    "moe_layer_create": (_I, [ctypes.POINTER(moe_params), _P, _P, _P, _P, ctypes.POINTER(_P)]),
    "moe_layer_destroy": (_I, [_P]),
    "moe_route": (_I, [_P, _P, _I, _P, _P, _P, _P, _P, _P]),
    "cold_gather": (_I, [_P, _P, _I, _P, _P, _P, _P]),
    "moe_gather_join": (_I, [_P, _P]),
    "moe_ffn_workspace_bytes": (_I, [_P, _I, ctypes.POINTER(_Z)]),
    "moe_grouped_ffn": (_I, [_P, _P, _I, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_combine": (_I, [_P, _P, _I, _I, _I, _P, _I, _P]),
    "moe_grouped_ffn_noalloc": (_I, [_P, _P, _I, _P, _P, _P, _P, _P, _P]),
    "residency_update": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "moe_layer_set_prefill_kind": (_I, [_P, _I]),
    "moe_mxf4_peak_probe": (_I, [_I, _I, _P, _P]),
    "moe_layer_set_decode_kind": (_I, [_P, _I]),
    "moe_layer_set_residency_defer": (_I, [_P, _I]),
    "moe_residency_plan": (_I, [_P, _P, _I, _I, _I, ctypes.c_float, _P, _P, _P]),
    "moe_quant_mxfp4": (_I, [_P, _I, _I, _P, _P, _P]),
    "moe_layer_get_loc": (_I, [_P, _P]),
    "moe_layer_get_counts": (_I, [_P, _P]),
    "moe_get_status": (_I, [_P, ctypes.POINTER(_I)]),
    "moe_clear_status": (_I, [_P]),
    "moe_get_diag": (_I, [_P, _P]),
    "moe_strerror": (ctypes.c_char_p, [_I]),
    "moe_layer_inject_fault": (_I, [_P, _I]),
    "moe_layer_set_copy_ctas": (_I, [_P, _I]),
    "moe_layer_profile": (_I, [_P, _I]),
    "moe_layer_profile_read": (_I, [_P, _P, _I, ctypes.POINTER(_I)]),
    "moe_layer_profile_read_ffn": (_I, [_P, _P, _I, ctypes.POINTER(_I)]),
    "moe_link_probe": (_I, [_P, _P, _Z, _I, _P]),
    "moe_debug_e2m1_pairs": (_I, [_P, _P]),
    "moe_debug_e2m1_round": (_I, [_P, _I, _P, _P]),
    "moe_debug_wait_timeout": (_I, [_P, _P, _P]),
}

for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {lib.moe_strerror(code).decode()} ({code})")


def check(code: int, where: str) -> int:
    if code != MOE_OK:
        raise MoeError(code, where)
    return code


def ptr(t) -> int:
    """Raw pointer of a tensor (torch or numpy) or an int; None -> NULL."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(t)}")


def stream_handle(stream) -> int:
    """cudaStream_t of a torch stream (None -> torch's current stream)."""
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream
