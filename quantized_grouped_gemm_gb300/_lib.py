"""ctypes declarations of the C ABI in ``include/moe.h`` (argument marshalling only).

Loading fails loudly when ``libmoe_gb300.so`` has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_DEVICE_STATUS = -4
MOE_ERR_DEVICE_TIMEOUT = -5
MOE_ERR_WORKSPACE = -6
MOE_STATUS_BAD_EXPERT = 0x1
MOE_STATUS_TIMEOUT = 0x2
MOE_STATIC_SCRATCH_BYTES = 131072

_P = ctypes.c_void_p


class moe_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("I", ctypes.c_int), ("I_shared", ctypes.c_int), ("group", ctypes.c_int)]


class moe_q4(ctypes.Structure):
    _fields_ = [("codes_dev", _P), ("scales_dev", _P), ("biases_dev", _P)]


class moe_expert_weights(ctypes.Structure):
    _fields_ = [("gate", moe_q4), ("up", moe_q4), ("down", moe_q4), ("num_experts", ctypes.c_int)]


class moe_routing(ctypes.Structure):
    _fields_ = [("topk_idx_dev", _P), ("topk_w_dev", _P), ("counts_dev", _P), ("offsets_dev", _P),
                ("perm_dev", _P), ("pos_dev", _P), ("tiles_dev", _P), ("num_tiles_dev", _P)]


class moe_options(ctypes.Structure):
    _fields_ = [("tile_rows", ctypes.c_int), ("decode_max_tokens", ctypes.c_int), ("decode_path", ctypes.c_int),
                ("deterministic", ctypes.c_int), ("host_routing", ctypes.c_int),
                ("unfused_dequant", ctypes.c_int), ("gemm_rows", ctypes.c_int), ("reserved", ctypes.c_int * 1)]


_SPS = ctypes.POINTER(moe_shape)
_SIG = {
    "moe_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_check_shape": (ctypes.c_int, [_SPS]),
    "moe_workspace_bytes": (ctypes.c_size_t, [_SPS, ctypes.POINTER(moe_options)]),
    "moe_max_tiles": (ctypes.c_size_t, [ctypes.c_int] * 4),
    "moe_packed_bytes": (ctypes.c_size_t, [_SPS, ctypes.c_int, ctypes.c_int]),
    "moe_pack_weights": (ctypes.c_int, [_SPS, ctypes.POINTER(moe_expert_weights), ctypes.c_int, _P,
                                        ctypes.c_size_t, _P]),
    "moe_route": (ctypes.c_int, [_SPS, _P, _P, _P, ctypes.POINTER(moe_routing), _P, ctypes.c_size_t,
                                 ctypes.POINTER(moe_options), _P]),
    "moe_router_logits": (ctypes.c_int, [_SPS, _P, _P, _P, _P, _P]),
    "moe_grouped_ffn": (ctypes.c_int, [_SPS, _P, ctypes.POINTER(moe_routing), _P, _P, _P, ctypes.c_size_t,
                                       ctypes.POINTER(moe_options), _P]),
    "moe_ffn_gate_up": (ctypes.c_int, [_SPS, _P, ctypes.POINTER(moe_routing), _P, _P, _P, ctypes.c_size_t,
                                       ctypes.POINTER(moe_options), _P]),
    "moe_ffn_down": (ctypes.c_int, [_SPS, ctypes.POINTER(moe_routing), _P, _P, _P, ctypes.c_size_t,
                                    ctypes.POINTER(moe_options), _P]),
    "moe_combine": (ctypes.c_int, [_SPS, ctypes.POINTER(moe_routing), _P, ctypes.c_size_t, _P,
                                   ctypes.POINTER(moe_options), _P]),
    "moe_forward": (ctypes.c_int, [_SPS, _P, _P, _P, _P, _P, ctypes.POINTER(moe_routing), _P, ctypes.c_size_t, _P,
                                   ctypes.POINTER(moe_options), _P]),
    "moe_read_status": (ctypes.c_int, [_P, _P, ctypes.POINTER(ctypes.c_int)]),
    "moe_launch_count": (ctypes.c_ulonglong, []),
    "moe_forward_decode_static": (ctypes.c_int, [_SPS, _P, _P, _P, _P, _P, ctypes.POINTER(moe_routing), _P, _P]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library; raises if it is missing (build it with build.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} (run quantized_grouped_gemm_gb300.build.build())")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIG.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIG)
