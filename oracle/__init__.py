"""CPU oracle of the sparse-MoE expert path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this package.  The product path (``quantized_grouped_gemm_gb300``)
never imports it and shares no code with it.

This module is argument marshalling over ``moe_oracle.cpp`` (plain C++, fp64, the pinned
fp32 router order); all arithmetic lives there.  Parity of every function is pinned by
``tests/test_oracle_pins.py`` against closed forms, brute force and hand-derived values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle shared library (plain g++, no fast-math, fp contraction off)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared",
           "-fPIC", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            L.oracle_bf16_round.restype = ctypes.c_uint16
            L.oracle_bf16_round.argtypes = [ctypes.c_double]
            L.oracle_dequant_one.restype = ctypes.c_uint16
            L.oracle_dequant_one.argtypes = [ctypes.c_uint16, ctypes.c_uint16, ctypes.c_int]
            L.oracle_dequant_matrix.argtypes = [ctypes.c_int, ctypes.c_int, _P, _P, _P, _P]
            L.oracle_q4_bytes.restype = ctypes.c_double
            L.oracle_q4_bytes.argtypes = [ctypes.c_double, ctypes.c_double]
            L.oracle_router_logit.restype = ctypes.c_float
            L.oracle_router_logit.argtypes = [ctypes.c_int, _P, _P, _P]
            L.oracle_router_logits.argtypes = [ctypes.c_int] * 3 + [_P] * 4
            L.oracle_topk.argtypes = [ctypes.c_int] * 3 + [_P] * 3
            L.oracle_route_meta.restype = ctypes.c_int
            L.oracle_route_meta.argtypes = [ctypes.c_int] * 4 + [_P] * 6 + [ctypes.c_int]
            L.oracle_expert_ffn.argtypes = [ctypes.c_int, ctypes.c_int, _P, ctypes.c_int, _P, _P, _P]
            L.oracle_moe_tokens.argtypes = [ctypes.c_int] * 4 + [_P, _P, ctypes.c_int] + [_P] * 5
            L.oracle_num_threads.restype = ctypes.c_int
            L.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


class _Q4(ctypes.Structure):
    _fields_ = [("codes", _P), ("scales", _P), ("biases", _P)]


class _Experts(ctypes.Structure):
    _fields_ = [("gate", _Q4), ("up", _Q4), ("down", _Q4)]


def _experts_struct(w) -> _Experts:
    def q(m):
        return _Q4(m.codes.ctypes.data, m.scales.ctypes.data, m.biases.ctypes.data)
    return _Experts(q(w.gate), q(w.up), q(w.down))


# ---------------------------------------------------------------------------------------
def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def bf16_round(x: float) -> int:
    return int(lib().oracle_bf16_round(float(x)))


def dequant_one(scale_bits: int, bias_bits: int, q: int) -> int:
    return int(lib().oracle_dequant_one(scale_bits, bias_bits, q))


def dequant_matrix(codes: np.ndarray, scales: np.ndarray, biases: np.ndarray) -> np.ndarray:
    """[N, K/2] codes + [N, K/64] scales/biases -> [N, K] bf16 bits."""
    N, Kh = codes.shape
    K = 2 * Kh
    out = np.empty((N, K), dtype=np.uint16)
    lib().oracle_dequant_matrix(N, K, _ptr(np.ascontiguousarray(codes)), _ptr(np.ascontiguousarray(scales)),
                                _ptr(np.ascontiguousarray(biases)), _ptr(out))
    return out


def q4_bytes(N: float, K: float) -> float:
    return float(lib().oracle_q4_bytes(N, K))


def router_logits(x: np.ndarray, w_router: np.ndarray, logit_bias: Optional[np.ndarray] = None) -> np.ndarray:
    T, d = x.shape
    E = w_router.shape[0]
    out = np.empty((T, E), dtype=np.float32)
    lib().oracle_router_logits(T, d, E, _ptr(np.ascontiguousarray(x)), _ptr(np.ascontiguousarray(w_router)),
                               _ptr(None if logit_bias is None else np.ascontiguousarray(logit_bias, np.float32)),
                               _ptr(out))
    return out


def topk(logits: np.ndarray, k: int = 8):
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    lib().oracle_topk(T, E, k, _ptr(np.ascontiguousarray(logits, np.float32)), _ptr(idx), _ptr(w))
    return idx, w


def route_meta(topk_idx: np.ndarray, E: int = 256, tile_rows: int = 32):
    T, k = topk_idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    pos = np.empty(T * k, dtype=np.int32)
    max_tiles = (T * k + tile_rows - 1) // tile_rows + E
    tiles = np.zeros((max_tiles, 3), dtype=np.int32)
    nt = lib().oracle_route_meta(T, E, k, tile_rows, _ptr(np.ascontiguousarray(topk_idx, np.int32)),
                                 _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(pos), _ptr(tiles), max_tiles)
    return dict(counts=counts, offsets=offsets, perm=perm, pos=pos.reshape(T, k), tiles=tiles[:nt],
                num_tiles=nt)


def route(x, w_router, logit_bias=None, k: int = 8, tile_rows: int = 32):
    """Steps a1-a6 of the path: logits, top-k + weights, histogram/scan/scatter/block map."""
    logits = router_logits(x, w_router, logit_bias)
    idx, w = topk(logits, k)
    meta = route_meta(idx, w_router.shape[0], tile_rows)
    meta.update(logits=logits, topk_idx=idx, topk_w=w)
    return meta


def expert_ffn(weights, e: int, x_row: np.ndarray, return_h: bool = False):
    d = x_row.shape[0]
    I = weights.gate.codes.shape[1]
    y = np.empty(d, dtype=np.float64)
    h = np.empty(I, dtype=np.float64)
    W = _experts_struct(weights)
    lib().oracle_expert_ffn(d, I, ctypes.byref(W), e, _ptr(np.ascontiguousarray(x_row)), _ptr(y), _ptr(h))
    return (y, h) if return_h else y


def moe_tokens(x: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray, routed, shared, tokens=None) -> np.ndarray:
    """Output rows (fp64, [len(tokens), d]) of the MoE layer for the listed tokens."""
    T, d = x.shape
    k = topk_idx.shape[1]
    I = routed.gate.codes.shape[1]
    I_sh = shared.gate.codes.shape[1] if shared is not None else 0
    tok = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    out = np.empty((len(tok), d), dtype=np.float64)
    R = _experts_struct(routed)
    S = _experts_struct(shared) if shared is not None else None
    lib().oracle_moe_tokens(d, k, I, I_sh, ctypes.byref(R), ctypes.byref(S) if S is not None else None,
                            len(tok), _ptr(tok), _ptr(np.ascontiguousarray(x)),
                            _ptr(np.ascontiguousarray(topk_idx, np.int32)),
                            _ptr(np.ascontiguousarray(topk_w, np.float64)), _ptr(out))
    return out
