"""GB300 (sm_103a) sparse-MoE expert path -- Python binding of ``include/moe.h``.

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libmoe_gb300.so``.  PyTorch provides device memory and streams.  bf16 tensors may be passed
as ``torch.bfloat16`` or as 16-bit integer tensors holding the bit patterns.

Calls have the names of the C ABI: ``moe_route``, ``moe_grouped_ffn`` (= ``moe_ffn_gate_up``
then ``moe_ffn_down``), ``moe_combine``, ``moe_forward``, ``moe_pack_weights``,
``moe_read_status``.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import (MOE_ERR_CUDA, MOE_ERR_DEVICE_STATUS, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_INVALID_ARG,
                   MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_OK, MOE_STATUS_BAD_EXPERT, MOE_STATUS_TIMEOUT)

__all__ = ["MoEError", "shape", "options", "Routing", "workspace", "moe_workspace_bytes", "moe_packed_bytes",
           "moe_pack_weights", "moe_route", "moe_grouped_ffn", "moe_ffn_gate_up", "moe_ffn_down", "moe_combine",
           "moe_forward", "moe_read_status", "moe_check_shape", "moe_launch_count", "moe_forward_decode_static",
           "lib"]


class MoEError(RuntimeError):
    def __init__(self, what: str, rc: int):
        super().__init__(f"{what}: {lib().moe_error_string(rc).decode()} ({rc})")
        self.rc = rc


def lib():
    return _lib.load()


def _check(rc: int, what: str) -> None:
    if rc != MOE_OK:
        raise MoEError(what, rc)


def shape(T: int, d: int, E: int = 256, k: int = 8, I: int = 512, I_shared: Optional[int] = None,
          group: int = 64) -> _lib.moe_shape:
    return _lib.moe_shape(T, d, E, k, I, I if I_shared is None else I_shared, group)


DECODE_AUTO, DECODE_GEMV = 0, 1


def options(tile_rows: int = 32, decode_max_tokens: int = 1, decode_path: int = DECODE_AUTO,
            deterministic: int = 0, host_routing: int = 0, unfused_dequant: int = 0,
            gemm_rows: int = 0) -> _lib.moe_options:
    """decode_path: DECODE_AUTO (one fused launch per token when it fits) or DECODE_GEMV.
    deterministic: 1 = prefill sums each token's rows in a fixed order at every size.
    host_routing: 1 = ablation of GPU-resident routing: the scan and block map run on the
    host after a device-to-host copy of the counts (synchronises the stream; same results).
    unfused_dequant: 1 = ablation of on-chip dequantisation: each FFN call first writes the
    projection's weights as bf16 into the (larger) workspace, then streams them (same results).
    gemm_rows: 16, 32, 64 or 128 = largest token block of the grouped GEMMs (0: default 128)."""
    return _lib.moe_options(tile_rows, decode_max_tokens, decode_path, deterministic, host_routing, unfused_dequant,
                            gemm_rows)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _o(opts):
    return ctypes.byref(opts) if opts is not None else None


def moe_check_shape(shp) -> int:
    return lib().moe_check_shape(ctypes.byref(shp))


def moe_workspace_bytes(shp, opts=None) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(shp), _o(opts)))


def moe_packed_bytes(shp, num_experts: int, intermediate: int) -> int:
    return int(lib().moe_packed_bytes(ctypes.byref(shp), num_experts, intermediate))


def moe_launch_count() -> int:
    return int(lib().moe_launch_count())


def workspace(shp, opts=None, device="cuda") -> torch.Tensor:
    """A zero-filled workspace (the library needs it zeroed once, before first use)."""
    n = moe_workspace_bytes(shp, opts)
    if n == 0:
        raise MoEError("moe_workspace_bytes", moe_check_shape(shp) or MOE_ERR_INVALID_ARG)
    return torch.zeros(n, dtype=torch.uint8, device=device)


class Routing:
    """Caller-owned device buffers of the routing results (see moe_routing in moe.h)."""

    def __init__(self, T: int, k: int = 8, E: int = 256, tile_rows: int = 32, device="cuda"):
        i32 = dict(dtype=torch.int32, device=device)
        self.topk_idx = torch.empty(max(T, 1), k, **i32)
        self.topk_w = torch.empty(max(T, 1), k, dtype=torch.float32, device=device)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.perm = torch.empty(max(k * T, 1), **i32)
        self.pos = torch.empty(max(T, 1), k, **i32)
        mt = int(lib().moe_max_tiles(T, k, E, tile_rows))
        self.tiles = torch.empty(mt, 3, **i32)
        self.num_tiles = torch.zeros(1, **i32)
        self._s = _lib.moe_routing(*(t.data_ptr() for t in (self.topk_idx, self.topk_w, self.counts, self.offsets,
                                                              self.perm, self.pos, self.tiles, self.num_tiles)))

    def ref(self):
        return ctypes.byref(self._s)


def _q4(m: Sequence[torch.Tensor]) -> _lib.moe_q4:
    codes, scales, biases = m
    return _lib.moe_q4(codes.data_ptr(), scales.data_ptr(), biases.data_ptr())


def moe_pack_weights(shp, gate, up, down, intermediate: int, out: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """Relayout one expert stack (each of gate/up/down = (codes, scales, biases) device tensors,
    expert outermost) into the packed 4-bit form; returns the packed uint8 tensor."""
    E = gate[0].shape[0]
    n = moe_packed_bytes(shp, E, intermediate)
    if n == 0:
        raise MoEError("moe_packed_bytes", MOE_ERR_UNSUPPORTED)
    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=gate[0].device)
    w = _lib.moe_expert_weights(_q4(gate), _q4(up), _q4(down), E)
    _check(lib().moe_pack_weights(ctypes.byref(shp), ctypes.byref(w), intermediate, _p(out), out.numel(),
                                  _s(stream)), "moe_pack_weights")
    return out


def moe_route(shp, x, w_router, logit_bias, routing: Routing, ws, opts=None, stream=None) -> None:
    _check(lib().moe_route(ctypes.byref(shp), _p(x), _p(w_router), _p(logit_bias), routing.ref(), _p(ws),
                           ws.numel(), _o(opts), _s(stream)), "moe_route")


def moe_router_logits(shp, x, w_router, logit_bias, out, stream=None) -> None:
    """Every exact router logit (fp32 [T][E] into out), as moe_route defines them."""
    _check(lib().moe_router_logits(ctypes.byref(shp), _p(x), _p(w_router), _p(logit_bias), _p(out), _s(stream)),
           "moe_router_logits")


def moe_ffn_gate_up(shp, x, routing: Routing, packed_routed, packed_shared, ws, opts=None, stream=None) -> None:
    _check(lib().moe_ffn_gate_up(ctypes.byref(shp), _p(x), routing.ref(), _p(packed_routed), _p(packed_shared),
                                 _p(ws), ws.numel(), _o(opts), _s(stream)), "moe_ffn_gate_up")


def moe_ffn_down(shp, routing: Routing, packed_routed, packed_shared, ws, opts=None, stream=None) -> None:
    _check(lib().moe_ffn_down(ctypes.byref(shp), routing.ref(), _p(packed_routed), _p(packed_shared), _p(ws),
                              ws.numel(), _o(opts), _s(stream)), "moe_ffn_down")


def moe_grouped_ffn(shp, x, routing: Routing, packed_routed, packed_shared, ws, opts=None, stream=None) -> None:
    _check(lib().moe_grouped_ffn(ctypes.byref(shp), _p(x), routing.ref(), _p(packed_routed), _p(packed_shared),
                                 _p(ws), ws.numel(), _o(opts), _s(stream)), "moe_grouped_ffn")


def moe_combine(shp, routing: Routing, ws, y, opts=None, stream=None) -> None:
    _check(lib().moe_combine(ctypes.byref(shp), routing.ref(), _p(ws), ws.numel(), _p(y), _o(opts), _s(stream)),
           "moe_combine")


def moe_forward(shp, x, w_router, logit_bias, packed_routed, packed_shared, routing: Routing, ws, y, opts=None,
                stream=None) -> None:
    _check(lib().moe_forward(ctypes.byref(shp), _p(x), _p(w_router), _p(logit_bias), _p(packed_routed),
                             _p(packed_shared), routing.ref(), _p(ws), ws.numel(), _p(y), _o(opts), _s(stream)),
           "moe_forward")


def moe_forward_decode_static(shp, x, w_router, logit_bias, packed_routed, packed_shared, routing: Routing, y,
                              stream=None) -> None:
    """One-token forward with no workspace: the scratch is a fixed device array inside the
    library (see moe_forward_decode_static in include/moe.h).  For callers that cannot
    allocate scratch memory; calls that overlap on the GPU race on the shared array."""
    _check(lib().moe_forward_decode_static(ctypes.byref(shp), _p(x), _p(w_router), _p(logit_bias),
                                           _p(packed_routed), _p(packed_shared), routing.ref(), _p(y), _s(stream)),
           "moe_forward_decode_static")


def moe_read_status(ws, stream=None):
    """Synchronise, read and clear the device status word: (return code, raw status bits)."""
    bits = ctypes.c_int(0)
    rc = lib().moe_read_status(_p(ws), _s(stream), ctypes.byref(bits))
    return rc, bits.value
