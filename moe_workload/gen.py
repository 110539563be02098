"""Seeded synthetic inputs for the sparse-MoE expert path.

This module only draws numbers; it holds none of the method's arithmetic.  Both the
CPU oracle (tests, CPU baseline) and the CUDA path (tests, bench) take their inputs
from here, so the two sides always see identical bytes.

Random bits come from a counter-based generator: SplitMix64 (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014) applied to
``key(seed, stream) + (index + 1) * golden_gamma``.  Every tensor has its own stream
id, so the bytes of one tensor never depend on which other tensors were drawn.

Distributions (shapes and parameters follow the workloads of the MoE layer):

* ``normal_bf16``: an Irwin-Hall sum of twelve 16-bit uniforms minus 6.  It has mean
  0 and variance 1 (to 2**-32), is bounded by |z| < 6 and is computed with exact
  integer arithmetic, so every platform gives the same bits.  It stands in for the
  N(mean, std) draws of the workloads.  The float64 value ``mean + std * z`` is rounded
  to float32 and then to bf16 (round to nearest even).
* ``uniform``: 24-bit uniforms ``u = (bits >> 40) / 2**24`` in [0, 1), mapped to [lo, hi).
* codes: uniform random bytes, i.e. two independent uniform 4-bit codes per byte in
  the checkpoint layout (code k of a row is the low nibble of byte k // 2 when k is
  even and the high nibble when k is odd).
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _mix_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (used for per-stream keys)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def _mix_arr_inplace(z: np.ndarray, tmp: np.ndarray) -> None:
    """SplitMix64 finaliser on a uint64 array, in place (wrapping arithmetic)."""
    for shift, mult in ((30, _M1), (27, _M2)):
        np.right_shift(z, np.uint64(shift), out=tmp)
        np.bitwise_xor(z, tmp, out=z)
        np.multiply(z, np.uint64(mult), out=z)
    np.right_shift(z, np.uint64(31), out=tmp)
    np.bitwise_xor(z, tmp, out=z)


def stream_key(seed: int, stream: int) -> int:
    return _mix_int(_mix_int(seed * GOLDEN_GAMMA + 0x1234567) ^ (stream * 0xD1B54A32D192ED03))


_CHUNK = 1 << 18


def stream_bits(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """``n`` uint64 words of stream ``stream`` starting at counter ``start``."""
    key = np.uint64(stream_key(seed, stream))
    out = np.empty(n, dtype=np.uint64)
    tmp = np.empty(min(n, _CHUNK), dtype=np.uint64)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        z = out[c0:c1]
        z[:] = np.arange(start + c0 + 1, start + c1 + 1, dtype=np.uint64)
        np.multiply(z, np.uint64(GOLDEN_GAMMA), out=z)
        np.add(z, key, out=z)
        _mix_arr_inplace(z, tmp[: c1 - c0])
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniform(seed: int, stream: int, n: int, lo: float, hi: float) -> np.ndarray:
    bits = stream_bits(seed, stream, n)
    u = (bits >> np.uint64(40)).astype(np.float64) * (1.0 / (1 << 24))
    return lo + (hi - lo) * u


def irwin_hall12(seed: int, stream: int, n: int) -> np.ndarray:
    """n approximately standard-normal float64 values (exact integer sums)."""
    bits = stream_bits(seed, stream, 3 * n).reshape(n, 3)
    acc = np.zeros(n, dtype=np.int64)
    for w in range(3):
        col = bits[:, w]
        for s in range(4):
            acc += ((col >> np.uint64(16 * s)) & np.uint64(0xFFFF)).astype(np.int64)
    # each field f gives (f + 0.5) / 65536 in (0, 1); twelve of them minus 6
    return (acc.astype(np.float64) + 6.0) / 65536.0 - 6.0


def normal_bf16(seed: int, stream: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    z = irwin_hall12(seed, stream, n)
    return f32_to_bf16_bits((mean + std * z).astype(np.float32)).reshape(shape)


def uniform_bf16(seed: int, stream: int, shape, lo: float, hi: float) -> np.ndarray:
    n = int(np.prod(shape))
    return f32_to_bf16_bits(uniform(seed, stream, n, lo, hi).astype(np.float32)).reshape(shape)


def random_bytes(seed: int, stream: int, shape) -> np.ndarray:
    n = int(np.prod(shape))
    words = (n + 7) // 8
    return stream_bits(seed, stream, words).view(np.uint8)[:n].reshape(shape)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of 0..n-1 driven by the stream (modulo bias < 2**-50)."""
    bits = stream_bits(seed, stream, n)
    p = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(bits[i] % np.uint64(i + 1))
        p[i], p[j] = p[j], p[i]
    return p
