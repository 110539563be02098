"""The roofline numerators bench.py reports (CPU): algorithmic bytes and FLOPs of the gate/up
and down kernels, checked against closed forms and against the library's packed weight size
(4-bit codes plus a bf16 scale and bias per 64 weights)."""
import ctypes
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from quantized_grouped_gemm_gb300 import _lib  # noqa: E402
from quantized_grouped_gemm_gb300 import build as build_mod  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.load()


class _Shape:
    def __init__(self, T, d, I):
        self.T, self.d, self.I = T, d, I


def test_prefill_counts_closed_form():
    T, d, I = 512, 2048, 512
    counts = np.full(256, 16, dtype=np.int64)
    A = bench.algorithmic_counts(_Shape(T, d, I), counts)
    per_matrix = I * d // 2 + I * (d // 64) * 4   # codes + bf16 scale and bias per 64: 589,824 B
    assert per_matrix == 589824
    assert A["touched"] == 257                                       # every expert + the shared one
    rows = 9 * T                                                     # 8 routed rows per token + shared
    assert A["gu_bytes"] == 257 * 2 * per_matrix + rows * d * 2 + rows * 2 * I * 2 == 331481088
    assert A["gu_flops"] == 2.0 * rows * d * 2 * I == 19327352832.0
    assert A["dn_flops"] == A["gu_flops"] / 2
    assert A["weights_bytes"] == 257 * 3 * per_matrix


def test_untouched_experts_are_not_counted():
    counts = np.zeros(256, dtype=np.int64)
    counts[:10] = 5
    A = bench.algorithmic_counts(_Shape(64, 256, 128), counts)
    assert A["touched"] == 11


def test_weight_bytes_agree_with_the_packed_size(lib):
    """3 matrices per expert in bench's count = the library's packed bytes minus its header."""
    for d, I in ((2048, 512), (512, 128), (7168, 256)):
        s = _lib.moe_shape(64, d, 256, 8, I, I, 64)
        packed = lib.moe_packed_bytes(ctypes.byref(s), 1, I)
        counts = np.zeros(256, dtype=np.int64)
        A = bench.algorithmic_counts(_Shape(64, d, I), counts)      # touched = the shared expert only
        assert A["weights_bytes"] == packed - 256, (d, I)
