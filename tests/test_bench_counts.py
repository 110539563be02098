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
    # weights + the activation rows read once + h (bf16) written once
    assert A["gu_bytes"] == 257 * 2 * per_matrix + rows * d * 2 + rows * I * 2 == 326762496
    # weights + h read once + the fp32 weighted sum written once
    assert A["dn_bytes"] == 257 * per_matrix + rows * I * 2 + T * d * 4 == 160497664
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


@pytest.mark.parametrize("n,multi,probe", [(20, 8, 8), (5, 8, 8), (8, 8, None), (100, 8, 8), (7, 4, None), (1, 1, 8)])
def test_step_plan_runs_exactly_n_steps(n, multi, probe):
    """bench.py times exactly the requested steps: graph blocks of `multi` steps, probe blocks
    (phase by phase) every `probe` blocks starting with the first, and a partial block last."""
    plan = bench.step_plan(n, multi, probe)
    steps = []
    for kind, s in plan:
        steps += list(range(s, s + multi)) if kind == "multi" else [s]
    assert steps == list(range(n))
    if probe:
        assert plan[0][0] == "probe"
        # one probe step per probe block: a small share of the timed steps
        assert sum(k == "probe" for k, _ in plan) == -(-(-(-n // multi)) // probe)
    assert all(s % multi == 0 for kind, s in plan if kind == "multi")
