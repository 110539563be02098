"""The MoE-layer workloads and the recipe that draws each of their tensors.

Shapes (T tokens, hidden d, E routed experts, top-k, expert intermediate I, shared
intermediate I_shared, quant group 64) and distributions:

* activations x: bf16 ~N(0, 1)
* router weight W_r [E, d]: bf16 ~N(0, 0.02)
* expert weights: 4-bit codes uniform in [0, 15], groups of 64 along the input dim,
  one bf16 scale ~U(0.001, 0.01) and one bf16 bias ~U(-0.08, 0) per group
* skewed workload: the router logits get a per-expert fp32 bias
  3 * ln(r**-1.2 / H), H = sum_r r**-1.2, for the expert at rank r of a seeded
  random permutation of the experts

Layouts (expert is the outermost dimension; the checkpoint layout of the pages):

* gate, up codes   uint8  [E, I, d/2],  scales/biases bf16 bits [E, I, d/64]
* down codes       uint8  [E, d, I/2],  scales/biases bf16 bits [E, d, I/64]
* the shared expert is the same with E = 1 and I = I_shared.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from . import gen

BASE_SEED = 20261202

# per-tensor stream ids; a layer copy adds 1000 * layer
S_X, S_ROUTER, S_ZIPF_PERM, S_DECODE_X = 1, 2, 3, 4
S_ROUTED = 10   # + 3 * matrix (gate 0, up 1, down 2) + part (codes 0, scales 1, biases 2)
S_SHARED = 30


@dataclass(frozen=True)
class MoEShape:
    T: int
    d: int
    E: int = 256
    k: int = 8
    I: int = 512
    I_shared: int = 512
    group: int = 64


@dataclass(frozen=True)
class Workload:
    name: str
    shape: MoEShape
    seed: int
    router_std: float = 0.02
    zipf_s: Optional[float] = None
    zipf_scale: float = 3.0
    chunk: Optional[int] = None      # tokens per chunk (None: one chunk of T)
    layers: int = 1                  # independent layer copies of the weights
    steps: int = 1                   # decode steps (fresh activations per step)
    description: str = ""


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_t128_d512", MoEShape(T=128, d=512, I=128, I_shared=128), BASE_SEED + 1,
                 description="tiny MoE layer: T=128, d=512, 256 experts, top-8, I=128 + shared I=128"),
        Workload("prefill_t512_d2048", MoEShape(T=512, d=2048), BASE_SEED + 2,
                 description="prefill chunk of 512 tokens: d=2048, 256 experts, top-8, I=512 + shared I=512"),
        Workload("prefill_t4096_d2048", MoEShape(T=4096, d=2048), BASE_SEED + 3,
                 description="prefill chunk of 4096 tokens: d=2048, 256 experts, top-8, I=512 + shared I=512"),
        Workload("skew_t16384_d2048", MoEShape(T=16384, d=2048), BASE_SEED + 4, zipf_s=1.2, chunk=4096,
                 description="skewed long prefill: 16384 tokens in 4 chunks of 4096, Zipf(1.2) router bias"),
        Workload("decode_t1_d2048", MoEShape(T=1, d=2048), BASE_SEED + 5, layers=40, steps=1000,
                 description="batch-1 decode: 1 token per step, 40 layer copies, 1000 steps"),
    ]
}


@dataclass
class Q4:
    """One 4-bit group-affine matrix stack: codes, bf16 scales, bf16 biases."""
    codes: np.ndarray    # uint8  [E, N, K/2]
    scales: np.ndarray   # uint16 [E, N, K/64]
    biases: np.ndarray   # uint16 [E, N, K/64]


@dataclass
class ExpertWeights:
    gate: Q4
    up: Q4
    down: Q4

    @property
    def num_experts(self) -> int:
        return self.gate.codes.shape[0]


@dataclass
class LayerInputs:
    w_router: np.ndarray                 # uint16 [E, d]
    logit_bias: Optional[np.ndarray]     # float32 [E] or None
    routed: ExpertWeights
    shared: ExpertWeights
    extra: dict = field(default_factory=dict)


def _q4(seed: int, stream0: int, E: int, N: int, K: int) -> Q4:
    codes = gen.random_bytes(seed, stream0 + 0, (E, N, K // 2))
    scales = gen.uniform_bf16(seed, stream0 + 1, (E, N, K // 64), 0.001, 0.01)
    biases = gen.uniform_bf16(seed, stream0 + 2, (E, N, K // 64), -0.08, 0.0)
    return Q4(codes, scales, biases)


def make_expert_weights(seed: int, stream0: int, E: int, d: int, I: int) -> ExpertWeights:
    return ExpertWeights(
        gate=_q4(seed, stream0 + 0, E, I, d),
        up=_q4(seed, stream0 + 3, E, I, d),
        down=_q4(seed, stream0 + 6, E, d, I),
    )


def zipf_logit_bias(seed: int, E: int, s: float, scale: float) -> np.ndarray:
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** (-s)
    bias_by_rank = scale * np.log(p / p.sum())
    perm = gen.permutation(seed, S_ZIPF_PERM, E)
    out = np.empty(E, dtype=np.float64)
    out[perm] = bias_by_rank          # expert perm[r-1] has rank r
    return out.astype(np.float32)


def make_layer(wl: Workload, layer: int = 0) -> LayerInputs:
    sh = wl.shape
    off = 1000 * layer
    w_router = gen.normal_bf16(wl.seed, S_ROUTER + off, (sh.E, sh.d), 0.0, wl.router_std)
    bias = zipf_logit_bias(wl.seed, sh.E, wl.zipf_s, wl.zipf_scale) if wl.zipf_s else None
    routed = make_expert_weights(wl.seed, S_ROUTED + off, sh.E, sh.d, sh.I)
    shared = make_expert_weights(wl.seed, S_SHARED + off, 1, sh.d, sh.I_shared)
    return LayerInputs(w_router, bias, routed, shared)


def make_x(wl: Workload) -> np.ndarray:
    """All T prefill activations, bf16 bits [T, d] (chunks are row slices)."""
    return gen.normal_bf16(wl.seed, S_X, (wl.shape.T, wl.shape.d))


def make_decode_x(wl: Workload, steps: int) -> np.ndarray:
    """Fresh activations for ``steps`` decode steps, bf16 bits [steps, d]."""
    return gen.normal_bf16(wl.seed, S_DECODE_X, (steps, wl.shape.d))


def custom_workload(name: str, T: int, d: int, I: int, I_shared: Optional[int] = None, E: int = 256,
                    k: int = 8, seed: int = BASE_SEED + 100, **kw) -> Workload:
    """A workload with the same distributions and other sizes (tests, edge cases)."""
    return Workload(name, MoEShape(T=T, d=d, E=E, k=k, I=I, I_shared=I if I_shared is None else I_shared),
                    seed, **kw)
