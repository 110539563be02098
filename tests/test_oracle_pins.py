"""Pins of the CPU oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: hand-derived values
(tests/golden/), closed forms, brute force on tiny inputs, or a special case that
reduces to a plain dense routine written independently here with numpy.
"""
import collections
import json
import math
import os
import struct

import numpy as np
import pytest

import oracle
from moe_workload import gen, configs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_val(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def to_bf16_exact(v: float) -> int:
    """bits of a float that is exactly representable in bf16 (asserted)."""
    u = struct.unpack("<I", struct.pack("<f", v))[0]
    assert u & 0xFFFF == 0, v
    return u >> 16


# ----------------------------------------------------------------------------- dequant
def test_dequant_hand_group_2x64():
    fx = json.load(open(os.path.join(GOLDEN, "dequant_group_2x64.json")))
    codes = np.stack([np.frombuffer(bytes.fromhex(r["codes_hex"]), dtype=np.uint8) for r in fx["rows"]])
    scales = np.array([[int(r["scale_bits"], 16)] for r in fx["rows"]], dtype=np.uint16)
    biases = np.array([[int(r["bias_bits"], 16)] for r in fx["rows"]], dtype=np.uint16)
    w = oracle.dequant_matrix(codes, scales, biases)
    assert w.shape == (2, 64)
    r0, r1 = fx["rows"]
    for k in range(64):
        q0 = r0["code_of_k"][k]
        assert bf16_val(w[0, k]) == r0["expected_by_code"][str(q0)], (k, q0)
        q1 = r1["code_of_k"][k]
        assert int(w[1, k]) == int(r1["expected_bits_by_code"][str(q1)], 16), (k, q1, hex(w[1, k]))
    # s*q == -b gives +0, not -0
    assert int(oracle.dequant_one(0x3C24, 0xBD24, 4)) == 0x0000


def test_nibble_order():
    # byte 0x1F: code 0 is the low nibble (15), code 1 the high nibble (1)
    codes = np.zeros((1, 32), dtype=np.uint8)
    codes[0, 0] = 0x1F
    w = oracle.dequant_matrix(codes, np.array([[0x3F80]], np.uint16), np.array([[0x0000]], np.uint16))
    assert bf16_val(w[0, 0]) == 15.0 and bf16_val(w[0, 1]) == 1.0 and bf16_val(w[0, 2]) == 0.0


def test_dequant_group_index_and_single_rounding():
    # weight k uses group k // 64; scale 1 for group 0, 2 for group 1
    codes = np.full((1, 64), 0x11, dtype=np.uint8)    # all codes 1, K = 128
    w = oracle.dequant_matrix(codes, np.array([[0x3F80, 0x4000]], np.uint16), np.array([[0, 0]], np.uint16))
    assert all(bf16_val(v) == 1.0 for v in w[0, :64]) and all(bf16_val(v) == 2.0 for v in w[0, 64:])
    # exact value 1 + 2^-8 + 2^-14 (s = 1 + 2^-7, q = 1, b = -2^-8 + 2^-14 is not bf16 ...) -> use a
    # construction with a true sum just above a bf16 midpoint: s*q = 2^-9 (tiny), b = 1 + 2^-7
    # sum = 1 + 2^-7 + 2^-9: mantissa (2^-7 + 2^-9)*128 = 1.25 -> rounds to 1 -> 1 + 2^-7
    s = to_bf16_exact(2.0 ** -9)
    b = to_bf16_exact(1.0 + 2.0 ** -7)
    assert bf16_val(oracle.dequant_one(s, b, 1)) == 1.0 + 2.0 ** -7
    # q = 2: 1 + 2^-7 + 2^-8 -> mantissa 1.5 -> tie -> even (2) -> 1 + 2^-6
    assert bf16_val(oracle.dequant_one(s, b, 2)) == 1.0 + 2.0 ** -6
    # q = 3: 1 + 2^-7 + 3*2^-9 -> 1.75 -> 2 -> 1 + 2^-6
    assert bf16_val(oracle.dequant_one(s, b, 3)) == 1.0 + 2.0 ** -6
    # a case where rounding s*q to float first then adding would double-round:
    # s = 1 + 2^-7 (bf16), q = 15: s*q = 15 + 15/128 = 15.1171875 (exact, 12 bits);
    # b = 2^-20 breaks the tie of 15.125? 15.1171875 + 2^-20 -> bf16 quantum at 15 is 2^-4:
    # 15.1171875 / 2^-4 = 241.875 -> 242 -> 15.125
    assert bf16_val(oracle.dequant_one(to_bf16_exact(1.0 + 2.0 ** -7), to_bf16_exact(2.0 ** -20), 15)) == 15.125


def test_bf16_round_ties_and_sticky():
    assert oracle.bf16_round(1.0) == 0x3F80
    assert oracle.bf16_round(1.0 + 2.0 ** -8) == 0x3F80           # tie -> even
    assert oracle.bf16_round(1.0 + 3 * 2.0 ** -8) == 0x3F82       # tie -> even (up)
    assert oracle.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81  # above the tie
    assert oracle.bf16_round(-1.0 - 2.0 ** -8 - 2.0 ** -30) == 0xBF81
    assert oracle.bf16_round(0.0) == 0x0000 and oracle.bf16_round(-0.0) == 0x8000


def test_q4_bytes_closed_form():
    # 4-bit codes plus one bf16 scale and one bf16 bias per 64 weights: 0.5625 B per weight
    assert oracle.q4_bytes(1, 64) == 36.0
    # the pages: ~70 GB of bf16 weights (35B parameters) shrink to a 19.4 GB checkpoint
    q4_gb = 35e9 * oracle.q4_bytes(1, 64) / 64 / 1e9
    assert abs(q4_gb - 19.4) / 19.4 < 0.02
    assert abs(35e9 * 2 / 1e9 - 70) < 1e-9


# ----------------------------------------------------------------------------- router
def _router_case_from_fixture():
    fx = json.load(open(os.path.join(GOLDEN, "router_order_case.json")))
    d = 256
    x = np.zeros((1, d), np.uint16)
    w = np.zeros((1, d), np.uint16)
    for k, v in fx["nonzero_x"].items():
        x[0, int(k)] = to_bf16_exact(v)
    for k, v in fx["nonzero_w"].items():
        w[0, int(k)] = to_bf16_exact(v)
    return fx, x, w


def test_router_pinned_order_hand_case():
    fx, x, w = _router_case_from_fixture()
    assert oracle.router_logits(x, w)[0, 0] == fx["expected_logit"]
    assert oracle.router_logits(x, w, np.array([0.5], np.float32))[0, 0] == fx["expected_logit_with_bias_0.5"]
    # the two other orders give different values, so the case does pin the order
    assert fx["sequential_fp32_sum"] != fx["expected_logit"] != fx["exact_sum"]


def test_router_lane_interleave_moves_each_term():
    # a single product at k lands in chain (k % 256) // 8 whatever i is: moving one unit
    # product around must not change the result (catches dropped or mis-indexed terms)
    d = 512
    for k in [0, 7, 8, 255, 256, 300, 511]:
        x = np.zeros((1, d), np.uint16)
        w = np.zeros((1, d), np.uint16)
        x[0, k] = to_bf16_exact(1.5)
        w[0, k] = to_bf16_exact(-2.0)
        assert oracle.router_logits(x, w)[0, 0] == -3.0


def test_router_within_fp32_error_bound():
    wl = configs.custom_workload("t", T=16, d=2048, I=64)
    lay = configs.make_layer(wl)
    x = configs.make_x(wl)
    lg = oracle.router_logits(x, lay.w_router)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    wf = gen.bf16_bits_to_f32(lay.w_router).astype(np.float64)
    exact = xf @ wf.T                       # fp64: exact to ~1e-16 for these sizes
    absdot = np.abs(xf) @ np.abs(wf).T
    gamma = 69 * 2.0 ** -24 / (1 - 69 * 2.0 ** -24)   # 64 chained fma + 5 tree adds
    err = np.abs(lg.astype(np.float64) - exact)
    assert np.all(err <= gamma * absdot + 1e-30)
    assert err.max() > 0                    # fp32 really rounds here


def test_router_bias_added_after_tree():
    fx, x, w = _router_case_from_fixture()
    b = np.array([2.0 ** 24], np.float32)   # 3 + 2^24 -> 2^24 + 4 in fp32 (tie to even at 2^24+3?)
    v = oracle.router_logits(x, w, b)[0, 0]
    assert v == np.float32(np.float32(3.0) + np.float32(2.0 ** 24))


# ----------------------------------------------------------------------------- top-k
def test_topk_bruteforce_and_ties():
    rng = np.random.default_rng(0)
    T, E, k = 24, 256, 8
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[0, 10] = lg[0, 3] = lg[0, 200] = 9.0        # three-way tie at the top
    lg[1, :] = 0.0                                  # all equal: experts 0..7
    lg[2, 17] = np.float32(-0.0)
    lg[2, 5] = np.float32(0.0)
    lg[2, :] = np.where(np.arange(E) < 2, 0.0, -1.0).astype(np.float32)
    lg[2, 1] = -0.0                                 # -0 == +0: lower index first
    lg[3, 40] = np.nan                              # NaN counts as -inf
    idx, w = oracle.topk(lg, k)
    for t in range(T):
        key = [(-(-math.inf if math.isnan(v) else float(v)), e) for e, v in enumerate(lg[t])]
        want = [e for _, e in sorted(key)[:k]]
        assert list(idx[t]) == want, t
    assert list(idx[0, :3]) == [3, 10, 200]
    assert list(idx[1]) == list(range(8))
    assert list(idx[2, :2]) == [0, 1]
    assert 40 not in idx[3]


def test_router_tie_from_duplicate_rows():
    wl = configs.custom_workload("t", T=8, d=256, I=64)
    lay = configs.make_layer(wl)
    x = configs.make_x(wl)
    wr = lay.w_router.copy()
    wr[77] = wr[12]                     # identical rows -> identical logits
    lg = oracle.router_logits(x, wr)
    assert np.array_equal(lg[:, 77], lg[:, 12])
    wr[:] = wr[5]                       # every expert identical: top-8 is 0..7, weights 1/8
    idx, w = oracle.topk(oracle.router_logits(x, wr))
    assert (idx == np.arange(8)).all() and np.allclose(w, 1 / 8, rtol=0, atol=1e-15)


def test_routing_weights_softmax_closed_form():
    rng = np.random.default_rng(1)
    lg = (rng.standard_normal((32, 256)) * 2).astype(np.float32)
    idx, w = oracle.topk(lg)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)
    assert (np.diff(w, axis=1) <= 0).all()
    for t in range(32):
        full = np.exp(lg[t].astype(np.float64) - lg[t].max())
        full /= full.sum()                                    # softmax over all 256
        renorm = full[idx[t]] / full[idx[t]].sum()            # renormalised over the kept 8
        assert np.allclose(w[t], renorm, rtol=1e-13, atol=0)


# ----------------------------------------------------------------------------- routing metadata
@pytest.mark.parametrize("T,BM", [(1, 32), (13, 16), (64, 32), (2048, 32)])
def test_route_meta_invariants(T, BM):
    rng = np.random.default_rng(T)
    E, k = 256, 8
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    m = oracle.route_meta(idx, E, BM)
    cnt = collections.Counter(idx.ravel().tolist())
    assert [cnt.get(e, 0) for e in range(E)] == m["counts"].tolist()       # brute-force histogram
    assert m["counts"].sum() == k * T
    off = m["offsets"]
    assert off[0] == 0 and off[E] == k * T and (np.diff(off) >= 0).all()
    assert (np.diff(off) == m["counts"]).all()
    perm, pos = m["perm"], m["pos"].ravel()
    assert sorted(perm.tolist()) == list(range(k * T))                      # bijection
    assert (pos[perm] == np.arange(k * T)).all()
    for e in range(E):
        grp = perm[off[e]:off[e + 1]]
        assert (idx.ravel()[grp] == e).all()
        toks = grp // k
        assert (np.diff(toks) > 0).all()                                   # ascending tokens
    tiles = m["tiles"]
    assert tiles[:, 2].sum() == k * T and (tiles[:, 2] >= 1).all() and (tiles[:, 2] <= BM).all()
    covered = np.zeros(k * T, np.int32)
    for e, r0, n in tiles:
        assert off[e] <= r0 and r0 + n <= off[e + 1]
        covered[r0:r0 + n] += 1
    assert (covered == 1).all()
    assert list(tiles[:, 0]) == sorted(tiles[:, 0])
    assert m["num_tiles"] == sum((c + BM - 1) // BM for c in m["counts"])
    # inside a group the tiles follow the rows: the first starts at the group's offset, each
    # next one where the previous ended, and only the group's last tile may hold fewer than BM
    for e in range(E):
        te = tiles[tiles[:, 0] == e]
        if m["counts"][e] == 0:
            assert len(te) == 0
            continue
        assert te[0, 1] == off[e] and te[-1, 1] + te[-1, 2] == off[e + 1]
        assert (te[1:, 1] == te[:-1, 1] + te[:-1, 2]).all()
        assert (te[:-1, 2] == BM).all() and 1 <= te[-1, 2] <= BM
    if T == 2048:                        # the pages: 2K tokens -> 16,384 assignments, 64 per expert
        assert k * T == 16384 and m["counts"].mean() == 64.0


def test_route_meta_short_tile_is_last_of_its_group():
    """Hand case: expert 5 gets 3 rows, expert 9 gets 40, tile_rows 16: the block map is
    (5, 0, 3), (9, 3, 16), (9, 19, 16), (9, 35, 8) -- the short tile closes each group."""
    idx = np.zeros((40, 8), np.int32)
    for t in range(40):
        others = [e for e in range(20, 256) if e % 7 == t % 7][:6]
        idx[t] = [9] + ([5] if t < 3 else [10 + t % 5 * 2 + 1]) + others
    m = oracle.route_meta(idx, 256, 16)
    te = [tuple(r) for r in m["tiles"] if r[0] in (5, 9)]
    assert te == [(5, 0, 3), (9, 3, 16), (9, 19, 16), (9, 35, 8)]


# ----------------------------------------------------------------------------- FFN
def _unpack_codes(codes: np.ndarray) -> np.ndarray:
    """[.., K/2] bytes -> [.., K] codes (independent numpy unpack)."""
    lo = codes & 0x0F
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2).astype(np.float64)


def _exact_weights(E, N, K, rng):
    """codes with scale 1/16 and bias 0: w = q / 16 is exact in bf16."""
    codes = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    scales = np.full((E, N, K // 64), 0x3D80, np.uint16)
    biases = np.zeros((E, N, K // 64), np.uint16)
    return configs.Q4(codes, scales, biases)


def test_ffn_reduces_to_dense_swiglu():
    rng = np.random.default_rng(7)
    d, I = 128, 64
    W = configs.ExpertWeights(_exact_weights(2, I, d, rng), _exact_weights(2, I, d, rng),
                              _exact_weights(2, d, I, rng))
    x = gen.normal_bf16(3, 3, (d,))
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    for e in range(2):
        Wg = _unpack_codes(W.gate.codes[e]) / 16
        Wu = _unpack_codes(W.up.codes[e]) / 16
        Wd = _unpack_codes(W.down.codes[e]) / 16
        g, u = Wg @ xf, Wu @ xf
        h = g / (1 + np.exp(-g)) * u
        y = Wd @ h
        y_or, h_or = oracle.expert_ffn(W, e, x, return_h=True)
        assert np.allclose(h_or, h, rtol=1e-12, atol=1e-12)
        assert np.allclose(y_or, y, rtol=1e-12, atol=1e-9)


def test_moe_identical_experts_and_zero_shared():
    """All routed experts identical -> out = y_e + y_shared whatever the weights (sum w = 1);
    a shared expert with zero weights adds nothing."""
    wl = configs.custom_workload("t", T=4, d=128, I=64, I_shared=64)
    lay = configs.make_layer(wl)
    x = configs.make_x(wl)
    one = lay.routed
    same = configs.ExpertWeights(*[configs.Q4(np.repeat(m.codes[:1], 256, 0), np.repeat(m.scales[:1], 256, 0),
                                              np.repeat(m.biases[:1], 256, 0)) for m in (one.gate, one.up, one.down)])
    r = oracle.route(x, lay.w_router)
    zero = configs.ExpertWeights(*[configs.Q4(np.zeros_like(m.codes), m.scales, np.zeros_like(m.biases))
                                   for m in (lay.shared.gate, lay.shared.up, lay.shared.down)])
    out = oracle.moe_tokens(x, r["topk_idx"], r["topk_w"], same, zero)
    for t in range(4):
        y0 = oracle.expert_ffn(same, 0, x[t])
        assert np.allclose(out[t], y0, rtol=1e-12, atol=1e-12)
    out_sh = oracle.moe_tokens(x, r["topk_idx"], r["topk_w"], same, lay.shared)
    ysh = np.stack([oracle.expert_ffn(lay.shared, 0, x[t]) for t in range(4)])
    assert np.allclose(out_sh - out, ysh, rtol=1e-12, atol=1e-12)
    assert np.abs(ysh).max() > 0.01


def _dense_swiglu(W, e, xf):
    """SwiGLU of expert e on one row with the exact weights of _exact_weights (q / 16), numpy."""
    g = (_unpack_codes(W.gate.codes[e]) / 16) @ xf
    u = (_unpack_codes(W.up.codes[e]) / 16) @ xf
    return (_unpack_codes(W.down.codes[e]) / 16) @ (g / (1 + np.exp(-g)) * u)


def test_weighted_combine_pairs_each_weight_with_its_slot_expert():
    """Eight distinct experts per token with exact weights and unequal routing weights: the
    layer output is sum_j w_j SwiGLU_{e_j}(x) + SwiGLU_shared(x) (the output projection
    weighted by the routing score, plus the shared expert: section "Reduce intermediate and
    state traffic"), written here with numpy.  A weight paired with another slot's expert,
    or a dropped shared term, lands far outside the tolerance (checked below)."""
    rng = np.random.default_rng(11)
    E, d, I, k, T = 256, 128, 64, 8, 4
    routed = configs.ExpertWeights(_exact_weights(E, I, d, rng), _exact_weights(E, I, d, rng),
                                   _exact_weights(E, d, I, rng))
    shared = configs.ExpertWeights(_exact_weights(1, I, d, rng), _exact_weights(1, I, d, rng),
                                   _exact_weights(1, d, I, rng))
    x = gen.normal_bf16(5, 5, (T, d), std=0.05)
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = np.sort(rng.uniform(0.02, 1.0, (T, k)), axis=1)[:, ::-1]
    w = np.ascontiguousarray(w / w.sum(1, keepdims=True))
    out = oracle.moe_tokens(x, idx, w, routed, shared)
    for t in range(T):
        xf = gen.bf16_bits_to_f32(x[t]).astype(np.float64)
        ys = [_dense_swiglu(routed, e, xf) for e in idx[t]]
        ysh = _dense_swiglu(shared, 0, xf)
        ref = sum(w[t, j] * ys[j] for j in range(k)) + ysh
        tol = 1e-9 * np.abs(ref).max()
        assert np.abs(out[t] - ref).max() <= tol
        # the pin discriminates: slots 0 and 1 swapped, or no shared expert, differ by far more
        swapped = ref + (w[t, 1] - w[t, 0]) * (ys[0] - ys[1])
        assert np.abs(swapped - ref).max() > 1e6 * tol
        assert np.abs(ysh).max() > 1e6 * tol


def test_chunking_leaves_outputs_unchanged():
    """The pages: chunked prefill does not change the model output (section 'Limit temporary
    memory with prompt chunking'); per token the MoE layer is independent of the others."""
    wl = configs.custom_workload("t", T=12, d=256, I=64, I_shared=64)
    lay = configs.make_layer(wl)
    x = configs.make_x(wl)
    r = oracle.route(x, lay.w_router)
    full = oracle.moe_tokens(x, r["topk_idx"], r["topk_w"], lay.routed, lay.shared)
    parts = []
    for c in range(3):
        xc = np.ascontiguousarray(x[4 * c:4 * c + 4])
        rc = oracle.route(xc, lay.w_router)
        assert np.array_equal(rc["topk_idx"], r["topk_idx"][4 * c:4 * c + 4])
        parts.append(oracle.moe_tokens(xc, rc["topk_idx"], rc["topk_w"], lay.routed, lay.shared))
    assert np.array_equal(np.concatenate(parts), full)


def test_silu_gate_is_first_projection():
    """Swapping gate and up changes the result (silu acts on the gate projection only)."""
    wl = configs.custom_workload("t", T=1, d=128, I=64)
    lay = configs.make_layer(wl)
    x = configs.make_x(wl)[0]
    W = lay.routed
    y = oracle.expert_ffn(W, 3, x)
    Wsw = configs.ExpertWeights(W.up, W.gate, W.down)
    y2 = oracle.expert_ffn(Wsw, 3, x)
    assert not np.allclose(y, y2)
    _, h = oracle.expert_ffn(W, 3, x, return_h=True)
    g = np.array([sum(gen.bf16_bits_to_f32(x[k]).astype(np.float64) * bf16_val(v) for k, v in enumerate(row))
                  for row in oracle.dequant_matrix(W.gate.codes[3], W.gate.scales[3], W.gate.biases[3])])
    u = np.array([sum(gen.bf16_bits_to_f32(x[k]).astype(np.float64) * bf16_val(v) for k, v in enumerate(row))
                  for row in oracle.dequant_matrix(W.up.codes[3], W.up.scales[3], W.up.biases[3])])
    assert np.allclose(h, g / (1 + np.exp(-g)) * u, rtol=1e-12, atol=1e-14)
