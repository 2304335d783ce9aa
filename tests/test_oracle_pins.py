"""Pins of the fp64 oracle against things other than itself (CPU only).

Each check is chosen so that a plausible slip in the oracle -- a dropped term, a wrong
index or sign, a transposed operand, a double rounding, a wrong tie-break -- fails at
least one of them: exact rational brute force (``exact_ref``), library routines
(torch's fp32->bf16 conversion, numpy sorts, scipy's softmax/expit), closed forms and
invariants of the method described in "Hyper Optimizing Kimi K3 in vLLM: Moving Fast
and Responsibly", Part 1 sections 1-3.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest

from exact_ref import (bf16_bits_to_fraction, fraction_to_bf16_bits, linear_exact)

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def _bits_of_f32(x: float) -> int:
    return _f32_bits(x) >> 16


def _rand_bf16(rng, shape, scale=1.0):
    """Random bf16 patterns by truncating fp32 draws (test data only)."""
    v = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


# ------------------------------------------------------------------ bf16 ----

@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xC000, -2.0), (0x0000, 0.0), (0x3F81, 1.0 + 2.0 ** -7),
    (0x7F7F, (2 - 2.0 ** -7) * 2.0 ** 127), (0x0080, 2.0 ** -126), (0x0001, 2.0 ** -133),
    (0x8001, -(2.0 ** -133)), (0x3E80, 0.25), (0x4040, 3.0),
])
def test_bf16_decode_known_patterns(oracle_mod, bits, value):
    assert oracle_mod.bf16_to_f64(np.array([bits], np.uint16))[0] == value


@pytest.mark.parametrize("value,bits", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),                    # halfway, even is 1.0
    (1.0 + 3 * 2.0 ** -8, 0x3F82),                # halfway, even is 1+2^-6
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),       # above halfway only in fp64: no fp32 step
    (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
    (1.0 + 2.0 ** -8 - 2.0 ** -40, 0x3F80),
    (2.0 ** -134, 0x0000),                        # half the smallest subnormal: tie to 0
    (3 * 2.0 ** -134, 0x0002),                    # 1.5 quanta: tie to even 2
    (2.0 ** -134 + 2.0 ** -160, 0x0001),
    ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),       # max + half ulp: overflows
    ((2 - 2.0 ** -8) * 2.0 ** 127 * (1 - 2.0 ** -30), 0x7F7F),
    (float("inf"), 0x7F80), (-float("inf"), 0xFF80), (-0.0, 0x8000),
])
def test_bf16_encode_fixed_cases(oracle_mod, value, bits):
    assert int(oracle_mod.f64_to_bf16(np.array([value]))[0]) == bits


def test_bf16_encode_matches_torch_rne_on_fp32_values(oracle_mod):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    raw = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # keep finite values, and force many exact halfway cases (low 16 bits = 0x8000)
    raw[::4] = (raw[::4] & 0xFFFF0000) | 0x8000
    f = raw.view(np.float32)
    f = f[np.isfinite(f)]
    ours = oracle_mod.f64_to_bf16(f.astype(np.float64))
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_bf16_encode_matches_exact_rational_rounding(oracle_mod):
    rng = np.random.default_rng(2)
    vals = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000),
                           rng.standard_normal(500) * 2.0 ** -130])
    ours = oracle_mod.f64_to_bf16(vals)
    for v, b in zip(vals, ours):
        assert int(b) == fraction_to_bf16_bits(Fraction(float(v))), v


# ---------------------------------------------------------------- linear ----

@pytest.mark.parametrize("B,N,K", [(1, 5, 8), (2, 7, 24), (3, 4, 64), (5, 3, 40)])
def test_linear_brute_force_exact(oracle_mod, B, N, K):
    rng = np.random.default_rng(B * 100 + N * 10 + K)
    X = _rand_bf16(rng, (B, K))
    W = _rand_bf16(rng, (N, K), 0.02)
    R = _rand_bf16(rng, (B, N))
    for res in (None, R):
        y, Y = oracle_mod.linear(X, W, res)
        ex = linear_exact(X.tolist(), W.tolist(), None if res is None else res.tolist())
        for b in range(B):
            for n in range(N):
                assert abs(Fraction(y[b, n]) - ex[b][n]) <= abs(ex[b][n]) * 2 ** -45 + Fraction(1, 2 ** 140)
                assert int(Y[b, n]) == fraction_to_bf16_bits(ex[b][n])


def test_linear_one_hot_selects_weight_column(oracle_mod):
    rng = np.random.default_rng(3)
    N, K = 37, 96
    W = _rand_bf16(rng, (N, K))
    X = np.zeros((3, K), np.uint16)
    ks = [0, 50, 95]
    for b, k in enumerate(ks):
        X[b, k] = 0x3F80  # 1.0
    _, Y = oracle_mod.linear(X, W)
    for b, k in enumerate(ks):
        np.testing.assert_array_equal(Y[b], W[:, k])


def test_linear_identity_weight_returns_input(oracle_mod):
    rng = np.random.default_rng(4)
    K = 64
    W = np.zeros((K, K), np.uint16)
    W[np.arange(K), np.arange(K)] = 0x3F80
    X = _rand_bf16(rng, (4, K))
    _, Y = oracle_mod.linear(X, W)
    # -0.0 * 1 + (+0) sums to +0: compare values, not sign of zero
    np.testing.assert_array_equal(oracle_mod.bf16_to_f64(Y), oracle_mod.bf16_to_f64(X))


def test_linear_small_integers_exact_and_transpose_sensitive(oracle_mod):
    rng = np.random.default_rng(5)
    B, N, K = 3, 6, 1024
    Xi = rng.integers(-4, 5, (B, K)).astype(np.float32)
    Wi = rng.integers(-4, 5, (N, K)).astype(np.float32)
    X = (Xi.view(np.uint32) >> 16).astype(np.uint16)
    W = (Wi.view(np.uint32) >> 16).astype(np.uint16)
    y, _ = oracle_mod.linear(X, W)
    np.testing.assert_array_equal(y, Xi.astype(np.int64) @ Wi.astype(np.int64).T)


def test_linear_is_linear_in_x(oracle_mod):
    rng = np.random.default_rng(6)
    K, N = 256, 9
    Xa = rng.integers(-8, 9, (2, K)).astype(np.float32)
    Xb = rng.integers(-8, 9, (2, K)).astype(np.float32)
    W = _rand_bf16(rng, (N, K))
    enc = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)
    ya, _ = oracle_mod.linear(enc(Xa), W)
    yb, _ = oracle_mod.linear(enc(Xb), W)
    yab, _ = oracle_mod.linear(enc(Xa + Xb), W)
    np.testing.assert_allclose(yab, ya + yb, rtol=1e-12, atol=1e-12)


def test_residual_pins(oracle_mod):
    rng = np.random.default_rng(7)
    B, N, K = 4, 33, 128
    X = _rand_bf16(rng, (B, K))
    R = _rand_bf16(rng, (B, N))
    _, Y = oracle_mod.linear(X, np.zeros((N, K), np.uint16), R)
    np.testing.assert_array_equal(oracle_mod.bf16_to_f64(Y), oracle_mod.bf16_to_f64(R))
    W = _rand_bf16(rng, (N, K))
    y0, Y0 = oracle_mod.linear(X, W, np.zeros((B, N), np.uint16))
    y1, Y1 = oracle_mod.linear(X, W)
    np.testing.assert_array_equal(Y0, Y1)
    np.testing.assert_array_equal(y0, y1)


# ---------------------------------------------------------------- router ----

def _brute_topk(logits, k):
    """numpy lexsort on (index asc, fp32 logit desc)."""
    B, E = logits.shape
    out = np.empty((B, k), np.int32)
    for b in range(B):
        key = logits[b].astype(np.float32)
        order = np.lexsort((np.arange(E), -key.astype(np.float64)))
        out[b] = order[:k]
    return out


def test_route_equal_logits(oracle_mod):
    idx, w, probs = oracle_mod.route(np.full((3, 384), 0.75), 8)
    np.testing.assert_array_equal(idx, np.tile(np.arange(8), (3, 1)))
    assert np.all(w == 1.0 / 8)
    assert np.all(probs == 1.0 / 384)


def test_route_matches_sort_and_softmax(oracle_mod):
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((64, 384)) * 1.7
    idx, w, probs = oracle_mod.route(logits, 8)
    np.testing.assert_array_equal(idx, _brute_topk(logits, 8))
    np.testing.assert_allclose(probs, scipy_special.softmax(logits, axis=1), rtol=1e-13)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)
    assert np.all(np.diff(w, axis=1) <= 0)
    sel = np.take_along_axis(logits, idx, 1)
    np.testing.assert_allclose(w / w[:, :1], np.exp(sel - sel[:, :1]), rtol=1e-13)
    sel_p = np.take_along_axis(probs, idx, 1)
    np.testing.assert_allclose(w, sel_p / sel_p.sum(1, keepdims=True), rtol=1e-13)


def test_route_ties_break_to_lower_index(oracle_mod):
    logits = np.zeros((1, 16))
    logits[0, [3, 7, 11, 12]] = 2.0
    logits[0, [1, 14]] = 1.0
    idx, w, _ = oracle_mod.route(logits, 5)
    assert idx[0].tolist() == [3, 7, 11, 12, 1]
    # ties at the fp32 decision precision: these differ only below fp32 resolution
    logits = np.zeros((1, 8))
    logits[0, 5] = 1.0
    logits[0, 2] = 1.0 - 2.0 ** -40
    idx, _, _ = oracle_mod.route(logits, 1)
    assert idx[0, 0] == 2


def test_route_k_equals_e_is_sorted_permutation(oracle_mod):
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((2, 384))
    idx, w, probs = oracle_mod.route(logits, 384)
    for b in range(2):
        assert sorted(idx[b].tolist()) == list(range(384))
        assert np.all(np.diff(logits[b, idx[b]]) <= 0)
        np.testing.assert_allclose(w[b], probs[b, idx[b]], rtol=1e-13)


def test_route_closed_form_weights(oracle_mod):
    # logits ln(4), ln(3), ln(2), ln(1): renormalised top-2 weights are 4/7 and 3/7
    logits = np.log(np.array([[2.0, 1.0, 4.0, 3.0]]))
    idx, w, probs = oracle_mod.route(logits, 2)
    assert idx[0].tolist() == [2, 3]
    np.testing.assert_allclose(w[0], [4 / 7, 3 / 7], rtol=1e-15)
    np.testing.assert_allclose(probs[0], [0.2, 0.1, 0.4, 0.3], rtol=1e-15)


def test_moe_front_concatenation_order(oracle_mod):
    """Router rows come first in the concatenated weight; latent rows after them."""
    rng = np.random.default_rng(10)
    B, K, E, L = 3, 64, 16, 12
    # one-hot tokens make every logit an exact weight entry
    X = np.zeros((B, K), np.uint16)
    ks = [1, 20, 63]
    for b, k in enumerate(ks):
        X[b, k] = 0x3F80
    Wcat = _rand_bf16(rng, (E + L, K))
    out = oracle_mod.moe_front(X, Wcat, E, L, 4)
    for b, k in enumerate(ks):
        np.testing.assert_array_equal(out["logits"][b], oracle_mod.bf16_to_f64(Wcat[:E, k]))
        np.testing.assert_array_equal(out["latent"][b], Wcat[E:, k])
    np.testing.assert_array_equal(out["idx"], _brute_topk(out["logits"], 4))


def test_moe_front_random_matches_brute_force(oracle_mod):
    rng = np.random.default_rng(11)
    B, K, E, L, k = 2, 48, 10, 6, 3
    X = _rand_bf16(rng, (B, K))
    Wcat = _rand_bf16(rng, (E + L, K), 0.3)
    out = oracle_mod.moe_front(X, Wcat, E, L, k)
    ex = linear_exact(X.tolist(), Wcat.tolist())
    for b in range(B):
        for e in range(E):
            assert abs(Fraction(out["logits"][b, e]) - ex[b][e]) <= abs(ex[b][e]) * 2 ** -45
        for i in range(L):
            assert int(out["latent"][b, i]) == fraction_to_bf16_bits(ex[b][E + i])
    np.testing.assert_array_equal(out["idx"], _brute_topk(out["logits"], k))


def test_route_map_brute_force(oracle_mod):
    rng = np.random.default_rng(12)
    B, k, E = 37, 8, 384
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(B)]).astype(np.int32)
    m = oracle_mod.route_map(idx, E)
    flat = idx.reshape(-1)
    order = sorted(range(B * k), key=lambda p: (flat[p], p))
    assert m["pairs"].tolist() == order
    for at, p in enumerate(order):
        assert m["pos"][p] == at
    np.testing.assert_array_equal(m["counts"], np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(m["offsets"], np.concatenate([[0], np.cumsum(m["counts"])]))
    assert m["used"].tolist() == sorted(set(flat.tolist()))
    assert m["num_used"] == len(set(flat.tolist()))


# --------------------------------------------------------------- experts ----

def test_silu_closed_forms(oracle_mod):
    scipy_special = pytest.importorskip("scipy.special")
    assert oracle_mod.silu(0.0) == 0.0
    for t in [0.1, 0.5, 1.0, 2.5, 7.0, 30.0]:
        assert math.isclose(oracle_mod.silu(t) - oracle_mod.silu(-t), t, rel_tol=1e-15)
        assert math.isclose(oracle_mod.silu(t), t * scipy_special.expit(t), rel_tol=1e-15)
    assert oracle_mod.silu(60.0) == pytest.approx(60.0, rel=1e-20)
    assert abs(oracle_mod.silu(-60.0)) < 1e-24


def test_expert_mlp_brute_force(oracle_mod):
    rng = np.random.default_rng(13)
    H, I = 24, 8
    x = _rand_bf16(rng, (H,))
    Wgu = _rand_bf16(rng, (2 * I, H), 0.5)
    Wd = _rand_bf16(rng, (H, I), 0.5)
    a, y = oracle_mod.expert_mlp(x, Wgu, Wd)
    xs = x.tolist()
    a_ref = []
    for i in range(I):
        g = sum(bf16_bits_to_fraction(p) * bf16_bits_to_fraction(q) for p, q in zip(xs, Wgu[i].tolist()))
        u = sum(bf16_bits_to_fraction(p) * bf16_bits_to_fraction(q) for p, q in zip(xs, Wgu[I + i].tolist()))
        gf = float(g)
        act = Fraction(gf / (1.0 + math.exp(-gf))) * u
        a_ref.append(fraction_to_bf16_bits(act))
    # the activation value passes through exp(); allow one bf16 step on a near-halfway case
    diff = np.abs(a.astype(np.int32) - np.array(a_ref, np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.8
    a_use = a.tolist()
    for h in range(H):
        ex = sum(bf16_bits_to_fraction(p) * bf16_bits_to_fraction(q) for p, q in zip(a_use, Wd[h].tolist()))
        assert abs(Fraction(y[h]) - ex) <= abs(ex) * 2 ** -45 + Fraction(1, 2 ** 120)


def test_expert_gate_and_up_are_not_swapped(oracle_mod):
    # gate row = 0 gives silu(0) = 0 -> a = 0 regardless of up; the swap gives nonzero
    H, I = 8, 2
    x = np.full(H, 0x3F80, np.uint16)            # ones
    Wgu = np.zeros((2 * I, H), np.uint16)
    Wgu[I:, :] = 0x3F80                          # up rows = 1 -> up = 8
    Wd = np.full((H, I), 0x3F80, np.uint16)
    a, y = oracle_mod.expert_mlp(x, Wgu, Wd)
    assert np.all(a == 0) and np.all(y == 0)
    Wgu2 = np.zeros((2 * I, H), np.uint16)
    Wgu2[:I, :] = 0x3F80                         # gate = 8, up = 0 -> 0 as well
    Wgu2[I:, 0] = 0x3F80                         # up = 1
    a2, y2 = oracle_mod.expert_mlp(x, Wgu2, Wd)
    s8 = 8.0 / (1.0 + math.exp(-8.0))
    np.testing.assert_array_equal(a2, oracle_mod.f64_to_bf16(np.full(I, s8)))
    np.testing.assert_allclose(y2, np.full(H, I * oracle_mod.bf16_to_f64(a2[:1])[0]), rtol=1e-15)


def test_combine_closed_form(oracle_mod):
    w = np.array([[0.5, 0.25, 0.25]])
    yp = np.array([[[2.0, -4.0], [4.0, 8.0], [-8.0, 0.0]]])
    s = np.array([[1.0, 1.0]])
    y, Y = oracle_mod.combine(w, yp, s)
    np.testing.assert_array_equal(y, [[0.0 + 1.0, -2.0 + 2.0 + 1.0]])
    y2, _ = oracle_mod.combine(w, yp, None)
    np.testing.assert_array_equal(y2, [[0.0, 0.0]])


def _tiny_bank(rng, E, H, I):
    return _rand_bf16(rng, (E, 2 * I, H), 0.3), _rand_bf16(rng, (E, H, I), 0.3)


def test_moe_experts_all_slots_on_one_expert_equals_dense_mlp(oracle_mod):
    rng = np.random.default_rng(14)
    E, H, I, k, B = 6, 32, 16, 8, 3
    Wgu, Wd = _tiny_bank(rng, E, H, I)
    X = _rand_bf16(rng, (B, H))
    idx = np.full((B, k), 4, np.int32)
    w = np.full((B, k), 1.0 / k)
    y, Y = oracle_mod.moe_experts(X, idx, w, Wgu, Wd)
    for b in range(B):
        _, yd = oracle_mod.expert_mlp(X[b], Wgu[4], Wd[4])
        np.testing.assert_allclose(y[b], yd, rtol=1e-13, atol=1e-15)


def test_moe_experts_identical_experts_any_weight_split(oracle_mod):
    rng = np.random.default_rng(15)
    E, H, I, k, B = 4, 16, 8, 2, 2
    Wgu, Wd = _tiny_bank(rng, E, H, I)
    Wgu[2], Wd[2] = Wgu[0], Wd[0]
    X = _rand_bf16(rng, (B, H))
    idx = np.array([[0, 2], [2, 0]], np.int32)
    ya, _ = oracle_mod.moe_experts(X, idx, np.array([[0.7, 0.3], [0.1, 0.9]]), Wgu, Wd)
    yb, _ = oracle_mod.moe_experts(X, idx, np.array([[0.2, 0.8], [0.5, 0.5]]), Wgu, Wd)
    np.testing.assert_allclose(ya, yb, rtol=1e-13, atol=1e-15)


def test_moe_experts_routing_index_is_used(oracle_mod):
    """Token b with a single expert e (weight 1) must equal that expert's MLP."""
    rng = np.random.default_rng(16)
    E, H, I, B = 5, 16, 8, 5
    Wgu, Wd = _tiny_bank(rng, E, H, I)
    X = _rand_bf16(rng, (B, H))
    idx = np.array([[3], [0], [4], [1], [2]], np.int32)
    y, _ = oracle_mod.moe_experts(X, idx, np.ones((B, 1)), Wgu, Wd)
    for b in range(B):
        _, yd = oracle_mod.expert_mlp(X[b], Wgu[idx[b, 0]], Wd[idx[b, 0]])
        np.testing.assert_allclose(y[b], yd, rtol=1e-13, atol=1e-15)


def test_moe_experts_shared_expert_adds_with_weight_one(oracle_mod):
    rng = np.random.default_rng(17)
    E, H, I, k, B = 4, 16, 8, 2, 2
    Wgu, Wd = _tiny_bank(rng, E, H, I)
    Wgu_s, Wd_s = _rand_bf16(rng, (2 * I, H), 0.3), _rand_bf16(rng, (H, I), 0.3)
    X = _rand_bf16(rng, (B, H))
    idx = np.array([[1, 3], [0, 2]], np.int32)
    w = np.array([[0.6, 0.4], [0.5, 0.5]])
    y_r, _ = oracle_mod.moe_experts(X, idx, w, Wgu, Wd)
    y_rs, _ = oracle_mod.moe_experts(X, idx, w, Wgu, Wd, Wgu_s, Wd_s)
    for b in range(B):
        _, ys = oracle_mod.expert_mlp(X[b], Wgu_s, Wd_s)
        np.testing.assert_allclose(y_rs[b] - y_r[b], ys, rtol=1e-12, atol=1e-13)
