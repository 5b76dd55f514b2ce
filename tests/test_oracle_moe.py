"""Pins for the oracle's routing, dispatch, expert FFN and combine (CPU only).

The checks come from outside the oracle: hand-derived fixtures, closed forms,
scipy's independent logistic, Python-level brute force (sorted(), explicit loops,
integer nibble extraction) and invariants of the layer.
"""

import json
import math
import os

import numpy as np
import pytest

import synthetic
from oracle import moe, quant

from conftest import GOLDEN


# ---------------------------------------------------------------- elementwise

def test_sigmoid_closed_forms_and_scipy():
    special = pytest.importorskip("scipy.special")
    z = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(moe.sigmoid(z), special.expit(z), rtol=1e-15, atol=1e-300)
    assert moe.sigmoid(0.0) == 0.5
    assert abs(moe.sigmoid(math.log(3.0)) - 0.75) < 1e-16
    np.testing.assert_allclose(moe.sigmoid(z) + moe.sigmoid(-z), 1.0, rtol=0, atol=1e-15)
    assert moe.sigmoid(-1000.0) == 0.0 and moe.sigmoid(1000.0) == 1.0


def test_silu_closed_forms():
    assert moe.silu(0.0) == 0.0
    assert abs(moe.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(moe.silu(50.0) - 50.0) < 1e-15
    assert abs(moe.silu(-50.0)) < 1e-18


def test_bf16_round_trip_and_rne():
    bits = np.arange(0, 1 << 16, 7, dtype=np.uint32).astype(np.uint16)
    vals = moe.bf16_bits_to_f64(bits)
    finite = np.isfinite(vals)
    np.testing.assert_array_equal(moe.f32_to_bf16_bits(vals[finite]), bits[finite])
    # 1 + 2^-8 is exactly half way between bf16 1.0 and 1 + 2^-7: ties go to even (1.0)
    assert moe.f32_to_bf16_bits(np.float32(1 + 2 ** -8)) == 0x3F80
    assert moe.f32_to_bf16_bits(np.float32(1 + 3 * 2 ** -8)) == 0x3F82   # tie, odd below -> up
    assert moe.f32_to_bf16_bits(np.float32(1 + 2 ** -8 + 2 ** -20)) == 0x3F81


# ---------------------------------------------------------------- routing

def test_route_hand_derived_cases():
    with open(os.path.join(GOLDEN, "route_tiny.json")) as f:
        fx = json.load(f)
    x = np.array([fx["x"]])
    wr = np.array(fx["w_router"], dtype=np.float32)
    for c in fx["cases"]:
        r = moe.route(x, wr, None if c["bias"] is None else np.array(c["bias"]), c["k"])
        np.testing.assert_array_equal(r["idx"][0], c["idx"])
        np.testing.assert_allclose(r["w"][0], c["w"], rtol=1e-15)


def _route_brute(x, wr, bias, k):
    """Per token: Python sorted() by (-sel, id), scores with math.exp."""
    T, E = x.shape[0], wr.shape[0]
    idx, w = [], []
    for t in range(T):
        s, sel = [], []
        for e in range(E):
            l = math.fsum(float(x[t, h]) * float(wr[e, h]) for h in range(x.shape[1]))
            se = 1.0 / (1.0 + math.exp(-l))
            s.append(se)
            sel.append(se + (0.0 if bias is None else float(bias[e])))
        top = sorted(sorted(range(E), key=lambda e: (-sel[e], e))[:k])
        tot = math.fsum(s[e] for e in top)
        idx.append(top)
        w.append([s[e] / tot for e in top])
    return np.array(idx), np.array(w)


@pytest.mark.parametrize("with_bias", [False, True])
def test_route_matches_brute_force(with_bias):
    T, H, E, k = 5, 24, 11, 3
    rng = np.random.default_rng(5)
    x = moe.bf16_bits_to_f64(synthetic.activations_bits(T, H, seed=7))
    wr = (rng.standard_normal((E, H)) * 0.3).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.2).astype(np.float32) if with_bias else None
    r = moe.route(x, wr, bias, k)
    bi, bw = _route_brute(x, wr, bias, k)
    np.testing.assert_array_equal(r["idx"], bi)
    np.testing.assert_allclose(r["w"], bw, rtol=1e-14)


def test_route_exact_ties_go_to_lower_id():
    H, E = 8, 6
    x = moe.bf16_bits_to_f64(synthetic.activations_bits(3, H, seed=1))
    wr = np.tile(np.linspace(-0.1, 0.1, H, dtype=np.float32), (E, 1))   # all logits equal
    r = moe.route(x, wr, None, 4)
    np.testing.assert_array_equal(r["idx"], np.tile([0, 1, 2, 3], (3, 1)))
    np.testing.assert_allclose(r["w"], 0.25, rtol=1e-15)
    assert np.all(r["gap"] == 0)


def test_route_k_equals_e_and_invariants():
    T, H, E = 16, 64, 16
    x = moe.bf16_bits_to_f64(synthetic.activations_bits(T, H, seed=2))
    wr = synthetic.router_weights(E, H, seed=2)
    r = moe.route(x, wr, None, E)
    np.testing.assert_array_equal(r["idx"], np.tile(np.arange(E), (T, 1)))
    np.testing.assert_allclose(r["w"], r["score"] / r["score"].sum(1, keepdims=True), rtol=1e-15)
    r = moe.route(x, wr, synthetic.zipf_bias(E, beta=0.05), 4)
    for t in range(T):
        assert len(set(r["idx"][t])) == 4 and np.all(np.diff(r["idx"][t]) > 0)
    np.testing.assert_allclose(r["w"].sum(1), 1.0, rtol=0, atol=1e-15)
    assert np.all(r["gap"] >= 0)


# ---------------------------------------------------------------- dispatch

def test_dispatch_matches_python_stable_sort():
    rng = np.random.default_rng(6)
    T, E, k = 37, 13, 4
    idx = np.array([sorted(rng.choice(E, size=k, replace=False)) for _ in range(T)])
    d = moe.dispatch(idx, E)
    flat = idx.reshape(-1).tolist()
    perm = [p for e in range(E) for p in range(len(flat)) if flat[p] == e]
    np.testing.assert_array_equal(d["perm"], perm)
    counts = [flat.count(e) for e in range(E)]
    np.testing.assert_array_equal(d["counts"], counts)
    off = [0]
    for c in counts:
        off.append(off[-1] + c)
    np.testing.assert_array_equal(d["offsets"], off)
    for q, p in enumerate(perm):
        assert d["inv_perm"][p] == q
    np.testing.assert_array_equal(d["active"], [e for e in range(E) if counts[e]])
    assert d["n_active"] == sum(1 for c in counts if c)


# ---------------------------------------------------------------- FFN / layer

def test_swiglu_hand_derived():
    with open(os.path.join(GOLDEN, "swiglu_tiny.json")) as f:
        fx = json.load(f)
    y = moe.expert_ffn(np.array([fx["x"]]), np.array(fx["w_gate"]), np.array(fx["w_up"]), np.array(fx["w_down"]))
    np.testing.assert_allclose(y[0], fx["y"], rtol=1e-15)


def test_identity_down_reduces_to_swiglu_activation():
    rng = np.random.default_rng(8)
    H = I = 8
    x = rng.standard_normal((3, H))
    Wg, Wu = rng.standard_normal((I, H)), rng.standard_normal((I, H))
    y = moe.expert_ffn(x, Wg, Wu, np.eye(H))
    g, u = np.einsum("th,ih->ti", x, Wg), np.einsum("th,ih->ti", x, Wu)
    np.testing.assert_allclose(y, g / (1 + np.exp(-g)) * u, rtol=1e-12, atol=1e-15)


def _tiny_layer(T=4, seed=0):
    cfg = synthetic.CONFIGS["tiny"]
    inp = synthetic.layer_inputs_small(cfg, T=T)
    experts = [quant.quantize_expert(*w, cfg.group) for w in inp["experts_fp32"]]
    shared = quant.quantize_expert(*inp["shared_fp32"], cfg.group)
    return cfg, inp, experts, shared


def _dequant_by_bytes(packed, scales, K, G):
    """Independent per-element dequant using Python integers."""
    N = packed.shape[0]
    out = np.empty((N, K))
    for n in range(N):
        row = packed[n].tolist()
        sc = [float(v) for v in scales[n]]
        for k in range(K):
            b = row[k >> 1]
            u = (b >> 4) if (k & 1) else (b & 15)
            out[n, k] = (u - 8) * sc[k // G]
    return out


def test_layer_matches_dense_brute_force_on_tiny_config():
    """All experts evaluated densely for every token, masked by the routing weights."""
    cfg, inp, experts, shared = _tiny_layer()
    H, I, E, k, G = cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group
    out = moe.moe_layer(inp["x_bits"], inp["w_router"], None, experts, shared, H, I, E, k, G)
    x = out["x"]
    T = x.shape[0]
    gate_w = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            gate_w[t, out["idx"][t, j]] = out["w"][t, j]

    def ffn_dense(ex):
        comb = _dequant_by_bytes(ex["w_gate_up"], ex["s_gate_up"], H, G)
        wd = _dequant_by_bytes(ex["w_down"], ex["s_down"], I, G)
        y = np.zeros((T, H))
        for t in range(T):
            for i in range(I):
                blk, o = divmod(i, 16)
                gi = float(np.dot(comb[32 * blk + o], x[t]))
                ui = float(np.dot(comb[32 * blk + 16 + o], x[t]))
                hi = gi / (1.0 + math.exp(-gi)) * ui
                y[t] += hi * wd[:, i]
        return y

    y = ffn_dense(shared)
    for e in range(E):
        y += gate_w[:, [e]] * ffn_dense(experts[e])
    np.testing.assert_allclose(out["y"], y, rtol=1e-12, atol=1e-14)
    # exactly k distinct experts per token and weights summing to one
    assert np.all((gate_w > 0).sum(1) == k)
    np.testing.assert_allclose(gate_w.sum(1), 1.0, atol=1e-15)


def test_token_order_invariance_is_exact():
    cfg, inp, experts, shared = _tiny_layer(T=6)
    H, I, E, k, G = cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group
    a = moe.moe_layer(inp["x_bits"], inp["w_router"], None, experts, shared, H, I, E, k, G)
    order = np.array([3, 0, 5, 1, 4, 2])
    b = moe.moe_layer(inp["x_bits"][order], inp["w_router"], None, experts, shared, H, I, E, k, G)
    np.testing.assert_array_equal(b["idx"], a["idx"][order])
    np.testing.assert_allclose(b["y"], a["y"][order], rtol=1e-13, atol=1e-15)


def test_zero_down_expert_contributes_nothing():
    cfg, inp, experts, shared = _tiny_layer()
    H, I, E, k, G = cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group
    base = moe.moe_layer(inp["x_bits"], inp["w_router"], None, experts, shared, H, I, E, k, G)
    e0 = int(base["idx"][0, 0])
    zeroed = list(experts)
    zeroed[e0] = dict(experts[e0])
    zeroed[e0]["s_down"] = np.zeros_like(experts[e0]["s_down"])
    out = moe.moe_layer(inp["x_bits"], inp["w_router"], None, zeroed, shared, H, I, E, k, G)
    rows = base["inv_perm"][np.nonzero(base["idx"].reshape(-1) == e0)[0]]
    assert np.all(out["expert_out"][rows] == 0)
    want = base["y"].copy()
    for t in range(base["idx"].shape[0]):
        for j in range(k):
            if base["idx"][t, j] == e0:
                want[t] -= base["w"][t, j] * base["expert_out"][base["inv_perm"][t * k + j]]
    np.testing.assert_allclose(out["y"], want, rtol=1e-12, atol=1e-14)


def test_zero_input_gives_zero_output():
    cfg, inp, experts, shared = _tiny_layer()
    H, I, E, k, G = cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group
    x0 = np.zeros_like(inp["x_bits"])
    out = moe.moe_layer(x0, inp["w_router"], None, experts, shared, H, I, E, k, G)
    # every score is sigmoid(0) = 1/2: a full tie resolved to the lowest ids
    np.testing.assert_array_equal(out["idx"], np.tile(np.arange(k), (x0.shape[0], 1)))
    assert np.all(out["y"] == 0)


def test_expert_out_order_and_shared_rows():
    cfg, inp, experts, shared = _tiny_layer()
    H, I, E, k, G = cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group
    out = moe.moe_layer(inp["x_bits"], inp["w_router"], None, experts, shared, H, I, E, k, G)
    T = out["x"].shape[0]
    for q in range(T * k):
        p = out["perm"][q]
        t, e = p // k, out["idx"].reshape(-1)[p]
        Wg, Wu, Wd = quant.dequantize_expert(experts[e], H, I, G)
        np.testing.assert_allclose(out["expert_out"][q], moe.expert_ffn(out["x"][[t]], Wg, Wu, Wd)[0], rtol=1e-12, atol=1e-15)
    Sg, Su, Sd = quant.dequantize_expert(shared, H, I, G)
    np.testing.assert_allclose(out["expert_out"][T * k:], moe.expert_ffn(out["x"], Sg, Su, Sd), rtol=1e-12, atol=1e-15)


def test_token_subset_matches_full_layer():
    cfg, inp, experts, shared = _tiny_layer(T=5)
    H, I, E, k, G = cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group
    full = moe.moe_layer(inp["x_bits"], inp["w_router"], None, experts, shared, H, I, E, k, G)
    sub = moe.moe_layer(inp["x_bits"], inp["w_router"], None, experts, shared, H, I, E, k, G, tokens=[1, 3])
    np.testing.assert_allclose(sub["y"][[1, 3]], full["y"][[1, 3]], rtol=1e-12, atol=1e-15)
    assert np.all(np.isnan(sub["y"][[0, 2, 4]]))
