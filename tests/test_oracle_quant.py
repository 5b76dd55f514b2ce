"""Pins for the oracle's packed 4-bit group format (CPU only).

Each test checks the oracle against something other than itself: a hand-derived
fixture, a closed form, an exactly representable round trip, or a per-element
reimplementation with Python integers.
"""

import json
import os

import numpy as np
import pytest

from oracle import quant

from conftest import GOLDEN


def _fixture():
    with open(os.path.join(GOLDEN, "quant_tiny.json")) as f:
        return json.load(f)


def test_hand_derived_example_bytes_and_scales():
    fx = _fixture()
    W = np.array(fx["w"], dtype=np.float32)
    packed, scales = quant.quantize_matrix(W, fx["group"])
    want_bytes = np.array([[int(h, 16) for h in row] for row in fx["packed_hex"]], dtype=np.uint8)
    want_scales = np.array([[int(h, 16) for h in row] for row in fx["scale_bits_hex"]], dtype=np.uint16)
    np.testing.assert_array_equal(packed, want_bytes)
    np.testing.assert_array_equal(scales.view(np.uint16), want_scales)


def test_hand_derived_example_dequant():
    fx = _fixture()
    K = len(fx["w"][0])
    packed = np.array([[int(h, 16) for h in row] for row in fx["packed_hex"]], dtype=np.uint8)
    scales = np.array([[int(h, 16) for h in row] for row in fx["scale_bits_hex"]], dtype=np.uint16).view(np.float16)
    got = quant.dequantize_matrix(packed, scales, K, fx["group"])
    np.testing.assert_array_equal(got, np.array(fx["dequant"]))


def test_exactly_representable_weights_round_trip():
    """Weights q*s with s an fp16 power-of-two scale and max|q| = 7 come back exactly."""
    rng = np.random.default_rng(1)
    N, K, G = 6, 64, 32
    q = rng.integers(-7, 8, size=(N, K))
    q[:, 0::G] = 7                                   # force max|q| = 7 in every group
    s = 2.0 ** rng.integers(-12, 2, size=(N, K // G))
    W = (q.reshape(N, K // G, G) * s[:, :, None]).reshape(N, K).astype(np.float32)
    packed, scales = quant.quantize_matrix(W, G)
    np.testing.assert_array_equal(scales.astype(np.float64), s)
    np.testing.assert_array_equal(quant.dequantize_matrix(packed, scales, K, G), W.astype(np.float64))
    # nibble value is q + 8, read back with Python integer arithmetic
    for n in range(N):
        for k in range(K):
            byte = int(packed[n, k // 2])
            u = (byte >> 4) if (k % 2) else (byte & 15)
            assert u - 8 == q[n, k]


def test_zero_group_gives_zero_scale_and_code_8():
    W = np.zeros((2, 64), dtype=np.float32)
    W[1, 32:] = np.linspace(-1, 1, 32, dtype=np.float32)
    packed, scales = quant.quantize_matrix(W, 32)
    assert scales[0, 0] == 0 and scales[0, 1] == 0 and scales[1, 0] == 0
    assert np.all(packed[0] == 0x88) and np.all(packed[1, :16] == 0x88)


def test_scale_is_rne_of_fp64_quotient():
    rng = np.random.default_rng(2)
    W = (rng.standard_normal((32, 256)) * 0.02).astype(np.float32)
    _, scales = quant.quantize_matrix(W, 128)
    amax = np.abs(W.astype(np.float64)).reshape(32, 2, 128).max(axis=2)
    exact = amax / 7.0
    s = scales.astype(np.float64)
    # correct rounding: no fp16 value lies strictly closer to the exact quotient
    up = np.nextafter(scales, np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(scales, np.float16(-np.inf)).astype(np.float64)
    assert np.all(np.abs(s - exact) <= np.abs(up - exact))
    assert np.all(np.abs(s - exact) <= np.abs(dn - exact))


def test_error_bound_and_code_range_on_gaussian_weights():
    rng = np.random.default_rng(3)
    N, K, G = 64, 512, 128
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    q, scales = quant.quantize_codes(W, G)
    s = np.repeat(scales.astype(np.float64), G, axis=1)
    What = q.astype(np.float64) * s
    # round-to-nearest on an unclipped code: error at most half a step
    assert np.all(np.abs(W.astype(np.float64) - What) <= 0.5 * s * (1 + 1e-12))
    assert q.min() >= -8 and q.max() <= 7
    # the element of largest magnitude maps to +-7 in every group
    Wg = np.abs(W).reshape(N, K // G, G)
    qg = np.abs(q.astype(np.int64)).reshape(N, K // G, G)
    am = Wg.argmax(axis=2)
    assert np.all(np.take_along_axis(qg, am[:, :, None], axis=2) == 7)


def test_non_finite_scale_rejected():
    W = np.zeros((1, 32), dtype=np.float32)
    W[0, 3] = np.inf
    with pytest.raises(ValueError):
        quant.quantize_matrix(W, 32)
    W[0, 3] = 7.0 * 70000.0
    with pytest.raises(ValueError):
        quant.quantize_matrix(W, 32)


def test_interleave_row_order_by_hand():
    I = 32
    gate = np.arange(I)[:, None] * np.ones((1, 3))
    up = 100 + np.arange(I)[:, None] * np.ones((1, 3))
    comb = quant.interleave_rows(gate, up)
    want = list(range(0, 16)) + [100 + i for i in range(16)] + list(range(16, 32)) + [100 + i for i in range(16, 32)]
    np.testing.assert_array_equal(comb[:, 0], want)
    g2, u2 = quant.deinterleave_rows(comb)
    np.testing.assert_array_equal(g2, gate)
    np.testing.assert_array_equal(u2, up)


def test_expert_round_trip_matches_per_matrix_quantization():
    rng = np.random.default_rng(4)
    H, I, G = 64, 32, 32
    Wg = (rng.standard_normal((I, H)) * 0.02).astype(np.float32)
    Wu = (rng.standard_normal((I, H)) * 0.02).astype(np.float32)
    Wd = (rng.standard_normal((H, I)) * 0.02).astype(np.float32)
    ex = quant.quantize_expert(Wg, Wu, Wd, G)
    assert ex["w_gate_up"].shape == (2 * I, H // 2) and ex["s_gate_up"].shape == (2 * I, H // G)
    g, u, d = quant.dequantize_expert(ex, H, I, G)
    for W, got in ((Wg, g), (Wu, u), (Wd, d)):
        p, s = quant.quantize_matrix(W, G)
        np.testing.assert_array_equal(got, quant.dequantize_matrix(p, s, W.shape[1], G))
        assert np.max(np.abs(got - W)) < 0.02
