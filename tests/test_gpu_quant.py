"""GPU quantizer vs the oracle's format definition: packed bytes and scales bit-exact."""

import numpy as np
import pytest
import torch

import quantized_routed_expert_03_gb300 as qre
from quantized_routed_expert_03_gb300.layer import packed_rows, scale_rows
from oracle import quant as oquant

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _gpu_quantize(W, G):
    """Quantizes on the device; returns packed bytes and scales row-major."""
    N, K = W.shape
    w = torch.from_numpy(np.ascontiguousarray(W)).to(DEV)
    packed = torch.empty(N * K // 2, dtype=torch.uint8, device=DEV)
    scales = torch.empty(N * K // G, dtype=torch.int16, device=DEV)
    qre.qre_quantize(N, K, G, w, packed, scales)
    torch.cuda.synchronize()
    return packed_rows(packed.cpu().numpy(), N, K), scale_rows(scales.cpu().numpy(), N, K, G)


@pytest.mark.parametrize("G", [32, 64, 128])
def test_quantize_bit_exact_gaussian(G):
    rng = np.random.default_rng(G)
    W = (rng.standard_normal((256, 1024)) * 0.02).astype(np.float32)
    p, s = _gpu_quantize(W, G)
    po, so = oquant.quantize_matrix(W, G)
    np.testing.assert_array_equal(p, po)
    np.testing.assert_array_equal(s.view(np.uint16), so.view(np.uint16))


def test_quantize_special_values_bit_exact():
    """Zero groups, exact half-way codes, subnormal fp16 scales, mixed magnitudes."""
    rng = np.random.default_rng(11)
    N, K, G = 128, 256, 32
    q = rng.integers(-7, 8, size=(N, K))
    s = 2.0 ** rng.integers(-20, 4, size=(N, K // G))
    W = (q.reshape(N, K // G, G) * s[:, :, None]).reshape(N, K)
    W[:, ::G] = 7 * np.repeat(s, 1, axis=1)                # max |q| = 7 in every group
    W[3::7, 5::11] += 0.5 * np.repeat(s, G, axis=1)[3::7, 5::11]   # exact .5 ties
    W[5] = 0.0                                             # a zero row
    W[6, :G] = -0.0
    W[7] = rng.standard_normal(K) * 1e-6                   # scales among the fp16 subnormals
    W[9] = rng.standard_normal(K) * 1e-9                   # scales that round to zero
    W[8] = rng.standard_normal(K) * 1e3
    W = W.astype(np.float32)
    p, sc = _gpu_quantize(W, G)
    po, so = oquant.quantize_matrix(W, G)
    np.testing.assert_array_equal(p, po)
    np.testing.assert_array_equal(sc.view(np.uint16), so.view(np.uint16))


def test_quantize_gate_up_interleave_bit_exact():
    rng = np.random.default_rng(12)
    I, H, G = 128, 512, 128
    Wg = (rng.standard_normal((I, H)) * 0.02).astype(np.float32)
    Wu = (rng.standard_normal((I, H)) * 0.02).astype(np.float32)
    wg, wu = (torch.from_numpy(a).to(DEV) for a in (Wg, Wu))
    packed = torch.empty(2 * I * H // 2, dtype=torch.uint8, device=DEV)
    scales = torch.empty(2 * I * H // G, dtype=torch.int16, device=DEV)
    qre.qre_quantize_gate_up(I, H, G, wg, wu, packed, scales)
    torch.cuda.synchronize()
    ex = oquant.quantize_expert(Wg, Wu, np.zeros((H, I), np.float32), G)
    np.testing.assert_array_equal(packed_rows(packed.cpu().numpy(), 2 * I, H), ex["w_gate_up"])
    np.testing.assert_array_equal(scale_rows(scales.cpu().numpy(), 2 * I, H, G).view(np.uint16),
                                  ex["s_gate_up"].view(np.uint16))


def test_quantize_non_finite_sets_status():
    qre.qre_clear_device_status()
    W = np.zeros((128, 64), dtype=np.float32)
    W[1, 40] = np.inf
    _gpu_quantize(W, 32)
    st = qre.qre_read_device_status()
    qre.qre_clear_device_status()
    assert st & qre.QRE_DEV_BAD_SCALE
    with pytest.raises(ValueError):
        oquant.quantize_matrix(W[:2], 32)
