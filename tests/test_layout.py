"""The host helpers that read the library's tiled weight storage back into
row-major arrays agree with the storage formula stated for qre_slot (no GPU)."""

import numpy as np

from quantized_routed_expert_03_gb300.layer import packed_rows, scale_rows


def _tiled_packed_by_formula(P):
    """Places row-major packed bytes P [N][K/2] at the byte offsets the format
    states, one byte at a time."""
    N, K = P.shape[0], 2 * P.shape[1]
    raw = np.full(N * K // 2, 0xEE, np.uint8)
    for n in range(N):
        for k in range(0, K, 2):
            off = ((n // 128) * (K // 64) + k // 64) * 4096 + 2048 * ((k % 64) // 32) + 16 * (n % 128) + (k % 32) // 2
            raw[off] = P[n, k // 2]
    return raw


def test_packed_rows_inverts_the_stated_tiling():
    rng = np.random.default_rng(0)
    N, K = 256, 192
    P = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    raw = _tiled_packed_by_formula(P)
    assert not (raw == 0xEE).all()
    np.testing.assert_array_equal(packed_rows(raw, N, K), P)


def test_warp_slice_is_contiguous():
    """32 rows of one 32-column slice occupy 512 consecutive bytes."""
    N, K = 128, 128
    P = np.arange(N * K // 2, dtype=np.int64).reshape(N, K // 2)
    raw = _tiled_packed_by_formula((P % 251).astype(np.uint8))
    offs = []
    for n in range(32, 64):
        for b in range(16, 32):          # bytes of columns 32..63 (second half of stage 0)
            offs.append(((n // 128) * (K // 64)) * 4096 + 2048 + 16 * (n % 128) + (b - 16))
    offs = np.array(offs)
    assert offs.max() - offs.min() == 511 and len(set(offs.tolist())) == 512


def test_scale_rows_inverts_the_stated_tiling():
    rng = np.random.default_rng(1)
    N, K, G = 256, 512, 64
    S = rng.standard_normal((N, K // G)).astype(np.float16)
    raw = np.zeros(N * K // G, np.float16)
    for n in range(N):
        for g in range(K // G):
            raw[((n // 128) * (K // G) + g) * 128 + n % 128] = S[n, g]
    np.testing.assert_array_equal(scale_rows(raw.view(np.uint16), N, K, G).view(np.uint16), S.view(np.uint16))
