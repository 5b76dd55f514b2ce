"""qre_combine against the oracle's combine: y_t = sum_j w[t,j] expert_out[inv_perm[t*k+j]]
+ expert_out[T*k + t] (fp32 FMAs in ascending pick order vs fp64), and a pick whose
row index is out of range (what a dispatch that met a bad expert id leaves
behind) contributes nothing instead of being read."""

import numpy as np
import pytest
import torch

import quantized_routed_expert_03_gb300 as qre
from oracle import moe as omoe

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _combine(T, H, k, seed, bad=()):
    rng = np.random.default_rng(seed)
    P = T * k
    eo = rng.standard_normal((P + T, H)).astype(np.float32)
    w = rng.random((T, k)).astype(np.float32)
    w /= w.sum(1, keepdims=True)
    inv = rng.permutation(P).astype(np.int32)
    for i, v in bad:
        inv[i] = v
    shape = qre.make_shape(H, 128, max(k, 16), k, 32)
    y = torch.full((T, H), float("nan"), device=DEV)
    yb = torch.zeros((T, H), dtype=torch.int16, device=DEV)
    qre.qre_combine(shape, T, torch.from_numpy(eo).to(DEV), torch.from_numpy(w).to(DEV),
                    torch.from_numpy(inv).to(DEV), y, yb)
    torch.cuda.synchronize()
    keep = (inv >= 0) & (inv < P)
    w_ref = np.where(keep.reshape(T, k), w, 0.0)
    ref = omoe.combine(eo, w_ref, np.where(keep, inv, 0), T, k)
    return y.cpu().numpy(), yb.cpu().numpy().view(np.uint16), ref


@pytest.mark.parametrize("T,H,k", [(1, 4096, 8), (8, 4096, 8), (13, 640, 8), (5, 512, 16), (300, 256, 6)])
def test_combine_matches_oracle(T, H, k):
    y, yb, ref = _combine(T, H, k, seed=T * 7 + k)
    err = np.abs(y - ref).max() / np.abs(ref).max()
    assert err < 1e-6, err
    np.testing.assert_array_equal(yb, omoe.f32_to_bf16_bits(y))


@pytest.mark.parametrize("T,H,k", [(1, 512, 8), (6, 512, 8), (5, 512, 16)])
def test_combine_skips_out_of_range_rows(T, H, k):
    P = T * k
    bad = [(0, -1), (P - 1, P + 5), (P // 2, 1 << 30)]
    y, _, ref = _combine(T, H, k, seed=11, bad=bad)
    assert np.isfinite(y).all()
    err = np.abs(y - ref).max() / np.abs(ref).max()
    assert err < 1e-6, err
