"""qre_route_noalloc: the router for callers that cannot allocate device memory.

Such callers (code inside a framework that owns all device allocations, loops
that must not allocate while they run, callers that only hold the buffers they
were given) cannot pass a workspace.  The entry point keeps its scratch in a
fixed array inside the library; its results must equal qre_route's.  This file
is collected last so that a failure here leaves every other test already run.
"""

import numpy as np
import pytest
import torch

import synthetic
import quantized_routed_expert_03_gb300 as qre

from gpu_support import bits_to_bf16_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _inputs(T, H, E, step, bias):
    x = bits_to_bf16_tensor(synthetic.activations_bits(T, H, seed=4, layer=0, step=step), DEV)
    wr = torch.from_numpy(synthetic.router_weights(E, H, seed=4)).to(DEV)
    b = torch.from_numpy(synthetic.zipf_bias(E, seed=4, beta=0.05)).to(DEV) if bias else None
    return x, wr, b


@pytest.mark.parametrize("H,E,k,T,bias", [(4096, 288, 8, 8, False), (4096, 288, 8, 200, True),
                                          (256, 16, 4, 4, False)])
def test_noalloc_route_equals_workspace_route_twice(H, E, k, T, bias):
    shape = qre.make_shape(H, 128, E, k, 32)
    ws = torch.empty(max(qre.qre_workspace_size(shape, T), 256), dtype=torch.uint8, device=DEV)
    for step in range(2):                       # two calls in a row share the fixed scratch
        x, wr, b = _inputs(T, H, E, step, bias)
        idx_a = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
        w_a = torch.full((T, k), -1.0, dtype=torch.float32, device=DEV)
        idx_b, w_b = idx_a.clone(), w_a.clone()
        qre.qre_route(shape, T, x, wr, b, idx_a, w_a, ws)
        qre.qre_route_noalloc(shape, T, x, wr, b, idx_b, w_b)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(idx_b.cpu().numpy(), idx_a.cpu().numpy())
        np.testing.assert_array_equal(w_b.cpu().numpy(), w_a.cpu().numpy())


def test_noalloc_route_rejects_sizes_beyond_its_scratch():
    shape = qre.make_shape(4096, 2048, 288, 8, 128)
    T = 65536 // 288 + 1
    with pytest.raises(qre.QreError) as ei:
        qre.qre_route_noalloc(shape, T, 16, 16, None, 16, 16)
    assert ei.value.status == qre.QRE_ERR_UNSUPPORTED
    assert "fixed scratch" in str(ei.value)
