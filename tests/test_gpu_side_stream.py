"""The shared expert on a side stream (qre_expert_ffn_shared) beside the router,
the dispatch and the routed experts (qre_expert_ffn_routed): the same bits as
one qre_expert_ffn call, eagerly and inside a captured CUDA graph, and the
oracle's result within the path's tolerance.  The glm53-flash-offload README's
side-stream shared expert ("Decode kernels") changed its outputs (~2e-3 per
layer, "Quality"); here every expert row is computed by the same arithmetic
whichever launch computes it, and the combine order is fixed."""

import numpy as np
import pytest
import torch

import synthetic
import quantized_routed_expert_03_gb300 as qre

from gpu_support import BuiltLayer, bits_to_bf16_tensor, numpy_source
from test_gpu_layer import MID, ODD, PREFILL_TOL, _check_layer, _inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FP8 = synthetic.LayerConfig("fp8", 512, 512, 32, 4, 128, 8)


def _forward(built, x_bits, wr, side):
    L = built.layer
    T = x_bits.shape[0]
    x = bits_to_bf16_tensor(x_bits, DEV)
    w = torch.from_numpy(wr).to(DEV)
    L.expert_out.fill_(float("nan"))
    L.forward(x, w, None, T, shared_stream=side)
    torch.cuda.synchronize()
    P = T * built.k
    return {"expert_out": L.expert_out[:P + T].cpu().numpy(), "y": L.y[:T].cpu().numpy(),
            "idx": L.topk_idx[:T].cpu().numpy(), "w": L.topk_w[:T].cpu().numpy(),
            "counts": L.counts.cpu().numpy(), "offsets": L.offsets.cpu().numpy(),
            "perm": L.perm[:P].cpu().numpy(), "inv_perm": L.inv_perm[:P].cpu().numpy(),
            "n_active": int(L.n_active[0].item()), "active": L.active.cpu().numpy(),
            "y_bf16": L.y_bf16[:T].view(torch.int16).cpu().numpy().view(np.uint16)}


@pytest.mark.parametrize("cfg,T,tol", [(FP8, 1, 1e-5), (FP8, 8, 1e-5), (MID, 5, 1e-5), (ODD, 8, 1e-5),
                                       (MID, 40, PREFILL_TOL), (ODD, 130, PREFILL_TOL)],
                         ids=["fp8_T1", "fp8_T8", "mid_T5", "odd_G64_T8", "prefill_T40", "prefill_odd_T130"])
def test_side_stream_shared_expert_is_bit_identical(cfg, T, tol):
    built = BuiltLayer(cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group, T, DEV, numpy_source(cfg))
    x_bits, wr, _ = _inputs(cfg, T, step=31)
    one = _forward(built, x_bits, wr, None)
    two = _forward(built, x_bits, wr, torch.cuda.Stream(DEV))
    np.testing.assert_array_equal(two["expert_out"], one["expert_out"])
    np.testing.assert_array_equal(two["y"], one["y"])
    _check_layer(built, two, built.oracle_layer(x_bits, wr, None), tol=tol)
    assert qre.qre_read_device_status() == 0


@pytest.mark.parametrize("cfg,T", [(FP8, 1), (MID, 40)], ids=["decode", "prefill"])
def test_side_stream_in_a_cuda_graph(cfg, T):
    """Fork and join captured in a graph; replays give the fused path's bits."""
    built = BuiltLayer(cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group, T, DEV, numpy_source(cfg))
    L = built.layer
    wr = torch.from_numpy(synthetic.router_weights(cfg.n_experts, cfg.hidden, cfg.seed, 0)).to(DEV)
    xs = [bits_to_bf16_tensor(synthetic.activations_bits(T, cfg.hidden, cfg.seed, 0, 40 + i), DEV) for i in range(3)]
    x_in = torch.empty_like(xs[0])
    ref = []
    for x in xs:
        L.forward(x, wr, None, T)
        ref.append(L.y[:T].clone())
    main, side = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    with torch.cuda.stream(main):
        x_in.copy_(xs[0])
        L.forward(x_in, wr, None, T, shared_stream=side)   # eager warm-up (workspace, events)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        L.forward(x_in, wr, None, T, stream=main, shared_stream=side)
    for i, x in enumerate(xs):
        x_in.copy_(x)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(L.y[:T], ref[i]), f"replay {i}"
