"""Prefill staging: each layer's host-resident experts are copied into an HBM
staging area one layer ahead on a copy stream (qre_stage_experts), and the
layer's expert FFN reads the staged copies through a staged slot table (the
RTX PRO 6000 recipe, config.expert_cache.mechanism; the glm53-flash-offload
README, "Prefill staging").  Every layer's output must equal, bit for bit, the
same layer with all experts in device memory."""

import ctypes

import numpy as np
import pytest
import torch

import synthetic
import quantized_routed_expert_03_gb300 as qre
from quantized_routed_expert_03_gb300.layer import StagingArea, staged_prefill

from gpu_support import BuiltLayer, bits_to_bf16_tensor, numpy_source

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MID = synthetic.LayerConfig("mid", 512, 256, 32, 4, 128, 8)


def _layers(cfg, T, n_layers, host):
    out = []
    for l in range(n_layers):
        src = numpy_source(cfg, layer=l)
        rng = np.random.default_rng(100 + l)
        mask = (rng.random(cfg.n_experts + 1) < 0.5) if host else None
        if host:
            mask[cfg.n_experts] = False
        out.append(BuiltLayer(cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group, T, DEV, src,
                              host_mask=mask))
    return out


def _inputs(cfg, T, n_layers):
    return [(bits_to_bf16_tensor(synthetic.activations_bits(T, cfg.hidden, cfg.seed, l, 5), DEV),
             torch.from_numpy(synthetic.router_weights(cfg.n_experts, cfg.hidden, cfg.seed, l)).to(DEV), None)
            for l in range(n_layers)]


def _staged_table(area, E):
    raw = area.table.cpu().numpy().tobytes()
    arr = (qre.qre_slot * (E + 1)).from_buffer_copy(raw)
    return [(arr[e].w_gate_up, arr[e].tier) for e in range(E + 1)]


@pytest.mark.parametrize("T,n_slots", [(40, 32), (300, 32), (300, 3)], ids=["T40", "T300", "T300_3slots"])
def test_staged_prefill_is_bit_identical_to_hbm(T, n_slots):
    """Two staging areas alternate over three layers; with 3 slots only the first
    three host experts of a layer are staged and the rest are read zero-copy."""
    cfg, n_layers = MID, 3
    hbm = _layers(cfg, T, n_layers, host=False)
    host = _layers(cfg, T, n_layers, host=True)
    inputs = _inputs(cfg, T, n_layers)
    ref = []
    for b, (x, wr, bias) in zip(hbm, inputs):
        b.layer.forward(x, wr, bias, T)
        ref.append(b.layer.y[:T].clone())
    areas = [StagingArea(cfg.hidden, cfg.inter, cfg.group, cfg.n_experts, n_slots, DEV) for _ in range(2)]
    copy_stream = torch.cuda.Stream(DEV)
    staged_prefill([b.layer for b in host], inputs, areas, copy_stream, T)
    torch.cuda.synchronize()
    for l in range(n_layers):
        assert torch.equal(host[l].layer.y[:T], ref[l]), f"layer {l}"
    # the last layer's table: its first min(n_slots, #host) host experts point into its area, tier 0
    last = host[-1]
    area = areas[(n_layers - 1) % 2]
    hosted = [e for e in range(cfg.n_experts + 1) if last.where[e][0] == "host"]
    table = _staged_table(area, cfg.n_experts)
    for j, e in enumerate(hosted):
        if j < n_slots:
            assert table[e] == (area.arena.addresses(j)[0], 0)
        else:
            assert table[e][1] == 1
    assert area.n_staged == min(n_slots, len(hosted))
    for j, e in enumerate(hosted[:n_slots]):      # the staged bytes are the expert's bytes
        for name in ("w_gate_up", "s_gate_up", "w_down", "s_down"):
            assert torch.equal(area.arena.view(j, name).cpu(), last.host_arena.view(last.where[e][1], name).cpu())
    assert qre.qre_read_device_status() == 0


def test_staged_prefill_in_a_cuda_graph():
    cfg, T, n_layers = MID, 40, 2
    hbm = _layers(cfg, T, n_layers, host=False)
    host = _layers(cfg, T, n_layers, host=True)
    inputs = _inputs(cfg, T, n_layers)
    ref = []
    for b, (x, wr, bias) in zip(hbm, inputs):
        b.layer.forward(x, wr, bias, T)
        ref.append(b.layer.y[:T].clone())
    areas = [StagingArea(cfg.hidden, cfg.inter, cfg.group, cfg.n_experts, 32, DEV) for _ in range(2)]
    main, copy_stream = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    with torch.cuda.stream(main):
        staged_prefill([b.layer for b in host], inputs, areas, copy_stream, T, stream=main)   # warm-up
    torch.cuda.synchronize()
    for b in host:
        b.layer.y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        staged_prefill([b.layer for b in host], inputs, areas, copy_stream, T, stream=main)
    g.replay()
    torch.cuda.synchronize()
    for l in range(n_layers):
        assert torch.equal(host[l].layer.y[:T], ref[l]), f"layer {l}"
