"""Seeded synthetic inputs for the routed MoE layer.

This module only draws inputs.  It holds none of the layer's arithmetic (no
routing, quantization or FFN); both the GPU library's tests/benchmark and the
CPU oracle receive the arrays it produces.

Distributions (the pages publish no data; these stand in for the serving traffic
the GLM-5.3-Flash recipes measure):
  * activations: z ~ N(0, 1) fp32 per token, divided by its RMS, rounded to bf16
    (round-to-nearest-even);
  * router weights and expert weights (gate, up, down): N(0, 0.02) fp32;
  * skewed routing: a per-layer selection bias b_e = -1.1 * beta * ln(r_e), r_e a
    seeded random popularity rank in 1..E, with beta calibrated once so that pick
    frequencies follow Zipf(1.1) (stored in ``tests/golden/zipf_beta.json``);
  * expert-cache placement: popularity ranks 1..40 are static HBM slots, 41..188
    HBM cache slots, the remaining 100 live in pinned host memory (GLM-5.3-Flash
    EXL3 3.05bpw on 1x RTX PRO 6000 recipe, ``config.expert_cache.layout``).

Every stream is keyed by (seed, layer, expert, tensor) through numpy's
``SeedSequence`` so that any single tensor can be regenerated on its own.  Large
configurations draw expert weights on the GPU with a torch generator keyed the
same way (``expert_fp32_torch``); a test that needs those weights on the CPU copies
the generated tensor back.
"""

from __future__ import annotations

import json
import os
from dataclasses import dataclass, field

import numpy as np

WEIGHT_STD = 0.02
ZIPF_S = 1.1
_T_ACT, _T_ROUTER, _T_GATE, _T_UP, _T_DOWN, _T_RANK = range(6)
_HERE = os.path.dirname(os.path.abspath(__file__))
ZIPF_BETA_FILE = os.path.join(_HERE, "tests", "golden", "zipf_beta.json")


@dataclass(frozen=True)
class LayerConfig:
    """Shape and workload of one synthetic MoE configuration."""
    name: str
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    group: int
    tokens: int
    layers: int = 1
    zipf: bool = False
    host_tier: bool = False          # popularity ranks > hbm_slots live in host memory
    hbm_slots: int = 188
    static_slots: int = 40
    live_cache: bool = False         # the HBM slots past the static ones are a live LFU cache
    seed: int = 0
    note: str = field(default="", compare=False)


CONFIGS = {
    "tiny": LayerConfig("tiny", 256, 128, 16, 4, 32, 4,
                        note="H256 I128 E16 k4 +1 shared, T4, G32, all HBM, seed 0"),
    "decode1": LayerConfig("decode1", 4096, 2048, 288, 8, 128, 1,
                           note="one full-size decode layer, T1, all 289 experts in HBM"),
    "decode8_zipf_x42": LayerConfig("decode8_zipf_x42", 4096, 2048, 288, 8, 128, 8, layers=42, zipf=True,
                                    note="T8, Zipf(1.1) routing bias, 42 independent layers, all in HBM"),
    "cache4_x42": LayerConfig("cache4_x42", 4096, 2048, 288, 8, 128, 4, layers=42, zipf=True, host_tier=True,
                              note="T4, Zipf(1.1), 42 layers; 188 HBM slots (40 static + 148 cache), "
                                   "100 experts per layer in pinned host memory read zero-copy"),
    "cache4_live_x16": LayerConfig("cache4_live_x16", 4096, 2048, 288, 8, 128, 4, layers=16, zipf=True,
                                   host_tier=True, live_cache=True,
                                   note="T4, Zipf(1.1), 16 layers; 40 static HBM experts + 148 HBM slots run as an "
                                        "LFU(0.995) cache (starting with ranks 41-188), misses copied from pinned "
                                        "host memory every step; the other experts read zero-copy until admitted"),
    "decode8_zipf_x1": LayerConfig("decode8_zipf_x1", 4096, 2048, 288, 8, 128, 8, layers=1, zipf=True,
                                   note="profiling case: one layer of decode8_zipf_x42 (3.7 GB of packed experts)"),
    "prefill2048_e64": LayerConfig("prefill2048_e64", 4096, 2048, 64, 8, 128, 2048,
                                   note="profiling case: the prefill8192 kernels on 64 experts and 2048 tokens "
                                        "(~256 tokens per expert, 0.84 GB of packed experts)"),
    "prefill8192": LayerConfig("prefill8192", 4096, 2048, 288, 8, 128, 8192,
                               note="T8192 prefill chunk, uniform routing, + shared expert"),
}


def _ss(seed: int, layer: int, expert: int, tensor: int) -> np.random.SeedSequence:
    return np.random.SeedSequence([int(seed), int(layer), int(expert) + 1, int(tensor)])


def _rng(seed, layer, expert, tensor) -> np.random.Generator:
    return np.random.default_rng(_ss(seed, layer, expert, tensor))


def torch_seed(seed: int, layer: int, expert: int, tensor: int) -> int:
    """63-bit seed for a torch generator, derived from the same key."""
    return int(_ss(seed, layer, expert, tensor).generate_state(1, np.uint64)[0] & ((1 << 63) - 1))


def f32_to_bf16_rne_bits(z: np.ndarray) -> np.ndarray:
    """Input preparation: fp32 -> bf16 bit patterns (round to nearest even)."""
    u = np.ascontiguousarray(z, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep = u >> 16
    rest = u & 0xFFFF
    up = (rest > 0x8000) | ((rest == 0x8000) & ((keep & 1) == 1))
    return ((keep + up) & 0xFFFF).astype(np.uint16)


def activations_bits(T: int, H: int, seed: int = 0, layer: int = 0, step: int = 0) -> np.ndarray:
    """bf16 activations [T,H] as uint16 bits: N(0,1) rows, RMS-normalised."""
    rng = np.random.default_rng(np.random.SeedSequence([int(seed), int(layer), 0, _T_ACT, int(step)]))
    z = rng.standard_normal((T, H), dtype=np.float32)
    rms = np.sqrt(np.mean(z.astype(np.float64) ** 2, axis=1, keepdims=True)).astype(np.float32)
    return f32_to_bf16_rne_bits(z / np.maximum(rms, np.float32(1e-30)))


def router_weights(E: int, H: int, seed: int = 0, layer: int = 0) -> np.ndarray:
    """Router weights W_r [E,H] fp32 ~ N(0, 0.02)."""
    return (_rng(seed, layer, -1, _T_ROUTER).standard_normal((E, H), dtype=np.float32)
            * np.float32(WEIGHT_STD))


def expert_fp32(H: int, I: int, seed: int = 0, layer: int = 0, expert: int = 0):
    """(W_gate [I,H], W_up [I,H], W_down [H,I]) fp32 ~ N(0, 0.02).  expert == E is the shared one."""
    out = []
    for tensor, shape in ((_T_GATE, (I, H)), (_T_UP, (I, H)), (_T_DOWN, (H, I))):
        out.append(_rng(seed, layer, expert, tensor).standard_normal(shape, dtype=np.float32)
                   * np.float32(WEIGHT_STD))
    return tuple(out)


def expert_fp32_torch(H: int, I: int, seed: int, layer: int, expert: int, device):
    """Same distributions as :func:`expert_fp32`, drawn by torch on ``device``.

    Used where the weights are too large to draw on the CPU.  The values differ
    from the numpy draw; whichever backend a run uses feeds both sides.
    """
    import torch
    out = []
    for tensor, shape in ((_T_GATE, (I, H)), (_T_UP, (I, H)), (_T_DOWN, (H, I))):
        g = torch.Generator(device=device)
        g.manual_seed(torch_seed(seed, layer, expert, tensor))
        out.append(torch.randn(shape, generator=g, device=device, dtype=torch.float32) * WEIGHT_STD)
    return tuple(out)


def popularity_ranks(E: int, seed: int = 0, layer: int = 0) -> np.ndarray:
    """A seeded random assignment of popularity ranks 1..E to experts 0..E-1."""
    return _rng(seed, layer, -1, _T_RANK).permutation(E).astype(np.int64) + 1


def zipf_beta() -> float:
    with open(ZIPF_BETA_FILE) as f:
        return float(json.load(f)["beta"])


def zipf_bias(E: int, seed: int = 0, layer: int = 0, beta: float | None = None) -> np.ndarray:
    """Selection bias b_e = -s * beta * ln(rank_e), fp32 [E]."""
    if beta is None:
        beta = zipf_beta()
    r = popularity_ranks(E, seed, layer).astype(np.float64)
    return (-ZIPF_S * beta * np.log(r)).astype(np.float32)


def host_resident(cfg: LayerConfig, layer: int) -> np.ndarray:
    """Boolean [E]: True where the expert lives in pinned host memory."""
    if not cfg.host_tier:
        return np.zeros(cfg.n_experts, dtype=bool)
    return popularity_ranks(cfg.n_experts, cfg.seed, layer) > cfg.hbm_slots


def layer_inputs_small(cfg: LayerConfig, layer: int = 0, step: int = 0, T: int | None = None) -> dict:
    """All fp32/bf16 inputs of one layer drawn on the CPU (small shapes only)."""
    T = cfg.tokens if T is None else T
    E, H, I = cfg.n_experts, cfg.hidden, cfg.inter
    experts = [expert_fp32(H, I, cfg.seed, layer, e) for e in range(E + 1)]
    return {
        "x_bits": activations_bits(T, H, cfg.seed, layer, step),
        "w_router": router_weights(E, H, cfg.seed, layer),
        "bias": zipf_bias(E, cfg.seed, layer) if cfg.zipf else None,
        "experts_fp32": experts[:E],
        "shared_fp32": experts[E],
    }
