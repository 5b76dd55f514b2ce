"""Shared set-up for the GPU parity tests and the benchmark's correctness checks.

Inputs come from ``synthetic`` only.  The GPU side quantizes fp32 weights with
the library's own kernels; the oracle side quantizes the same fp32 weights with
``oracle.quant``; the packed bytes of the two are compared bit for bit.
"""

from __future__ import annotations

import numpy as np
import torch

import synthetic
import quantized_routed_expert_03_gb300 as qre
from quantized_routed_expert_03_gb300.layer import ExpertArena, MoELayer
from oracle import moe as omoe
from oracle import quant as oquant


def bits_to_bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_tensor_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


class LazyOracleExperts:
    """Oracle-quantized experts produced on demand from a fp32 source function."""

    def __init__(self, source, G):
        self.source, self.G, self.cache = source, G, {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            wg, wu, wd = self.source(e)
            self.cache[e] = oquant.quantize_expert(wg, wu, wd, self.G)
        return self.cache[e]


class BuiltLayer:
    """One layer's weights on the device (arenas + slot table) and its oracle twin."""

    def __init__(self, H, I, E, k, G, t_max, device, fp32_source, host_mask=None, arena_order=None,
                 device_source=None):
        self.H, self.I, self.E, self.k, self.G = H, I, E, k, G
        self.device = device
        self.fp32_source = fp32_source            # e -> (wg, wu, wd) numpy fp32 (for the oracle)
        self.device_source = device_source        # e -> the same weights as device tensors (optional)
        self.layer = MoELayer(H, I, E, k, G, t_max, device=device)
        host_mask = np.zeros(E + 1, dtype=bool) if host_mask is None else np.asarray(host_mask)
        order = np.arange(E + 1) if arena_order is None else np.asarray(arena_order)
        n_host = int(host_mask.sum())
        self.dev_arena = ExpertArena(H, I, G, E + 1 - n_host, device=device)
        self.host_arena = ExpertArena(H, I, G, max(n_host, 1), host=True) if n_host else None
        staging = torch.empty(self.dev_arena.layout["stride"], dtype=torch.uint8, device=device)
        entries = [None] * (E + 1)
        di = hi = 0
        self.where = {}
        for e in order:
            wg, wu, wd = self.device_fp32(int(e))
            if host_mask[e]:
                self.host_arena.quantize_into(hi, wg, wu, wd, staging=staging)
                entries[e] = self.host_arena.addresses(hi) + (1,)
                self.where[int(e)] = ("host", hi)
                hi += 1
            else:
                self.dev_arena.quantize_into(di, wg, wu, wd)
                entries[e] = self.dev_arena.addresses(di) + (0,)
                self.where[int(e)] = ("dev", di)
                di += 1
        torch.cuda.synchronize()
        self.layer.set_slots(entries)
        self.oracle_experts = LazyOracleExperts(self.fp32_source, G)

    def device_fp32(self, e):
        if self.device_source is not None:
            return self.device_source(e)
        wg, wu, wd = self.fp32_source(e)
        return tuple(torch.from_numpy(np.ascontiguousarray(a)).to(self.device) for a in (wg, wu, wd))

    def packed_numpy(self, e) -> dict:
        kind, i = self.where[int(e)]
        arena = self.dev_arena if kind == "dev" else self.host_arena
        return arena.to_numpy(i)

    def oracle_layer(self, x_bits, w_router, bias, tokens=None):
        E = self.E
        experts = _ExpertsView(self.oracle_experts, E)
        return omoe.moe_layer(x_bits, w_router, bias, experts, self.oracle_experts[E], self.H, self.I, E, self.k,
                              self.G, tokens=tokens)


class _ExpertsView:
    def __init__(self, lazy, E):
        self.lazy, self.E = lazy, E

    def __getitem__(self, e):
        if not 0 <= int(e) < self.E:
            raise IndexError(e)
        return self.lazy[e]


def numpy_source(cfg, layer=0):
    """fp32 weights from the numpy generator (small shapes)."""
    H, I = cfg.hidden, cfg.inter

    def src(e):
        return synthetic.expert_fp32(H, I, cfg.seed, layer, e)
    return src


def torch_sources(cfg, layer, device):
    """(host, device) sources of fp32 weights drawn by the torch generator on the device.

    The device source feeds the library's quantizer; the host source copies the
    same draw back for the oracle.
    """
    H, I = cfg.hidden, cfg.inter

    def dev(e):
        return synthetic.expert_fp32_torch(H, I, cfg.seed, layer, e, device)

    def host(e):
        return tuple(t.cpu().numpy() for t in dev(e))
    return host, dev


def rel_rms(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_routing(gpu_idx, gpu_w, ref, gap_tol=2e-6, w_tol=2e-6):
    """Routing indices bit-exact except where the oracle's k/k+1 margin is below gap_tol.

    For such near-tie tokens the GPU's selection must still be a valid top-k of
    the oracle's selection scores within gap_tol.  Returns the number of near-tie
    tokens.
    """
    gpu_idx = np.asarray(gpu_idx)
    T, k = gpu_idx.shape
    near = np.nonzero(ref["gap"] < gap_tol)[0]
    exact = np.setdiff1d(np.arange(T), near)
    np.testing.assert_array_equal(gpu_idx[exact], ref["idx"][exact])
    np.testing.assert_allclose(np.asarray(gpu_w)[exact], ref["w"][exact], rtol=0, atol=w_tol)
    for t in near:
        sel = ref["sel"][t]
        chosen = set(int(e) for e in gpu_idx[t])
        assert len(chosen) == k and np.all(np.diff(gpu_idx[t]) > 0)
        others = [e for e in range(sel.size) if e not in chosen]
        assert min(sel[list(chosen)]) >= max(sel[others]) - gap_tol
    return int(near.size)
