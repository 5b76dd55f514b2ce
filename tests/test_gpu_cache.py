"""Device-side LFU expert cache (qre_cache_update / qre_cache_copy) vs the
policy-replay oracle, and a decode loop with the live cache vs all-HBM experts."""

import ctypes

import numpy as np
import pytest
import torch

import synthetic
import quantized_routed_expert_03_gb300 as qre
from quantized_routed_expert_03_gb300.layer import ExpertArena, MoELayer
from oracle import cache as ocache

from gpu_support import bits_to_bf16_tensor, numpy_source

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SLOT = ctypes.sizeof(qre.qre_slot)


def _slot_tensor(entries):
    arr = qre.slot_array(entries)
    raw = bytearray(memoryview(arr).cast("B"))
    return torch.frombuffer(raw, dtype=torch.uint8).to(DEV)


def _slots_from_tensor(t, n):
    raw = t.cpu().numpy().tobytes()
    arr = (qre.qre_slot * n).from_buffer_copy(raw)
    return [(arr[i].w_gate_up, arr[i].tier) for i in range(n)]


def _zipf_trace(n_calls, T, E, k, ranks, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    by_rank = np.argsort(ranks)            # expert of rank r+1
    trace = []
    for _ in range(n_calls):
        picks = set()
        for _ in range(T):
            picks |= set(by_rank[rng.choice(E, size=k, replace=False, p=p)].tolist())
        trace.append(sorted(picks))
    return trace


@pytest.mark.parametrize("max_copies", [64, 2])
def test_cache_manager_matches_policy_replay(max_copies):
    """Admissions, copy list, slots, scores and the slot table equal the LFU
    replay call by call; with a copy list of 2 entries the calls with more
    misses admit two and leave the rest on the host tier."""
    E, k, S, n_static = 288, 8, 148, 40
    shape = qre.make_shape(4096, 2048, E, k, 128)
    ranks = synthetic.popularity_ranks(E, seed=0, layer=5)
    static = [e for e in range(E) if ranks[e] <= n_static]
    init_slots = [int(np.nonzero(ranks == n_static + 1 + s)[0][0]) for s in range(S)]
    trace = _zipf_trace(80, T=4, E=E, k=k, ranks=ranks, seed=3)

    fake = lambda base, i, tier: (base + i * 0x10000, base + i * 0x10000 + 0x1000, base + i * 0x10000 + 0x2000,
                                  base + i * 0x10000 + 0x3000, tier)
    home = [fake(0x10000000, e, 1) for e in range(E + 1)]
    slot_mem = [fake(0x90000000, s, 0) for s in range(S)]
    table0 = [fake(0x50000000, e, 0) if e in static or e == E else home[e] for e in range(E + 1)]
    for s, e in enumerate(init_slots):
        table0[e] = slot_mem[s]
    d_home, d_slot, d_table = _slot_tensor(home), _slot_tensor(slot_mem), _slot_tensor(table0)
    expert_slot = np.full(E, -1, np.int32)
    expert_slot[static] = -2
    for s, e in enumerate(init_slots):
        expert_slot[e] = s
    d_es = torch.from_numpy(expert_slot).to(DEV)
    d_se = torch.tensor(init_slots, dtype=torch.int32, device=DEV)
    d_scores = torch.zeros(E, dtype=torch.float32, device=DEV)
    d_list = torch.full((2 * max_copies,), -1, dtype=torch.int32, device=DEV)
    d_n = torch.zeros(4, dtype=torch.int32, device=DEV)
    d_active = torch.zeros(E, dtype=torch.int32, device=DEV)
    d_nact = torch.zeros(4, dtype=torch.int32, device=DEV)

    ref = ocache.lfu_replay(trace, E, static, S, decay=0.995, init_slots=init_slots, max_admit=max_copies)
    capped = sum(1 for adm, byp in zip(ref["admitted"], ref["bypassed"]) if len(adm) == max_copies and byp)
    if max_copies == 2:
        assert capped > 0, "the trace must exercise the admission cap"
    for call, adm in zip(trace, ref["admitted"]):
        d_active[:len(call)] = torch.tensor(call, dtype=torch.int32)
        d_nact[0] = len(call)
        qre.qre_cache_update(shape, S, 0.995, d_active, d_nact, d_scores, d_es, d_se, d_home, d_slot, d_table,
                             d_list, d_n, max_copies)
        torch.cuda.synchronize()
        n = int(d_n[0].item())
        got = [tuple(x) for x in d_list[:2 * n].cpu().numpy().reshape(-1, 2).tolist()]
        assert got == [(e, s) for e, s, _ in adm]
    np.testing.assert_array_equal(d_se.cpu().numpy(), ref["slot_expert"])
    np.testing.assert_array_equal(d_scores.cpu().numpy(), ref["scores"])
    es = d_es.cpu().numpy()
    for s, e in enumerate(ref["slot_expert"]):
        assert es[e] == s
    table = _slots_from_tensor(d_table, E + 1)
    for s, e in enumerate(ref["slot_expert"]):
        assert table[e] == (slot_mem[s][0], 0)
    for e in range(E):
        if e not in static and e not in ref["slot_expert"]:
            assert table[e] == (home[e][0], 1)
    assert ref["misses"] > 0


def _build_cached_layer(cfg, n_static, S, T):
    H, I, E, k, G = cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group
    src = numpy_source(cfg)
    ranks = synthetic.popularity_ranks(E, cfg.seed, 0)
    static = [e for e in range(E) if ranks[e] <= n_static] + [E]
    home = ExpertArena(H, I, G, E + 1, host=True)
    hbm_static = ExpertArena(H, I, G, E + 1, device=DEV)
    slots = ExpertArena(H, I, G, S, device=DEV)
    ref_arena = ExpertArena(H, I, G, E + 1, device=DEV)
    staging = torch.empty(home.layout["stride"], dtype=torch.uint8, device=DEV)
    for e in range(E + 1):
        w = [torch.from_numpy(a).to(DEV) for a in src(e)]
        home.quantize_into(e, *w, staging=staging)
        ref_arena.quantize_into(e, *w)
        if e in static:
            hbm_static.quantize_into(e, *w)
    torch.cuda.synchronize()
    home_entries = [home.addresses(e) + (1,) for e in range(E + 1)]
    slot_entries = [slots.addresses(s) + (0,) for s in range(S)]
    table = [hbm_static.addresses(e) + (0,) if e in static else home_entries[e] for e in range(E + 1)]
    live = MoELayer(H, I, E, k, G, T, device=DEV)
    live.set_slots(table)
    ref = MoELayer(H, I, E, k, G, T, device=DEV)
    ref.set_slots([ref_arena.addresses(e) + (0,) for e in range(E + 1)])
    expert_slot = np.full(E, -1, np.int32)
    expert_slot[[e for e in static if e < E]] = -2
    state = {
        "home": _slot_tensor(home_entries), "slot_mem": _slot_tensor(slot_entries),
        "scores": torch.zeros(E, dtype=torch.float32, device=DEV),
        "expert_slot": torch.from_numpy(expert_slot).to(DEV),
        "slot_expert": torch.full((S,), -1, dtype=torch.int32, device=DEV),
        "copy_list": torch.zeros(2 * 64, dtype=torch.int32, device=DEV),
        "n_copies": torch.zeros(4, dtype=torch.int32, device=DEV),
        "keep": (home, hbm_static, slots, ref_arena),
    }
    return live, ref, state, slots


def test_cache_copy_moves_the_admitted_experts():
    cfg = synthetic.LayerConfig("mid", 512, 256, 32, 4, 128, 4)
    live, ref, st, slots = _build_cached_layer(cfg, n_static=4, S=6, T=4)
    shape = live.shape
    E = cfg.n_experts
    active = torch.tensor([e for e in range(E) if st["expert_slot"][e].item() == -1][:5], dtype=torch.int32,
                          device=DEV)
    nact = torch.tensor([active.numel(), 0, 0, 0], dtype=torch.int32, device=DEV)
    qre.qre_cache_update(shape, 6, 0.995, active, nact, st["scores"], st["expert_slot"], st["slot_expert"],
                         st["home"], st["slot_mem"], live.slots, st["copy_list"], st["n_copies"], 64)
    qre.qre_cache_copy(shape, st["home"], st["slot_mem"], st["copy_list"], st["n_copies"], 64)
    torch.cuda.synchronize()
    n = int(st["n_copies"][0].item())
    assert n == 5
    home = st["keep"][0]
    pairs = st["copy_list"][:2 * n].cpu().numpy().reshape(-1, 2)
    for e, s in pairs:
        for name in ("w_gate_up", "s_gate_up", "w_down", "s_down"):
            assert torch.equal(slots.view(int(s), name).cpu(), home.view(int(e), name).cpu())


@pytest.mark.parametrize("T,max_copies", [(1, 64), (4, 64), (4, 1)])
def test_decode_with_live_cache_is_bit_identical_to_hbm(T, max_copies):
    """A decode loop whose slot table the cache manager rewrites every step gives
    the same bits as all experts in device memory, also when a step has more
    misses than its copy list holds (max_copies = 1)."""
    cfg = synthetic.LayerConfig("mid", 512, 256, 32, 4, 128, T)
    S = 6
    live, ref, st, _ = _build_cached_layer(cfg, n_static=4, S=S, T=T)
    wr = torch.from_numpy(synthetic.router_weights(cfg.n_experts, cfg.hidden, cfg.seed, 0)).to(DEV)
    admitted = 0
    for step in range(12):
        x = bits_to_bf16_tensor(synthetic.activations_bits(T, cfg.hidden, cfg.seed, 0, 50 + step), DEV)
        live.route(x, wr, None, T)
        live.dispatch(T)
        qre.qre_cache_update(live.shape, S, 0.995, live.active, live.n_active, st["scores"], st["expert_slot"],
                             st["slot_expert"], st["home"], st["slot_mem"], live.slots, st["copy_list"],
                             st["n_copies"], max_copies)
        qre.qre_cache_copy(live.shape, st["home"], st["slot_mem"], st["copy_list"], st["n_copies"], max_copies)
        live.expert_ffn(x, T)
        live.combine(T)
        ref.forward(x, wr, None, T)
        torch.cuda.synchronize()
        n = int(st["n_copies"][0].item())
        assert n <= max_copies
        admitted += n
        assert torch.equal(live.y[:T], ref.y[:T]), f"step {step}"
    assert admitted > 0
    assert qre.qre_read_device_status() == 0
