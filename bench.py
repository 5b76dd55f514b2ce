#!/usr/bin/env python
"""Benchmark of the quantized routed-expert MoE layer on GB300.

One JSON line on rank 0.  A step is one pass of the whole layer path (route ->
dispatch -> expert FFN -> combine) over one batch of synthetic tokens; for the
42-layer workloads a step is a pass through all 42 layers.  ``value`` is
MoE-layer tokens/s (tokens x layers per second) with inputs resident in HBM,
timed with CUDA events over exactly K graph-replayed steps.  Weights rotate over
enough distinct layer weight sets that every step streams its experts from HBM
(more than L2 between reuses).

Workloads (``--workload``):
  decode1           H4096 I2048 E288 top-8 + shared, T = 1, all 289 experts in HBM
  decode8_zipf_x42  T = 8, Zipf(1.1) routing bias, 42 distinct layers
  cache4_x42        T = 4, Zipf(1.1), 42 layers, 100 experts/layer in pinned host memory
  cache4_live_x16   the same layout with the 148 HBM slots as a live LFU cache, 16 layers
  prefill8192       T = 8192 tokens through one layer (tcgen05 grouped GEMM)
  prefill2048_e64   the same kernels on 64 experts and 2048 tokens (a small profiling case)
  tiny              H256 I128 E16 top-4 + shared, T = 4
The line's top level is the ``--workload`` (decode1 by default); the workloads
named by ``--also`` (prefill8192 by default) are measured in the same run, each
with its own steps, roofline, clocks, e2e and oracle baseline, under
``workloads``.  ``--impl reference`` times the fp64 CPU oracle (the only
reference this build has) on a bounded sample of the same workload.
"""

from __future__ import annotations

import os

# The oracle legs use numpy's BLAS; give it every core of this process explicitly
# (before numpy is imported, which reads these once).
_NCPU = len(os.sched_getaffinity(0))
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_NCPU))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import threading  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "MoE-layer tokens/s at 1 GB300 and achieved HBM GB/s vs roofline (decode); prefill TFLOP/s"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DTYPE_DECODE = ("e4m3 x e4m3, fp32 accumulate (4-bit weights as exact E4M3 codes; x as 2 E4M3 terms, exact "
                "for bf16; h as 4 E4M3 terms, ~16 significant bits)")
DTYPE_DECODE_FP16 = "fp16 x fp16 (exact 4-bit codes; x and h as fp16 high part + remainder), fp32 accumulate"
DTYPE_PREFILL = "fp16 x fp16 (dequantized weights and h rounded to fp16; bf16 x exact), fp32 accumulate"


# ------------------------------------------------------------------ helpers

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


# DRAM bytes per expert-FFN call (both kernels) measured with ncu on a workload,
# for the FFN kernel code with the given hash (ffn_source_hash).  Reported only
# while the sources still hash to that value; a changed kernel reports null.
MEASURED_TRAFFIC = {"decode1": (117420416, "a0f8835ccb0da49a")}
FFN_SOURCES = ("ffn_decode.cu", "common.cuh", "tc.cuh", "internal.h")


def recorded_traffic(workload):
    rec = MEASURED_TRAFFIC.get(workload)
    if rec is None:
        return None
    return rec[0] if ffn_source_hash() == rec[1] else None


def ffn_source_hash():
    """sha256 prefix of the FFN kernel sources with // comments and blank lines
    removed: a change of code (not of comments) invalidates recorded counters."""
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "quantized_routed_expert_03_gb300", "csrc")
    h = hashlib.sha256()
    for f in FFN_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def max_over_ranks(value: float, world: int) -> float:
    """The largest of one number per rank (the slowest replica sets the time);
    the number itself when there is one rank.  Works on an NCCL or a gloo group."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    on_gpu = dist.get_backend() == "nccl"
    dev = torch.device("cuda", torch.cuda.current_device()) if on_gpu else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_step: int, steps: int, ms: float) -> float:
    """Whole-job tokens/s: every rank runs `steps` steps of `tokens_per_step`
    tokens in (at most) `ms` milliseconds."""
    return world * tokens_per_step * steps / (ms / 1e3)


def split_steps(K: int, per_graph: int):
    """(full replays of a per_graph-step graph, remaining steps) that make exactly K steps."""
    return K // per_graph, K % per_graph


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def read_probe_gbs(buf, reps=5) -> float:
    """Best read rate in GB/s of qre_read_probe over ``buf`` (a device tensor or a
    pinned host tensor, read zero-copy), CUDA events around each call."""
    import torch
    import quantized_routed_expert_03_gb300 as qre
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    nbytes = buf.numel() * buf.element_size() // 16 * 16
    qre.qre_read_probe(buf.data_ptr(), nbytes, sink)
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        qre.qre_read_probe(buf.data_ptr(), nbytes, sink)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return nbytes / (best / 1e3) / 1e9


def link_peaks(device) -> dict:
    """Host-link (1 GiB pinned host buffer read zero-copy) and device-memory (4 GiB)
    read rates of the library's streaming-read kernel."""
    import torch
    host = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    host.fill_(1)
    dev = torch.ones(4 << 30, dtype=torch.uint8, device=device)
    out = {"host_link_read_gbs": round(read_probe_gbs(host), 1), "hbm_read_gbs": round(read_probe_gbs(dev), 1),
           "probe": "qre_read_probe: 16-byte streaming loads, 8 in flight per thread, 4 CTAs of 512 threads per SM; "
                    "1 GiB pinned host buffer read zero-copy / 4 GiB device buffer; best of 5"}
    del host, dev
    return out


def default_sets(cfg) -> int:
    """Distinct layer weight sets the steps rotate over: a stack has its own
    layers; one decode layer is repeated in 8 copies (30 GB, far more than L2); a
    prefill step streams far more than L2 by itself."""
    if cfg.layers > 1:
        return cfg.layers
    if cfg.tokens > 8:
        return 1
    return 8 if cfg.hidden >= 4096 else 2


def expert_payload(cfg) -> int:
    """Packed bytes of one expert (weights + scales), the library's format."""
    H, I, G = cfg.hidden, cfg.inter, cfg.group
    return 2 * I * H // 2 + 2 * I * (H // G) * 2 + H * I // 2 + H * (I // G) * 2


def workload_config(name: str, n_sets: int, world: int) -> dict:
    """The ``config`` object of a workload's line (the same for both arms)."""
    cfg = synthetic.CONFIGS[name]
    return {"workload": name, "note": cfg.note, "tokens_per_step": cfg.tokens, "layers_per_step": cfg.layers,
            "hidden": cfg.hidden, "inter": cfg.inter, "experts": cfg.n_experts, "top_k": cfg.top_k,
            "group": cfg.group,
            "l2": f"inputs larger than L2: {n_sets} distinct layer weight set(s) rotated "
                  f"({n_sets * (cfg.n_experts + 1) * expert_payload(cfg) / 1e9:.1f} GB of packed experts)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "launch": "CUDA graph of captured steps"}


def side_note(args) -> dict:
    return {"shared_expert": "side stream (qre_expert_ffn_shared forked beside route/dispatch)"} if getattr(
        args, "side_stream", False) else {}


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [r for (t, r) in self.samples if t0 <= t <= t1 and len(r) >= 9]
        if not rows:
            rows = [r for (_, r) in self.samples if len(r) >= 9][-3:]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ our arm

class Workload:
    """Device weights for the timed steps: ``n_sets`` distinct layers that steps rotate over."""

    def __init__(self, name, device, n_sets=None, log=print):
        import torch
        from quantized_routed_expert_03_gb300.layer import ExpertArena, MoELayer
        self.cfg = cfg = synthetic.CONFIGS[name]
        self.name = name
        H, I, E, k, G, T = cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group, cfg.tokens
        self.T = T
        self.layers_per_step = cfg.layers
        self.n_sets = n_sets = default_sets(cfg) if n_sets is None else n_sets
        t0 = time.time()
        self.sets = []
        staging = None
        for r in range(n_sets):
            if cfg.live_cache:
                self.sets.append(self._live_set(cfg, r, device))
                if (r + 1) % 8 == 0:
                    log(f"[bench] {name}: built {r + 1}/{n_sets} layers ({time.time() - t0:.0f} s)")
                continue
            host = np.append(synthetic.host_resident(cfg, r), False)
            n_host = int(host.sum())
            dev = ExpertArena(H, I, G, E + 1 - n_host, device=device)
            harena = ExpertArena(H, I, G, n_host, host=True) if n_host else None
            if harena is not None and staging is None:
                staging = torch.empty(dev.layout["stride"], dtype=torch.uint8, device=device)
            entries, di, hi = [], 0, 0
            for e in range(E + 1):
                wg, wu, wd = synthetic.expert_fp32_torch(H, I, cfg.seed, r, e, device)
                if host[e]:
                    harena.quantize_into(hi, wg, wu, wd, staging=staging)
                    entries.append(harena.addresses(hi) + (1,))
                    hi += 1
                else:
                    dev.quantize_into(di, wg, wu, wd)
                    entries.append(dev.addresses(di) + (0,))
                    di += 1
                del wg, wu, wd
            L = MoELayer(H, I, E, k, G, T, device=device)
            L.set_slots(entries)
            wr = torch.from_numpy(synthetic.router_weights(E, H, cfg.seed, r)).to(device)
            bias = (torch.from_numpy(synthetic.zipf_bias(E, cfg.seed, r)).to(device) if cfg.zipf else None)
            self.sets.append({"layer": L, "dev": dev, "host": harena, "wr": wr, "bias": bias, "n_host": n_host,
                              "host_mask": host})
            if (r + 1) % 8 == 0:
                log(f"[bench] {name}: built {r + 1}/{n_sets} layers ({time.time() - t0:.0f} s)")
        torch.cuda.synchronize()
        self.expert_payload = self.sets[0]["dev"].layout["payload"]
        self.build_s = time.time() - t0
        log(f"[bench] {name}: weights ready, {n_sets} layer set(s), {self.build_s:.1f} s")

    def _live_set(self, cfg, r, device):
        """One layer with a live expert cache: ranks 1-40 (and the shared expert) in
        static HBM, cfg.hbm_slots - 40 HBM slots run by qre_cache_update /
        qre_cache_copy (first holding ranks 41..hbm_slots), and every non-static
        expert's home copy in pinned host memory."""
        import torch
        import quantized_routed_expert_03_gb300 as qre
        from quantized_routed_expert_03_gb300.layer import ExpertArena, MoELayer
        H, I, E, k, G, T = cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group, cfg.tokens
        S = cfg.hbm_slots - cfg.static_slots
        ranks = synthetic.popularity_ranks(E, cfg.seed, r)
        static = ranks <= cfg.static_slots
        n_home = int((~static).sum())
        st_arena = ExpertArena(H, I, G, int(static.sum()) + 1, device=device)
        slots = ExpertArena(H, I, G, S, device=device)
        home = ExpertArena(H, I, G, n_home, host=True)
        staging = torch.empty(home.layout["stride"], dtype=torch.uint8, device=device)
        table, home_entries = [None] * (E + 1), [None] * (E + 1)
        expert_slot = np.full(E, -1, np.int32)
        slot_expert = np.full(S, -1, np.int32)
        si = hi = 0
        for e in range(E + 1):
            wg, wu, wd = synthetic.expert_fp32_torch(H, I, cfg.seed, r, e, device)
            if e == E or static[e]:
                st_arena.quantize_into(si, wg, wu, wd)
                table[e] = home_entries[e] = st_arena.addresses(si) + (0,)
                if e < E:
                    expert_slot[e] = -2
                si += 1
            else:
                home.quantize_into(hi, wg, wu, wd, staging=staging)
                home_entries[e] = home.addresses(hi) + (1,)
                table[e] = home_entries[e]
                s = int(ranks[e]) - cfg.static_slots - 1
                if s < S:                       # initially cached: its weights in slot s
                    slots.quantize_into(s, wg, wu, wd)
                    table[e] = slots.addresses(s) + (0,)
                    expert_slot[e], slot_expert[s] = s, e
                hi += 1
            del wg, wu, wd
        L = MoELayer(H, I, E, k, G, T, device=device)
        L.set_slots(table)

        def dev_slots(entries):
            raw = bytearray(memoryview(qre.slot_array(entries)).cast("B"))
            return torch.frombuffer(raw, dtype=torch.uint8).to(device)
        max_copies = 16
        cache = {"home": dev_slots(home_entries), "slot_mem": dev_slots([slots.addresses(s) + (0,) for s in range(S)]),
                 "scores": torch.zeros(E, dtype=torch.float32, device=device),
                 "expert_slot": torch.from_numpy(expert_slot).to(device),
                 "slot_expert": torch.from_numpy(slot_expert).to(device),
                 "copy_list": torch.zeros(2 * max_copies, dtype=torch.int32, device=device),
                 "n_copies": torch.zeros(4, dtype=torch.int32, device=device), "S": S, "max_copies": max_copies}
        wr = torch.from_numpy(synthetic.router_weights(E, H, cfg.seed, r)).to(device)
        bias = torch.from_numpy(synthetic.zipf_bias(E, cfg.seed, r)).to(device)
        host_mask = np.append(~static, False)
        return {"layer": L, "dev": st_arena, "host": home, "slots_arena": slots, "wr": wr, "bias": bias,
                "n_host": n_home, "host_mask": host_mask, "cache": cache}

    def x_pool(self, n, device):
        """n distinct activation batches per layer set, [n_sets][n][T,H] bf16 on device."""
        import torch
        cfg = self.cfg
        out = []
        for r in range(self.n_sets):
            xs = np.stack([synthetic.activations_bits(self.T, cfg.hidden, cfg.seed, r, 1000 + i) for i in range(n)])
            out.append(torch.from_numpy(xs.view(np.int16)).to(device).view(torch.bfloat16))
        return out


def measure_workload(name, args, K, W, rank, local_rank, world, device, log, cpu_leg=True):
    """Times K steps of one workload (after W warm-up steps) and returns its record."""
    import torch
    import quantized_routed_expert_03_gb300 as qre
    wl = Workload(name, device, n_sets=args.sets if name == args.workload else None, log=log)
    cfg, T, H, k = wl.cfg, wl.T, wl.cfg.hidden, wl.cfg.top_k
    # host-mapped experts in the tables: cut the decode work at equal cost
    host_cost = args.host_unit_cost if args.host_unit_cost is not None else (3 if cfg.host_tier else 0)
    qre.qre_set_host_unit_cost(host_cost)
    stream = torch.cuda.Stream(device)

    # one captured unit = `per_graph` steps; each step covers one layer set
    # (single-layer workloads) or all layer sets (42-layer stacks)
    stack = wl.layers_per_step > 1
    prefill = T > 8
    per_graph = 1 if (stack or prefill) else wl.n_sets * 4
    # a live cache must see fresh routing every step (a short cycle of batches
    # would let it learn the cycle): one batch per step, warm-up and miss count
    n_x = min(K + W + 16, 256) if cfg.live_cache else (4 if stack else (2 if prefill else per_graph // wl.n_sets))
    xs = wl.x_pool(n_x, device)

    side = torch.cuda.Stream(device) if args.side_stream else None

    def one_layer(s, x):
        layer_step(s, x, T, stream, side)

    # live cache: the captured step reads a static input that each step refills
    # from the pool with one device copy (inside the timed region)
    live = cfg.live_cache
    if live:
        pool = torch.stack([torch.stack([xs[r][j] for r in range(wl.n_sets)]) for j in range(n_x)])
        x_static = pool[0].clone()

    def step_fn(j):
        if live:
            for r, s in enumerate(wl.sets):
                one_layer(s, x_static[r])
        elif stack:
            for r, s in enumerate(wl.sets):
                one_layer(s, xs[r][j % n_x])
        else:
            r = j % wl.n_sets
            one_layer(wl.sets[r], xs[r][(j // wl.n_sets) % n_x])

    def replay(g, j):
        if live:
            x_static.copy_(pool[j % n_x])
        g.replay()

    # eager warm-up (sets kernel attributes, loads modules) then capture
    with torch.cuda.stream(stream):
        for j in range(min(W, per_graph)):
            step_fn(j)
    stream.synchronize()

    def capture(nsteps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(nsteps):
                step_fn(j)
        return g

    n_full, rem = split_steps(K, per_graph)
    g_full = capture(per_graph) if n_full else None
    g_rem = capture(rem) if rem else None

    # warm-up replays: at least W steps, and every graph the timed region replays has run before
    warm = 0
    with torch.cuda.stream(stream):
        while warm < W or (g_full is not None and warm == 0):
            if g_full is not None:
                replay(g_full, warm)
                warm += per_graph
            if g_rem is not None:
                replay(g_rem, warm)
                warm += rem
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    if not args.no_clocks:
        sampler.start()
        time.sleep(0.6)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(n_full):
            replay(g_full, warm + i)
        if g_rem is not None:
            replay(g_rem, warm + n_full)
        end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_wall1 = time.time()
    ms = max_over_ranks(start.elapsed_time(end), world)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    # FFN stage: the expert FFN alone, back to back over the layer sets (each
    # with the routing its last timed step left), in a graph of its own on the
    # same stream, timed with CUDA events around whole replays.
    I = cfg.inter
    ffn_flops = 2.0 * 3 * H * I * (T * k + T)        # gate, up, down for every pick and the shared expert
    ffn_calls = [(r, wl.sets[r]) for r in range(len(wl.sets))] * (1 if (stack or prefill) else 4)
    g_ffn = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_ffn, stream=stream):
        for r, sset in ffn_calls:
            sset["layer"].expert_ffn(xs[r][0], T)
    for _ in range(3):
        g_ffn.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(3, min(50, int(0.05 / max(ms / K / 1e3, 1e-6) / len(ffn_calls) * wl.layers_per_step) + 1))
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g_ffn.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ffn_ms_call = max_over_ranks(e0.elapsed_time(e1), world) / (reps * len(ffn_calls))
    ffn_bytes, n_act, host_bytes = [], [], []
    for r, sset in ffn_calls:
        L = sset["layer"]
        a = int(L.n_active[0].item())
        ids = L.active[:a].cpu().numpy()
        n_act.append(a)
        ffn_bytes.append((a + 1) * wl.expert_payload + T * H * 2 + (T * k + T) * H * 4)
        if "cache" in sset:     # live cache: host-resident = neither static nor in a slot now
            es = sset["cache"]["expert_slot"].cpu().numpy()
            n_host_act = int((es[ids[ids < cfg.n_experts]] == -1).sum())
        else:
            n_host_act = int(sset["host_mask"][ids].sum()) if sset["n_host"] else 0
        host_bytes.append(n_host_act * wl.expert_payload)
    del g_ffn

    tokens_per_step = T * wl.layers_per_step
    value = job_throughput(world, tokens_per_step, K, ms)
    peaks, peak_src = load_peaks()
    fp8 = cfg.group == 128
    if not prefill:
        achieved = float(np.mean(ffn_bytes)) / (ffn_ms_call / 1e3) / 1e9
        peak = float(peaks["hbm_gbs"])
        traffic = (args.traffic if (args.traffic is not None and name == args.workload)
                   else recorded_traffic(name))
        roofline = {"bound": "hbm", "kernel": "qre_expert_ffn (gate/up + down dequant-GEMV kernels)",
                    "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "traffic": traffic,
                    "traffic_unit": "bytes per FFN call (ncu dram read + write)",
                    "peak_source": "of measured (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else
                    "of fallback 6.8 TB/s",
                    "ffn_us_mean": round(ffn_ms_call * 1e3, 2),
                    "ffn_bytes_mean": int(np.mean(ffn_bytes)),
                    "unique_experts_mean": round(float(np.mean(n_act)) + 1, 2),
                    "timed_region": "CUDA events around replays of a graph of expert-FFN calls over the "
                                    "layer sets (mean per call, slowest rank)"}
        if any(host_bytes):
            # experts read over the host link (pinned host memory, zero-copy) vs from HBM
            hb = float(np.mean(host_bytes))
            roofline["host_bytes_mean"] = int(hb)
            roofline["hbm_bytes_mean"] = int(float(np.mean(ffn_bytes)) - hb)
            roofline["hbm_gbs"] = round((float(np.mean(ffn_bytes)) - hb) / (ffn_ms_call / 1e3) / 1e9, 1)
            roofline["host_link_gbs"] = round(hb / (ffn_ms_call / 1e3) / 1e9, 1)
            roofline["frac_hbm"] = round(roofline["hbm_gbs"] / peak, 4)
            lp = link_peaks(device)
            roofline["host_link_peak"] = lp
            roofline["frac_host_link"] = round(roofline["host_link_gbs"] / lp["host_link_read_gbs"], 4)
        per_layer = float(np.mean(ffn_bytes)) + cfg.n_experts * H * 4
        roofline["step_hbm_gbs"] = round(per_layer * wl.layers_per_step / (ms / K / 1e3) / 1e9, 1)
        roofline["step_frac"] = round(roofline["step_hbm_gbs"] / peak, 4)
    else:
        achieved = ffn_flops / (ffn_ms_call / 1e3) / 1e12
        peak = float(peaks["bf16_tflops"])
        roofline = {"bound": "tensor", "kernel": "qre_expert_ffn (gather + two tcgen05 grouped GEMMs)",
                    "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(achieved / peak, 4),
                    "traffic": args.traffic if (args.traffic is not None and name == args.workload) else None,
                    "peak_source": ("of measured (MEASURED_PEAKS.json bf16_tflops, burst: the FFN graph is timed "
                                    "alone; fp16 has the same nominal dense rate as bf16)")
                                   if peak_src == "measured" else "of fallback 1.9 PFLOP/s burst",
                    "frac_of_sustained": round(achieved / float(peaks.get("bf16_tflops_sustained", peak)), 4),
                    "ffn_ms_mean": round(ffn_ms_call, 4), "ffn_tflop": round(ffn_flops / 1e12, 4),
                    "unique_experts_mean": round(float(np.mean(n_act)) + 1, 2),
                    "timed_region": "CUDA events around replays of a graph of expert-FFN calls (mean per call, "
                                    "slowest rank)"}
        roofline["step_tflops"] = round((ffn_flops + 2.0 * T * cfg.n_experts * H) / (ms / K / 1e3) / 1e12, 1)

    rec = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms / K, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_PREFILL if prefill else (DTYPE_DECODE if fp8 else DTYPE_DECODE_FP16),
        "data": "synthetic (seeded generators; random-init weights quantized to the library's 4-bit group format)",
        "config": {**workload_config(name, wl.n_sets, world), **side_note(args),
                   **({"host_unit_cost": host_cost} if host_cost > 1 else {})},
        "gpu_launches": None, "roofline": roofline, "clocks": clocks, "e2e": None,
    }
    # route + dispatch: one token two kernels (logits GEMV, selection with the
    # dispatch), else logits, selection and one (or three) dispatch kernels;
    # expert FFN: gate/up + down (decode) or gather + two grouped GEMMs; combine
    launches_per_layer = (2 if T == 1 else 2 + (1 if T * k <= 1024 else 3)) + (3 if prefill else 2) + 1
    if cfg.live_cache:
        launches_per_layer += 2
        rec["cache"] = cache_misses(wl, xs, T, first=warm + K + 1)
        rec["config"]["inputs"] = "a fresh token batch every step (one 512 KB device copy into the graph's input per step)"
        rec["cache"]["copy_gbs_per_step_time"] = round(
            rec["cache"]["copy_bytes_per_layer_step"] * wl.layers_per_step / (ms / K / 1e3) / 1e9, 1)
    rec["gpu_launches"] = launches_per_layer * wl.layers_per_step * K
    if not args.no_e2e:
        # its own step count: at least ~0.25 s of device work (a few timed steps
        # would mostly time the pipeline filling), at most --e2e-steps; the same
        # on every rank (ms is the slowest rank's)
        k_e2e = max(3, min(args.e2e_steps, max(K, int(0.25 / (ms / K / 1e3)))))
        rec["e2e"] = run_e2e(wl, xs, stream, device, tokens_per_step, world, k_e2e)
    if rank == 0 and cpu_leg and not args.no_cpu_baseline:
        rec["cpu_baseline"] = cpu_baseline(name, wl, device)
    rec["build_s"] = round(wl.build_s, 1)
    del g_full, g_rem
    wl.sets.clear()
    return rec


def layer_step(s, x, T, stream, side=None):
    """One layer of a step: route -> dispatch -> [expert cache update + miss
    copy, for a live cache] -> expert FFN -> combine, on the current stream."""
    import quantized_routed_expert_03_gb300 as qre
    L = s["layer"]
    if side is not None:   # the shared expert on a second stream (fork/join inside the graph)
        L.forward(x, s["wr"], s["bias"], T, stream=stream, shared_stream=side)
        return
    L.route_dispatch(x, s["wr"], s["bias"], T)
    c = s.get("cache")
    if c is not None:
        qre.qre_cache_update(L.shape, c["S"], 0.995, L.active, L.n_active, c["scores"], c["expert_slot"],
                             c["slot_expert"], c["home"], c["slot_mem"], L.slots, c["copy_list"], c["n_copies"],
                             c["max_copies"])
        qre.qre_cache_copy(L.shape, c["home"], c["slot_mem"], c["copy_list"], c["n_copies"], c["max_copies"])
    L.expert_ffn(x, T)
    L.combine(T)


def cache_misses(wl, xs, T, first, steps=8) -> dict:
    """Admissions (miss copies) per layer-step of a live cache over `steps` more
    steps on activation batches first, first + 1, ... (not used by the timed
    steps), counted on the host after each layer (outside any timed region)."""
    import torch
    n_adm = 0
    for j in range(first, first + steps):
        for r, s in enumerate(wl.sets):
            layer_step(s, xs[r][j % xs[r].shape[0]], T, None)
            torch.cuda.synchronize()
            n_adm += int(s["cache"]["n_copies"][0].item())
    per = n_adm / (steps * len(wl.sets))
    return {"misses_per_layer_step": round(per, 3), "copy_bytes_per_layer_step": int(per * wl.expert_payload),
            "counted_over": f"{steps} steps x {len(wl.sets)} layers after the timed region"}


def run_ours(args, rank, local_rank, world):
    import torch
    device = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(device)
    from quantized_routed_expert_03_gb300 import build as qbuild
    qbuild.build()
    import quantized_routed_expert_03_gb300 as qre
    qre.load_library()
    log = (lambda *a: print(*a, file=sys.stderr, flush=True)) if rank == 0 else (lambda *a: None)

    out = measure_workload(args.workload, args, args.steps, args.warmup, rank, local_rank, world, device, log)
    torch.cuda.empty_cache()
    also = [w for w in (args.also.split(",") if args.also else []) if w and w != args.workload]
    if also:
        out["workloads"] = {}
    for name in also:
        cfg = synthetic.CONFIGS[name]
        # each extra workload: a few steps of its own, sized to seconds of timed work
        K = max(3, min(args.steps, 10 if cfg.tokens > 8 else (20 if cfg.layers > 1 else args.steps)))
        rec = measure_workload(name, args, K, max(3, min(args.warmup, 5)), rank, local_rank, world, device, log)
        for key in ("metric", "unit", "n_gpus", "higher_is_better", "scaling", "vs_baseline", "data"):
            rec.pop(key, None)
        out["workloads"][name] = rec
        torch.cuda.empty_cache()
    return out


def run_e2e(wl, xs, stream, device, tokens_per_step, world, K):
    import torch
    T, H = wl.T, wl.cfg.hidden
    stack = wl.layers_per_step > 1
    sets = wl.sets
    xin_dev = [torch.empty((T, H), dtype=torch.bfloat16, device=device) for _ in sets]
    graphs = []

    # one graph per layer set (single-layer workloads) or one for the whole stack
    def body(idx):
        layer_step(sets[idx], xin_dev[idx], T, stream)
    with torch.cuda.stream(stream):
        for i in range(len(sets)):
            body(i)
    stream.synchronize()
    if stack:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(len(sets)):
                body(i)
        graphs = [g]
    else:
        for i in range(len(sets)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                body(i)
            graphs.append(g)
    n_x = xs[0].shape[0]
    host_x = [xs[r].cpu().pin_memory() for r in range(len(sets))]
    # two host output buffers per set: step j's output lands in buffer j % 2
    host_y = [[torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in sets] for _ in range(2)]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    h2d = (len(sets) if stack else 1) * T * H * 2
    d2h = h2d

    # single-layer workloads: the copies run on two copy streams, so that step
    # j + 1's input copy overlaps step j's replay; per layer set, events keep
    # the input from being overwritten before its last replay has read it, and
    # the output from being overwritten before it has been copied out
    cs_in, cs_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    g_done = [torch.cuda.Event() for _ in sets]
    in_done = [torch.cuda.Event() for _ in sets]
    out_done = [torch.cuda.Event() for _ in sets]
    used = [False] * len(sets)

    def one(j):
        b = j % 2
        if stack:
            for r in range(len(sets)):
                xin_dev[r].copy_(host_x[r][j % n_x], non_blocking=True)
            graphs[0].replay()
            for r in range(len(sets)):
                host_y[b][r].copy_(sets[r]["layer"].y_bf16[:T], non_blocking=True)
            done[b].record(stream)
            if j >= 1:
                done[1 - b].synchronize()   # step j - 1's output is on the host before step j + 1 is queued
        else:
            r = j % len(sets)
            # set r's previous step is j - n; when the host queues step j it has
            # step j - 2's output, so with two or more sets that step is done
            # (its replay read the input, its output was copied) and needs no wait
            if used[r] and len(sets) < 2:
                cs_in.wait_event(g_done[r])
            with torch.cuda.stream(cs_in):
                xin_dev[r].copy_(host_x[r][(j // len(sets)) % n_x], non_blocking=True)
            in_done[r].record(cs_in)
            stream.wait_event(in_done[r])
            if used[r] and len(sets) < 2:
                stream.wait_event(out_done[r])
            graphs[r].replay()
            g_done[r].record(stream)
            cs_out.wait_event(g_done[r])
            with torch.cuda.stream(cs_out):
                host_y[b][r].copy_(sets[r]["layer"].y_bf16[:T], non_blocking=True)
            out_done[r].record(cs_out)
            used[r] = True
            if j >= 1:
                out_done[(j - 1) % len(sets)].synchronize()   # step j - 1's output is on the host

    with torch.cuda.stream(stream):
        for j in range(max(3, 2 * len(graphs))):   # every graph replayed (its first replay is slow) before timing
            one(j)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        cs_in.wait_event(s0)   # no copy of the timed steps starts before the timed region
        for j in range(K):
            one(j)
        if not stack:
            stream.wait_event(out_done[(K - 1) % len(sets)])   # ends with the last output on the host
        s1.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(s0.elapsed_time(s1), world)
    return {"value": round(job_throughput(world, tokens_per_step, K, ms), 2), "unit": UNIT, "steps": K,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "the layer's C-ABI calls (route, dispatch, [cache update + miss copy], expert FFN, combine) "
                   "through the binding, captured in a CUDA graph; per step: pinned H2D input copy, replay, "
                   "pinned D2H of the bf16 output into one of two host buffers; the host waits for step j-1's "
                   "output before it queues step j+1 (at most two steps in flight); single-layer workloads "
                   "copy on two copy streams ordered by events, so a step's input copy overlaps the replay "
                   "before it; the timed region ends when the last output is on the host"}


# ------------------------------------------------------------------ oracle (CPU) legs

def _oracle_expert_source(cfg, layer, device):
    """Oracle-quantized experts of one layer, from the same generator the GPU side used."""
    from oracle import quant as oquant
    cache = {}

    def get(e):
        e = int(e)
        if e not in cache:
            if device is not None:
                import torch  # noqa: F401
                w = [t.cpu().numpy() for t in synthetic.expert_fp32_torch(cfg.hidden, cfg.inter, cfg.seed, layer,
                                                                           e, device)]
            else:
                w = synthetic.expert_fp32(cfg.hidden, cfg.inter, cfg.seed, layer, e)
            cache[e] = oquant.quantize_expert(*w, cfg.group)
        return cache[e]
    return get


def _blas_note() -> str:
    return f"numpy BLAS threads {os.environ.get('OPENBLAS_NUM_THREADS')} (OPENBLAS/OMP/MKL_NUM_THREADS)"


def cpu_baseline(name, wl, device):
    """The oracle timed on this host's cores for one full layer-token of the workload."""
    from oracle import moe as omoe
    cfg = wl.cfg
    get = _oracle_expert_source(cfg, 0, device)
    x_bits = synthetic.activations_bits(1, cfg.hidden, cfg.seed, 0, 1000)
    wr = synthetic.router_weights(cfg.n_experts, cfg.hidden, cfg.seed, 0)
    bias = synthetic.zipf_bias(cfg.n_experts, cfg.seed, 0) if cfg.zipf else None
    r = omoe.route(omoe.bf16_bits_to_f64(x_bits), wr, bias, cfg.top_k)
    need = list(r["idx"][0]) + [cfg.n_experts]
    for e in need:                       # quantization is weight preparation, not timed
        get(e)

    class View:
        def __getitem__(self, e):
            return get(e)
    # the same layer-token evaluated again and again until about 10 s of CPU work
    reps, dt = 0, 0.0
    while dt < 10.0 and reps < 40:
        t0 = time.perf_counter()
        omoe.moe_layer(x_bits, wr, bias, View(), get(cfg.n_experts), cfg.hidden, cfg.inter, cfg.n_experts,
                       cfg.top_k, cfg.group)
        dt += time.perf_counter() - t0
        reps += 1
    return {"value": round(reps / dt, 5), "unit": UNIT, "cores": _NCPU, "kind": "oracle",
            "sample": f"1 token through 1 layer of {name} (route + {len(need)} experts dequantized "
                      f"and applied in fp64 numpy), evaluated {reps} times; {dt:.1f} s; {_blas_note()}"}


def run_reference(args):
    """--impl reference: the oracle, on a per-step sample sized to end in a few minutes."""
    from oracle import moe as omoe
    from oracle import quant as oquant
    cfg = synthetic.CONFIGS[args.workload]
    H, I, E, k, G = cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group
    device = None
    try:
        import torch
        if torch.cuda.is_available():
            device = torch.device("cuda:0")
    except Exception:
        pass
    get = _oracle_expert_source(cfg, 0, device)
    wr = synthetic.router_weights(E, H, cfg.seed, 0)
    bias = synthetic.zipf_bias(E, cfg.seed, 0) if cfg.zipf else None
    # The FFN of one expert splits exactly into I/16 blocks of 16 intermediate
    # features (16 gate rows + 16 up rows of the interleaved matrix, 16 down
    # columns).  A layer-token is (k + 1) experts x I/16 blocks.  A step is the
    # route of one token plus m blocks of its experts.
    pool = [get(e) for e in range(2)] + [get(E)]
    blocks_per_token = (k + 1) * (I // 16)

    def block(ex, x, i):
        comb = oquant.dequantize_matrix(ex["w_gate_up"][32 * i:32 * i + 32], ex["s_gate_up"][32 * i:32 * i + 32], H, G)
        g, u = comb[:16], comb[16:]
        c0 = 16 * i
        wd = oquant.dequantize_matrix(ex["w_down"][:, c0 // 2:c0 // 2 + 8],
                                      ex["s_down"][:, c0 // G:c0 // G + 1], 16, 16)
        return wd @ (omoe.silu(g @ x) * (u @ x))

    def step(j, m):
        x_bits = synthetic.activations_bits(1, H, cfg.seed, 0, 1000 + j)
        x = omoe.bf16_bits_to_f64(x_bits)
        omoe.route(x, wr, bias, k)
        acc = np.zeros(H)
        for b in range(m):
            ex = pool[(j + b) % len(pool)]
            acc += block(ex, x[0], (j * m + b) % (I // 16))
        return acc

    t0 = time.perf_counter()
    step(0, 4)
    t_block = (time.perf_counter() - t0) / 4
    budget = 150.0 / max(1, args.steps + args.warmup)
    m = int(max(1, min(blocks_per_token, budget / max(t_block, 1e-6))))
    for j in range(args.warmup):
        step(j, m)
    t0 = time.perf_counter()
    for j in range(args.steps):
        step(args.warmup + j, m)
    dt = time.perf_counter() - t0
    tokens = args.steps * m / blocks_per_token * (cfg.tokens if cfg.layers == 1 else 1)
    value = tokens / dt
    sample = (f"per step: route 1 token + {m} of the {blocks_per_token} 16-feature FFN blocks of a "
              f"{args.workload} layer-token (fp64 numpy oracle); scaled to layer-tokens; {_blas_note()}")
    n_sets = args.sets if args.sets is not None else default_sets(cfg)
    return {"metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, n_sets, 1), "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": _NCPU, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def make_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode1", choices=sorted(synthetic.CONFIGS))
    ap.add_argument("--also", default="prefill8192",
                    help="comma-separated workloads measured after the main one, reported under 'workloads' "
                         "('' for none)")
    ap.add_argument("--e2e-steps", type=int, default=5000)
    ap.add_argument("--sets", type=int, default=None,
                    help="distinct layer weight sets to rotate over (default: enough to exceed L2)")
    ap.add_argument("--side-stream", action="store_true",
                    help="run the shared expert on a second stream beside the router and dispatch")
    ap.add_argument("--host-unit-cost", type=int, default=None,
                    help="decode work cut: cost of a host-mapped unit (default 3 with host-resident experts, else 0)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per FFN launch, when a capture of the current kernels exists")
    return ap


def main():
    ap = make_parser()
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    out = run_ours(args, rank, local_rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
