"""Device plumbing for one routed MoE layer: buffers, expert arenas, slot table.

PyTorch only allocates memory and supplies streams here; every computation is a
call into libqre.so through the binding in ``__init__``.

* :class:`ExpertArena` keeps the packed experts of a layer in one allocation,
  either device memory (HBM cache slots) or pinned host memory that the GPU
  reads zero-copy (the glm53-flash-offload README, "Zero-copy home": one
  exact-size pinned arena per layer).
* :class:`MoELayer` owns the per-call buffers and the device slot table, and
  runs route -> dispatch -> expert FFN -> combine on one stream, or with the
  shared expert on a second stream beside the router and the dispatch (the
  glm53-flash-offload README, "Decode kernels": the shared expert on a side
  stream); both give the same bits.
"""

from __future__ import annotations

import ctypes

import torch

from . import (make_shape, qre_combine, qre_dispatch, qre_expert_ffn, qre_expert_ffn_routed, qre_expert_ffn_shared,
               qre_quantize, qre_quantize_gate_up, qre_route, qre_route_dispatch, qre_shared_workspace_size, qre_slot,
               qre_stage_experts, qre_validate_slots, qre_workspace_size, slot_array)

_ALIGN = 256


def _a(n: int) -> int:
    return (n + _ALIGN - 1) // _ALIGN * _ALIGN


def expert_layout(H: int, I: int, G: int) -> dict:
    """Byte offsets of the four arrays of one packed expert, and its stride."""
    wgu, sgu = 2 * I * H // 2, 2 * I * (H // G) * 2
    wd, sd = H * I // 2, H * (I // G) * 2
    o_sgu = _a(wgu)
    o_wd = o_sgu + _a(sgu)
    o_sd = o_wd + _a(wd)
    return {"w_gate_up": (0, wgu), "s_gate_up": (o_sgu, sgu), "w_down": (o_wd, wd), "s_down": (o_sd, sd),
            "stride": o_sd + _a(sd), "payload": wgu + sgu + wd + sd}


class ExpertArena:
    """``n`` packed experts in one contiguous allocation (device, or pinned host)."""

    def __init__(self, H: int, I: int, G: int, n: int, device="cuda", host: bool = False):
        self.H, self.I, self.G, self.n, self.host = H, I, G, n, host
        self.layout = expert_layout(H, I, G)
        nbytes = self.layout["stride"] * n
        if host:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        else:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def view(self, e: int, name: str) -> torch.Tensor:
        off, size = self.layout[name]
        base = e * self.layout["stride"] + off
        return self.buf[base:base + size]

    def addresses(self, e: int) -> tuple:
        return tuple(self.view(e, n).data_ptr() for n in ("w_gate_up", "s_gate_up", "w_down", "s_down"))

    def quantize_into(self, e: int, w_gate, w_up, w_down, stream=None, staging=None) -> None:
        """Quantizes fp32 device weights (gate/up [I,H], down [H,I]) into slot e.

        For a host arena the kernels write a device staging buffer (``staging``,
        at least one expert stride) that is then copied into pinned memory.
        """
        H, I, G = self.H, self.I, self.G
        if self.host:
            if staging is None:
                staging = torch.empty(self.layout["stride"], dtype=torch.uint8, device=w_gate.device)
            dst = {n: staging[self.layout[n][0]:self.layout[n][0] + self.layout[n][1]]
                   for n in ("w_gate_up", "s_gate_up", "w_down", "s_down")}
        else:
            dst = {n: self.view(e, n) for n in ("w_gate_up", "s_gate_up", "w_down", "s_down")}
        qre_quantize_gate_up(I, H, G, w_gate, w_up, dst["w_gate_up"], dst["s_gate_up"], stream)
        qre_quantize(H, I, G, w_down, dst["w_down"], dst["s_down"], stream)
        if self.host:
            for n, t in dst.items():
                self.view(e, n).copy_(t, non_blocking=False)

    def to_numpy(self, e: int) -> dict:
        """The packed arrays of slot e on the host, row-major (for checks)."""
        H, I, G = self.H, self.I, self.G
        out = {}
        for n, (rows, cols) in {"w_gate_up": (2 * I, H), "w_down": (H, I)}.items():
            out[n] = packed_rows(self.view(e, n).cpu().numpy(), rows, cols)
        for n, (rows, cols) in {"s_gate_up": (2 * I, H), "s_down": (H, I)}.items():
            out[n] = scale_rows(self.view(e, n).cpu().numpy(), rows, cols, G)
        return out


def packed_rows(raw, rows: int, cols: int):
    """Row-major [rows][cols/2] bytes from the library's tiled packed storage.

    The storage holds 4 KB chunks, one per 128-row block and 64-column stage
    (block-major); inside a chunk, the 16 bytes of columns 0-31 of each of the
    128 rows in order, then the 16 bytes of columns 32-63.
    """
    import numpy as np
    t = np.asarray(raw, dtype=np.uint8).reshape(rows // 128, cols // 64, 2, 128, 16)
    return np.ascontiguousarray(t.transpose(0, 3, 1, 2, 4)).reshape(rows, cols // 2)


def scale_rows(raw, rows: int, cols: int, G: int):
    """Row-major fp16 [rows][cols/G] scales from the tiled storage: for each
    128-row block and group, the 128 rows' scales in order."""
    import numpy as np
    t = np.asarray(raw).view(np.float16).reshape(rows // 128, cols // G, 128)
    return np.ascontiguousarray(t.transpose(0, 2, 1)).reshape(rows, cols // G)


class MoELayer:
    """Buffers and slot table for calls with up to ``t_max`` tokens."""

    def __init__(self, H: int, I: int, E: int, k: int, G: int, t_max: int, device="cuda"):
        self.H, self.I, self.E, self.k, self.G, self.t_max = H, I, E, k, G, t_max
        self.shape = make_shape(H, I, E, k, G)
        self.device = torch.device(device)
        dev = self.device
        P = t_max * k
        i32 = dict(dtype=torch.int32, device=dev)
        self.topk_idx = torch.empty((t_max, k), **i32)
        self.topk_w = torch.empty((t_max, k), dtype=torch.float32, device=dev)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.perm = torch.empty(P, **i32)
        self.inv_perm = torch.empty(P, **i32)
        self.active = torch.empty(E, **i32)
        self.n_active = torch.zeros(4, **i32)
        self.expert_out = torch.empty((P + t_max, H), dtype=torch.float32, device=dev)
        self.y = torch.empty((t_max, H), dtype=torch.float32, device=dev)
        self.y_bf16 = torch.empty((t_max, H), dtype=torch.bfloat16, device=dev)
        self.ws_bytes = qre_workspace_size(self.shape, t_max)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.slots = torch.zeros((E + 1) * ctypes.sizeof(qre_slot), dtype=torch.uint8, device=dev)
        self.host_slots = None
        self.shared_ws = None          # workspace of the side-stream shared expert, allocated on first use
        self._fork = self._join = None

    def set_slots(self, entries, validate: bool = True) -> None:
        """entries: E + 1 tuples (w_gate_up, s_gate_up, w_down, s_down, tier); entry E is the shared expert."""
        assert len(entries) == self.E + 1
        arr = slot_array(entries)
        if validate:
            qre_validate_slots(self.shape, arr)
        raw = bytes(memoryview(arr).cast("B"))
        self.slots.copy_(torch.frombuffer(bytearray(raw), dtype=torch.uint8))
        self.host_slots = arr

    def route(self, x, w_router, bias, T, stream=None):
        qre_route(self.shape, T, x, w_router, bias, self.topk_idx, self.topk_w, self.workspace, self.ws_bytes, stream)

    def route_dispatch(self, x, w_router, bias, T, stream=None):
        """route + dispatch in one library call (fewer launches for decode batches)."""
        qre_route_dispatch(self.shape, T, x, w_router, bias, self.topk_idx, self.topk_w, self.counts, self.offsets,
                           self.perm, self.inv_perm, self.active, self.n_active, self.workspace, self.ws_bytes, stream)

    def dispatch(self, T, stream=None):
        qre_dispatch(self.shape, T, self.topk_idx, self.counts, self.offsets, self.perm, self.inv_perm, self.active,
                     self.n_active, self.workspace, self.ws_bytes, stream)

    def expert_ffn(self, x, T, stream=None, slots=None):
        """slots: another device slot table for this call (a staged one), default the layer's."""
        qre_expert_ffn(self.shape, T, x, self.slots if slots is None else slots, self.offsets, self.perm,
                       self.active, self.n_active, self.expert_out, self.workspace, self.ws_bytes, stream)

    def expert_ffn_routed(self, x, T, stream=None):
        qre_expert_ffn_routed(self.shape, T, x, self.slots, self.offsets, self.perm, self.active, self.n_active,
                              self.expert_out, self.workspace, self.ws_bytes, stream)

    def expert_ffn_shared(self, x, T, stream=None):
        if self.shared_ws is None:
            n = qre_shared_workspace_size(self.shape, self.t_max)
            self.shared_ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        qre_expert_ffn_shared(self.shape, T, x, self.slots, self.expert_out, self.shared_ws, None, stream)

    def combine(self, T, stream=None, bf16: bool = True):
        qre_combine(self.shape, T, self.expert_out, self.topk_w, self.inv_perm, self.y,
                    self.y_bf16 if bf16 else None, stream)

    def forward(self, x, w_router, bias, T=None, stream=None, shared_stream=None, slots=None):
        """Runs the whole layer on ``x`` ([T, H] bf16, device); results stay in the buffers.

        With ``shared_stream`` (a torch.cuda.Stream) the shared expert runs there,
        forked after ``x`` is ready and joined before the combine; the routed
        experts, router and dispatch stay on ``stream`` (default: the current one).
        The output bits are the same either way.  Works inside CUDA graph capture.
        """
        T = x.shape[0] if T is None else T
        if shared_stream is None:
            self.route_dispatch(x, w_router, bias, T, stream)
            self.expert_ffn(x, T, stream, slots)
            self.combine(T, stream)
            return self.y[:T]
        assert slots is None, "a staged table is not combined with the side-stream shared expert here"
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        if self._fork is None:
            self._fork, self._join = torch.cuda.Event(), torch.cuda.Event()
        self._fork.record(main)
        shared_stream.wait_event(self._fork)
        self.expert_ffn_shared(x, T, shared_stream)
        self._join.record(shared_stream)
        self.route_dispatch(x, w_router, bias, T, main)
        self.expert_ffn_routed(x, T, main)
        main.wait_event(self._join)
        self.combine(T, main)
        return self.y[:T]


class StagingArea:
    """HBM slots that hold one layer's host-resident experts during a prefill chunk.

    ``stage(layer, stream)`` copies the layer's tier-1 experts into the slots on
    ``stream`` (copy engines) and leaves a staged slot table in ``self.table``
    (device) that points at them.  Use two areas to stage layer l + 1 while layer
    l computes (:func:`staged_prefill`).
    """

    def __init__(self, H: int, I: int, G: int, E: int, n_slots: int, device="cuda"):
        self.E = E
        self.arena = ExpertArena(H, I, G, n_slots, device=device)
        self.host_staging = slot_array([self.arena.addresses(j) + (0,) for j in range(n_slots)])
        self.table = torch.zeros((E + 1) * ctypes.sizeof(qre_slot), dtype=torch.uint8, device=device)
        self.n_staged = 0

    def stage(self, layer: "MoELayer", stream=None) -> int:
        if getattr(layer, "stage_host_out", None) is None:   # per layer: stays valid while its upload is queued
            layer.stage_host_out = torch.empty((layer.E + 1) * ctypes.sizeof(qre_slot), dtype=torch.uint8,
                                               pin_memory=True)
        self.n_staged = qre_stage_experts(layer.shape, layer.host_slots, self.host_staging, layer.stage_host_out,
                                          self.table, stream)
        return self.n_staged


def staged_prefill(layers, inputs, areas, copy_stream, T, stream=None):
    """A prefill chunk through a stack of layers with each layer's host-resident
    experts staged into HBM one layer ahead on ``copy_stream``.

    layers: MoELayer objects; inputs: (x, w_router, bias) per layer (the layers are
    independent here: between MoE layers a model has attention, which is not this
    library's); areas: two StagingArea objects used alternately.  Ordering: layer l
    waits for its area's copies; the copies into an area wait until the layer that
    last read it has finished its expert FFN.  Works inside CUDA graph capture.
    """
    main = stream if stream is not None else torch.cuda.current_stream()
    staged = [torch.cuda.Event() for _ in areas]
    freed = [torch.cuda.Event() for _ in areas]
    copy_stream.wait_stream(main)
    areas[0].stage(layers[0], copy_stream)
    staged[0].record(copy_stream)
    for l, L in enumerate(layers):
        a = l % 2
        if l + 1 < len(layers):
            b = (l + 1) % 2
            if l >= 1:
                copy_stream.wait_event(freed[b])
            areas[b].stage(layers[l + 1], copy_stream)
            staged[b].record(copy_stream)
        main.wait_event(staged[a])
        x, wr, bias = inputs[l]
        L.forward(x, wr, bias, T, stream=main, slots=areas[a].table)
        freed[a].record(main)
    main.wait_stream(copy_stream)
